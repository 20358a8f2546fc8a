"""Slot mapping, KV-slot scatter and copy-on-write copy on the GPU: bit-exact
against the oracle, plus the device error word for bad indices."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import bits, to_gpu_meta

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_slot_mapping_random(pkv, seed):
    w = wl.random_case(seed, num_seqs=17, max_ctx=200, max_q=60)
    m = to_gpu_meta(w)
    got = pkv.pkv_slot_mapping(m["block_tables"], m["seq_lens"], m["query_start_loc"], w.num_tokens)
    assert pkv.pkv_get_last_error() == 0
    ref = oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc)
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("name", ["mixed", "long", "prefix"])
def test_slot_mapping_workloads(pkv, name):
    w = wl.make(name)
    m = to_gpu_meta(w)
    got = pkv.pkv_slot_mapping(m["block_tables"], m["seq_lens"], m["query_start_loc"], w.num_tokens)
    assert pkv.pkv_get_last_error() == 0
    assert np.array_equal(got.cpu().numpy(), oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc))


def test_slot_mapping_flags_short_table(pkv):
    w = wl.sized_case(5, [40, 30], [3, 1], 2, 1, 64, "f32")
    bt = w.block_tables[:, :2].copy()                # 40 tokens need 3 blocks: position 39 has no entry
    m = to_gpu_meta(w, bt)
    got = pkv.pkv_slot_mapping(m["block_tables"], m["seq_lens"], m["query_start_loc"], w.num_tokens).cpu().numpy()
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    assert got[0] == -1 and got[1] == -1 and got[2] == -1          # positions 37..39 live in block 2
    assert got[3] == bt[1, 29 // 16] * 16 + 29 % 16


@pytest.mark.parametrize("dtype,d,hkv", [("f32", 64, 1), ("f32", 128, 2), ("bf16", 128, 8)])
def test_write_bitexact(pkv, dtype, d, hkv):
    rng = np.random.default_rng(7)
    nb, T = 50, 300
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(3)
    kc = torch.randn((nb, hkv, 16, d), generator=g).to(tdt)
    vc = torch.randn((nb, hkv, 16, d), generator=g).to(tdt)
    k = torch.randn((T, hkv, d), generator=g).to(tdt)
    v = torch.randn((T, hkv, d), generator=g).to(tdt)
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[::17] = -1
    kc_g, vc_g = kc.cuda(), vc.cuda()
    pkv.pkv_write(k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), kc_g, vc_g)
    assert pkv.pkv_get_last_error() == 0
    ek, ev = bits(kc), bits(vc)
    oracle.write(bits(k), bits(v), slots, ek, ev)
    assert np.array_equal(bits(kc_g), ek) and np.array_equal(bits(vc_g), ev)


def test_write_flags_slot_past_pool(pkv):
    nb, hkv, d = 4, 1, 64
    kc = torch.zeros((nb, hkv, 16, d), device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((2, hkv, d), device="cuda")
    slots = torch.tensor([nb * 16, 5], dtype=torch.int64, device="cuda")
    pkv.pkv_write(k, k.clone(), slots, kc, vc)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    assert kc.sum().item() == d and kc[0, 0, 5].sum().item() == d     # the good token landed, nothing else


@pytest.mark.parametrize("dtype,d,hkv,n", [("bf16", 128, 8, 256), ("f32", 64, 1, 7), ("bf16", 128, 2, 1)])
def test_copy_blocks_bitexact(pkv, dtype, d, hkv, n):
    rng = np.random.default_rng(n)
    nb = 2 * n + 9
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(n)
    kc = torch.randn((nb, hkv, 16, d), generator=g).to(tdt)
    vc = torch.randn((nb, hkv, 16, d), generator=g).to(tdt)
    perm = rng.permutation(nb).astype(np.int32)
    src, dst = perm[:n].copy(), perm[n:2 * n].copy()
    kc_g, vc_g = kc.cuda(), vc.cuda()
    pkv.pkv_copy_blocks(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), kc_g, vc_g)
    assert pkv.pkv_get_last_error() == 0
    ek, ev = bits(kc), bits(vc)
    oracle.copy_blocks(src, dst, ek, ev)
    assert np.array_equal(bits(kc_g), ek) and np.array_equal(bits(vc_g), ev)


def test_copy_blocks_workload_pairs(pkv):
    w = wl.make("prefix")
    t = w.make_tensors("cuda")
    ek, ev = bits(t["k_cache"]), bits(t["v_cache"])
    pkv.pkv_copy_blocks(torch.from_numpy(w.cow_src).cuda(), torch.from_numpy(w.cow_dst).cuda(), t["k_cache"],
                        t["v_cache"])
    assert pkv.pkv_get_last_error() == 0
    oracle.copy_blocks(w.cow_src, w.cow_dst, ek, ev)
    assert np.array_equal(bits(t["k_cache"]), ek) and np.array_equal(bits(t["v_cache"]), ev)


def test_copy_blocks_flags_bad_id_and_leaves_canaries(pkv):
    nb = 6
    kc = torch.arange(nb * 16 * 64, dtype=torch.float32, device="cuda").reshape(nb, 1, 16, 64)
    vc = kc.clone()
    before = kc.clone()
    src = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    dst = torch.tensor([nb, 3], dtype=torch.int32, device="cuda")   # first pair names a block past the pool
    pkv.pkv_copy_blocks(src, dst, kc, vc)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    expect = before.clone()
    expect[3] = before[1]
    assert torch.equal(kc, expect) and torch.equal(vc, expect)


def test_empty_calls_are_noops(pkv):
    kc = torch.zeros((2, 1, 16, 64), device="cuda")
    pkv.pkv_write(torch.zeros((0, 1, 64), device="cuda"), torch.zeros((0, 1, 64), device="cuda"),
                  torch.zeros(0, dtype=torch.int64, device="cuda"), kc, kc.clone())
    pkv.pkv_copy_blocks(torch.zeros(0, dtype=torch.int32, device="cuda"),
                        torch.zeros(0, dtype=torch.int32, device="cuda"), kc, kc.clone())
    assert pkv.pkv_get_last_error() == 0
