"""A seeded sweep over batch shapes, on top of the hand-picked cases.

Each case draws its own element type, head layout, batch size and length mix, so that
combinations no hand-picked case names meet the kernels: one-request batches, odd
query-tile counts, decodes just past a split boundary, wide GQA groups over many kv
heads, batches with no decode or no prefill.  Every case runs one whole step (slot
mapping, K/V scatter, attention) and is checked against the oracle with the same
tolerances as the rest: bf16 max-abs 2e-2 and mean-abs 2e-3, fp32 1e-4.

The shared-prefix sweep draws the prefix groups too (their count, prefix lengths that
do and do not end on a 512-key split, member counts on both sides of the paired-tile
choice, suffix lengths from one key to several decode splits, malformed hints or
none) and checks ``paged_attention_cascade`` against the oracle's plain attention.

The one-token fp32 sweep draws batches whose requests each bring one token (head_dim 64
or 128, groups that do and do not split into two head chunks, contexts from one key up)
and runs ``paged_attention_step``, where the attention launch stores the new rows itself.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import bits, compare, gpu_step, oracle_step

pytestmark = pytest.mark.gpu

# fp64 oracle work per case, in multiply-adds x 2 over Q K^T and P V: the sweep's
# cases stay under a second or so of oracle time each
ORACLE_BUDGET = 6e9


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def draw_mixed(seed: int):
    rng = np.random.default_rng(10_000 + seed)
    dtype = "bf16" if rng.random() < 0.75 else "f32"
    d = 128 if dtype == "bf16" else int(rng.choice([64, 128]))
    group = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 16]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    while group * hkv > 64:
        hkv //= 2
    num_seqs = int(rng.integers(1, 16, endpoint=True))
    max_ctx = int(rng.choice([20, 300, 1100, 2600, 4500]))
    max_q = int(rng.choice([1, 17, 130, 400, 700]))
    decode_frac = float(rng.choice([0.0, 0.3, 0.7, 1.0]))
    while True:
        w = wl.random_case(seed, num_seqs, max_ctx, max_q, group, hkv, d, dtype, decode_frac)
        q = np.diff(w.query_start_loc)
        work = float(np.sum(q.astype(np.float64) * w.seq_lens)) * group * hkv * d * 4
        if work <= ORACLE_BUDGET or num_seqs == 1:
            return w
        num_seqs -= 1


@pytest.mark.parametrize("seed", range(96))
def test_mixed_step_sweep(pkv, seed):
    w = draw_mixed(seed)
    t_cpu = w.make_tensors("cpu")
    t_gpu = {k: v.cuda() for k, v in t_cpu.items()}
    out, slots, st = gpu_step(pkv, w, t_gpu)
    assert st == 0, pkv.status_string(st)
    ref, ref_slots, kc, vc = oracle_step(w, t_cpu)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    # the scatter is bit-exact: the pools after the step are equal as bit patterns
    assert np.array_equal(bits(t_gpu["k_cache"]).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(bits(t_gpu["v_cache"]).view(np.uint8), vc.view(np.uint8))
    compare(out, ref, w.dtype, f"{w.name} {w.dtype} d{w.head_dim} {w.num_q_heads}/{w.num_kv_heads}")


def draw_shared(seed: int):
    rng = np.random.default_rng(20_000 + seed)
    G = int(rng.integers(1, 3, endpoint=True))
    prefix_blocks = tuple(int(rng.choice([1, 7, 32, 33, 64, 95, 130])) for _ in range(G))
    members = tuple(int(rng.choice([1, 2, 9, 31, 33, 70])) for _ in range(G))
    group = int(rng.choice([1, 2, 4, 6, 8, 16]))
    hkv = int(rng.choice([1, 2, 4, 8]))
    while group * hkv > 64:
        hkv //= 2
    max_suffix = int(rng.choice([1, 15, 16, 17, 300, 2100]))
    long_suffix = int(rng.choice([0, 0, 0, 2049, 4000]))
    bystanders = int(rng.integers(0, 6, endpoint=True))
    bad_hints = bool(rng.random() < 0.5)
    return wl.shared_prefix_case(seed, prefix_blocks=prefix_blocks, members=members, num_kv_heads=hkv,
                                 group=group, max_suffix=max_suffix, bystanders=bystanders, bad_hints=bad_hints,
                                 long_suffix=long_suffix)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("seed", range(48))
def test_shared_prefix_sweep(pkv, seed):
    w, hints = draw_shared(seed)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    cas = pkv.paged_attention_cascade(t["q"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale,
                                      max(1, w.max_query_len), w.max_seq_len, dev(hints["prefix_block_tables"]),
                                      dev(hints["prefix_num_blocks"]), dev(hints["member_start"]),
                                      dev(hints["member_seqs"]))
    st = pkv.pkv_get_last_error()
    assert st == 0, pkv.status_string(st)
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", f"{w.name} {w.num_q_heads}/{w.num_kv_heads} prefixes {hints['prefix_num_blocks']}")


def draw_one_token_f32(seed: int):
    rng = np.random.default_rng(30_000 + seed)
    d = int(rng.choice([64, 128]))
    group = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))  # above 8: two head chunks per (token, kv head)
    hkv = int(rng.choice([1, 2, 4, 8]))
    while group * hkv > 64:
        hkv //= 2
    num_seqs = int(rng.integers(1, 40, endpoint=True))
    max_ctx = int(rng.choice([1, 20, 300, 1500, 4000]))
    while True:
        w = wl.random_case(seed, num_seqs, max_ctx, 1, group, hkv, d, "f32", decode_frac=1.0)
        work = float(np.sum(w.seq_lens.astype(np.float64))) * group * hkv * d * 4
        if work <= ORACLE_BUDGET or num_seqs == 1:
            return w
        num_seqs -= 1


@pytest.mark.parametrize("seed", range(24))
def test_fp32_one_token_step_sweep(pkv, seed):
    """paged_attention_step on fp32 batches of one-token requests, where the attention
    launch itself stores the new rows: slots and pools bit-exact, outputs within 1e-4."""
    w = draw_one_token_f32(seed)
    assert w.max_query_len == 1
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    m = {k: torch.from_numpy(np.ascontiguousarray(getattr(w, k))).cuda()
         for k in ("block_tables", "seq_lens", "query_start_loc")}
    slots = torch.full((w.num_tokens,), -7, dtype=torch.int64, device="cuda")
    out = pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], m["block_tables"],
                                   m["seq_lens"], m["query_start_loc"], w.scale, 1, max(1, w.max_seq_len),
                                   slot_mapping=slots)
    st = pkv.pkv_get_last_error()
    assert st == 0, pkv.status_string(st)
    ref, ref_slots, kc, vc = oracle_step(w, t_cpu)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    assert np.array_equal(bits(t["k_cache"]).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(bits(t["v_cache"]).view(np.uint8), vc.view(np.uint8))
    compare(out, ref, "f32", f"{w.name} d{w.head_dim} {w.num_q_heads}/{w.num_kv_heads}")
