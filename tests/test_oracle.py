"""Pins for the fp64 oracle, checked against things other than itself.

Each check ties the oracle to something the pages or the mathematics fix:
  * a library attention routine (torch's scaled_dot_product_attention in fp64)
    over dense, contiguous K/V that never pass through a block table
    ("Introduction" page, PagedAttention (intuition): the logical context is
    contiguous, the physical pages need not be);
  * closed forms (one key, identical keys, zero query, two keys, one dominant
    logit) and scipy's softmax for the weights themselves;
  * invariances the teardown's "PagedAttention" section implies: a permutation of
    physical block ids, and shared prefix blocks versus duplicated copies, leave
    the result bit-identical; one mixed batch equals separate calls
    ("Continuous batching" section);
  * slot mapping round trip: every logical position lands in its own slot and is
    read back exactly once;
  * byte-level references for the scatter and the copy-on-write copy;
  * a mutation check: plausible mistakes planted in a copy of the oracle's C
    source are each caught by these pins.
"""
import math
import os
import re
import subprocess

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
import workloads as wl

BLOCK = 16


def to_bits(x: torch.Tensor) -> np.ndarray:
    """fp32 -> numpy fp32; bf16 -> numpy int16 bit pattern (what the oracle reads)."""
    if x.dtype == torch.bfloat16:
        return x.contiguous().view(torch.int16).numpy().copy()
    return x.contiguous().numpy().copy()


def as_f64(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.float64).numpy()


def place_dense(dense_k, dense_v, block_tables, num_blocks, fill=0.0, dtype=torch.float32):
    """Test-side paging: put each request's dense [L, Hkv, d] K/V into a pool
    [num_blocks, Hkv, 16, d] at the blocks its table names (independent of the oracle)."""
    hkv, d = dense_k[0].shape[1], dense_k[0].shape[2]
    kc = torch.full((num_blocks, hkv, BLOCK, d), fill, dtype=dtype)
    vc = torch.full((num_blocks, hkv, BLOCK, d), fill, dtype=dtype)
    for i, (k, v) in enumerate(zip(dense_k, dense_v)):
        for u in range(k.shape[0]):
            b = int(block_tables[i][u // BLOCK])
            kc[b, :, u % BLOCK] = k[u]
            vc[b, :, u % BLOCK] = v[u]
    return kc, vc


def sdpa_reference(q, dense_k, dense_v, seq_lens, qsl, scale, group):
    """torch SDPA in fp64 over dense contexts with a bottom-right causal mask."""
    outs = []
    for i in range(len(seq_lens)):
        q_i = q[qsl[i]:qsl[i + 1]].to(torch.float64)          # [q, Hq, d]
        n_q, L = q_i.shape[0], int(seq_lens[i])
        if n_q == 0:
            continue
        k = dense_k[i].to(torch.float64).repeat_interleave(group, dim=1)  # [L, Hq, d]
        v = dense_v[i].to(torch.float64).repeat_interleave(group, dim=1)
        pos = torch.arange(L - n_q, L).unsqueeze(1)
        mask = torch.arange(L).unsqueeze(0) <= pos                        # [q, L]
        o = F.scaled_dot_product_attention(q_i.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                           attn_mask=mask, scale=float(np.float32(scale)))
        outs.append(o.transpose(0, 1))
    return torch.cat(outs).numpy() if outs else np.zeros((0,) + tuple(q.shape[1:]))


def random_dense_case(seed, num_seqs, max_ctx, max_q, group, hkv, d, dtype=torch.float32):
    w = wl.random_case(seed, num_seqs=num_seqs, max_ctx=max_ctx, max_q=max_q, group=group,
                       num_kv_heads=hkv, head_dim=d, dtype="f32" if dtype == torch.float32 else "bf16")
    g = torch.Generator().manual_seed(seed)
    dense_k = [torch.randn((int(L), hkv, d), generator=g).to(dtype) for L in w.seq_lens]
    dense_v = [torch.randn((int(L), hkv, d), generator=g).to(dtype) for L in w.seq_lens]
    q = torch.randn((w.num_tokens, w.num_q_heads, d), generator=g).to(dtype)
    return w, q, dense_k, dense_v


def run_oracle(w, q, kc, vc, bt=None, rows=None):
    return oracle.attention(to_bits(q), to_bits(kc), to_bits(vc), w.block_tables if bt is None else bt,
                            w.seq_lens, w.query_start_loc, w.scale, rows=rows)


# --------------------------------------------------------------------------- library routine

@pytest.mark.parametrize("seed,group,hkv,d,dtype", [
    (1, 1, 1, 8, torch.float32), (2, 2, 2, 8, torch.float32), (3, 4, 1, 64, torch.float32),
    (4, 2, 2, 64, torch.bfloat16), (5, 4, 2, 8, torch.bfloat16), (6, 1, 3, 64, torch.float32),
])
def test_matches_sdpa_on_dense_context(seed, group, hkv, d, dtype):
    w, q, dk, dv = random_dense_case(seed, num_seqs=6, max_ctx=80, max_q=40, group=group, hkv=hkv, d=d,
                                     dtype=dtype)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks, fill=float("nan"), dtype=dtype)
    got = run_oracle(w, q, kc, vc)
    ref = sdpa_reference(q, dk, dv, w.seq_lens, w.query_start_loc, w.scale, group)
    assert got.shape == ref.shape
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_unused_slots_are_never_read():
    # the pool is filled with NaN everywhere except the logical context; any read of
    # a slot at or past seq_len, or of a padding table entry, would poison the result
    w, q, dk, dv = random_dense_case(11, num_seqs=8, max_ctx=60, max_q=30, group=2, hkv=2, d=8)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks, fill=float("nan"))
    got = run_oracle(w, q, kc, vc)
    assert np.isfinite(got).all()


# --------------------------------------------------------------------------- closed forms

def _single(L, q_vec, k_rows, v_rows, scale, q_len=1):
    """One request, one kv head, Hq = 1, context given as dense rows."""
    d = q_vec.shape[-1]
    w = wl.sized_case(99, [L], [q_len], 1, 1, d, "f32", scale=scale)
    kc, vc = place_dense([k_rows.reshape(L, 1, d)], [v_rows.reshape(L, 1, d)], w.block_tables, w.num_blocks)
    q = q_vec.reshape(q_len, 1, d)
    return run_oracle(w, q, kc, vc)[:, 0, :]


def test_single_key_returns_its_value_exactly():
    g = torch.Generator().manual_seed(3)
    v = torch.randn((1, 64), generator=g)
    out = _single(1, torch.randn((64,), generator=g), torch.randn((1, 64), generator=g), v, 0.125)
    assert np.array_equal(out[0], v[0].double().numpy())


def test_identical_keys_give_mean_of_values():
    g = torch.Generator().manual_seed(4)
    L = 37
    k = torch.randn((1, 64), generator=g).repeat(L, 1)
    v = torch.randn((L, 64), generator=g)
    out = _single(L, torch.randn((64,), generator=g), k, v, 0.125)
    np.testing.assert_allclose(out[0], v.double().mean(0).numpy(), rtol=0, atol=1e-15)


def test_zero_query_gives_mean_over_visible_keys():
    # prefill chunk of 5 queries after 20 cached tokens, all queries zero:
    # row j sees keys 0..20+j and averages their values
    g = torch.Generator().manual_seed(5)
    L, n_q, d = 25, 5, 16
    k = torch.randn((L, d), generator=g)
    v = torch.randn((L, d), generator=g)
    w = wl.sized_case(7, [L], [n_q], 1, 1, d, "f32")
    kc, vc = place_dense([k.reshape(L, 1, d)], [v.reshape(L, 1, d)], w.block_tables, w.num_blocks)
    out = run_oracle(w, torch.zeros((n_q, 1, d)), kc, vc)[:, 0, :]
    for j in range(n_q):
        np.testing.assert_allclose(out[j], v[:L - n_q + j + 1].double().mean(0).numpy(), atol=1e-15)


def test_two_keys_sigmoid():
    g = torch.Generator().manual_seed(6)
    d = 32
    q, k, v = (torch.randn((d,), generator=g), torch.randn((2, d), generator=g),
               torch.randn((2, d), generator=g))
    scale = 0.3
    out = _single(2, q, k, v, scale)[0]
    s = [float(np.float32(scale)) * float(np.dot(q.double().numpy(), k[t].double().numpy())) for t in range(2)]
    a = 1.0 / (1.0 + math.exp(-(s[0] - s[1])))
    expect = a * v[0].double().numpy() + (1 - a) * v[1].double().numpy()
    np.testing.assert_allclose(out, expect, rtol=1e-13, atol=1e-14)


def test_dominant_logit_selects_its_value():
    g = torch.Generator().manual_seed(7)
    L, d = 50, 16
    k = torch.randn((L, d), generator=g) * 0.01
    q = torch.zeros(d)
    q[0] = 1.0
    k[23, 0] = 10.0
    v = torch.randn((L, d), generator=g)
    out = _single(L, q, k, v, 100.0)[0]        # logit gap ~ 1000 -> weight ratio e^-1000
    assert np.array_equal(out, v[23].double().numpy())


def test_weights_match_scipy_softmax():
    # one-hot values: output coordinate u is exactly the weight of key u
    g = torch.Generator().manual_seed(8)
    L, d = 40, 48
    k = torch.randn((L, d), generator=g)
    q = torch.randn((d,), generator=g)
    v = torch.zeros((L, d))
    v[torch.arange(L), torch.arange(L)] = 1.0
    out = _single(L, q, k, v, 0.2)[0]
    logits = float(np.float32(0.2)) * (k.double().numpy() @ q.double().numpy())
    expect = scipy.special.softmax(logits)
    np.testing.assert_allclose(out[:L], expect, rtol=1e-13, atol=1e-16)
    assert np.all(out[L:] == 0.0)
    assert abs(out.sum() - 1.0) < 1e-15


# --------------------------------------------------------------------------- invariances

def test_permuted_physical_ids_bit_identical():
    w, q, dk, dv = random_dense_case(21, num_seqs=7, max_ctx=90, max_q=35, group=4, hkv=2, d=64)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks)
    base = run_oracle(w, q, kc, vc)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_blocks).astype(np.int32)     # old id -> new id
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[torch.from_numpy(perm).long()] = kc
    vc2[torch.from_numpy(perm).long()] = vc
    got = run_oracle(w, q, kc2, vc2, bt=bt2)
    assert np.array_equal(base, got)


def test_shared_prefix_equals_duplicated_copies_bitwise():
    d, hkv, group = 64, 2, 2
    n_req, prefix_blocks = 4, 3
    g = torch.Generator().manual_seed(9)
    suffix = [5, 16, 23, 1]
    L = [prefix_blocks * BLOCK + s for s in suffix]
    pk = torch.randn((prefix_blocks * BLOCK, hkv, d), generator=g)
    pv = torch.randn((prefix_blocks * BLOCK, hkv, d), generator=g)
    dk = [torch.cat([pk, torch.randn((s, hkv, d), generator=g)]) for s in suffix]
    dv = [torch.cat([pv, torch.randn((s, hkv, d), generator=g)]) for s in suffix]
    nb_each = [(x + BLOCK - 1) // BLOCK for x in L]
    # duplicated: every request owns all of its blocks
    ids = iter(range(1000))
    bt_dup = np.full((n_req, max(nb_each)), -1, np.int32)
    for i, n in enumerate(nb_each):
        bt_dup[i, :n] = [next(ids) for _ in range(n)]
    pool_dup = next(ids)
    # shared: the prefix blocks are one set of physical ids referenced by every table
    bt_sh = np.full_like(bt_dup, -1)
    shared = list(range(prefix_blocks))
    nxt = prefix_blocks
    for i, n in enumerate(nb_each):
        bt_sh[i, :prefix_blocks] = shared
        for j in range(prefix_blocks, n):
            bt_sh[i, j] = nxt
            nxt += 1
    w = wl.sized_case(1, L, [1] * n_req, group * hkv, hkv, d, "f32")
    q = torch.randn((n_req, group * hkv, d), generator=g)
    kc_d, vc_d = place_dense(dk, dv, bt_dup, pool_dup)
    kc_s, vc_s = place_dense(dk, dv, bt_sh, nxt)
    a = oracle.attention(to_bits(q), to_bits(kc_d), to_bits(vc_d), bt_dup, w.seq_lens, w.query_start_loc,
                         w.scale)
    b = oracle.attention(to_bits(q), to_bits(kc_s), to_bits(vc_s), bt_sh, w.seq_lens, w.query_start_loc,
                         w.scale)
    assert np.array_equal(a, b)


def test_mixed_batch_equals_separate_calls():
    w, q, dk, dv = random_dense_case(31, num_seqs=9, max_ctx=70, max_q=30, group=2, hkv=2, d=8)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks)
    whole = run_oracle(w, q, kc, vc)
    qsl = w.query_start_loc
    for i in range(w.num_seqs):
        one = oracle.attention(to_bits(q[qsl[i]:qsl[i + 1]]), to_bits(kc), to_bits(vc),
                               w.block_tables[i:i + 1], w.seq_lens[i:i + 1],
                               np.array([0, qsl[i + 1] - qsl[i]], np.int32), w.scale)
        assert np.array_equal(one, whole[qsl[i]:qsl[i + 1]])


def test_row_subset_matches_full():
    w, q, dk, dv = random_dense_case(32, num_seqs=6, max_ctx=70, max_q=30, group=2, hkv=2, d=8)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks)
    whole = run_oracle(w, q, kc, vc)
    rows = np.array([w.num_tokens - 1, 0, 3, 3], np.int64)
    assert np.array_equal(run_oracle(w, q, kc, vc, rows=rows), whole[rows])


# --------------------------------------------------------------------------- slot mapping + scatter

def test_slot_mapping_round_trip_through_attention():
    # Write a whole context (as one prefill chunk) through slot_mapping + write with
    # one-hot values, zero keys: the last row must average each position's one-hot
    # exactly once, so every coordinate is 1/L.
    L, d = 45, 64
    w = wl.sized_case(12, [L], [L], 1, 1, d, "f32")
    kc = np.full((w.num_blocks, 1, BLOCK, d), np.nan, np.float32)
    vc = np.full_like(kc, np.nan)
    slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc)
    assert len(set(slots.tolist())) == L
    k = np.zeros((L, 1, d), np.float32)
    v = np.zeros((L, 1, d), np.float32)
    v[np.arange(L), 0, np.arange(L)] = 1.0
    oracle.write(k, v, slots, kc, vc)
    out = oracle.attention(np.zeros((L, 1, d), np.float32), kc, vc, w.block_tables, w.seq_lens,
                           w.query_start_loc, 1.0)
    np.testing.assert_allclose(out[-1, 0, :L], np.full(L, 1.0 / L), rtol=1e-15)
    assert np.all(out[-1, 0, L:] == 0)
    # row j sees positions 0..j
    for j in (0, 15, 16, 31):
        np.testing.assert_allclose(out[j, 0, :j + 1], np.full(j + 1, 1.0 / (j + 1)), rtol=1e-15)


def test_slot_mapping_decode_positions():
    # a decode token sits at position seq_len - 1: its slot is inside the table's
    # last used block, at offset (seq_len - 1) mod 16
    w = wl.make("decode")
    slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc)
    for i in range(w.num_seqs):
        p = int(w.seq_lens[i]) - 1
        assert slots[i] // BLOCK == w.block_tables[i, p // BLOCK]
        assert slots[i] % BLOCK == p % BLOCK


def test_write_matches_numpy_scatter_bytes():
    rng = np.random.default_rng(1)
    nb, hkv, d, T = 9, 3, 8, 40
    kc = rng.standard_normal((nb, hkv, BLOCK, d)).astype(np.float32)
    vc = rng.standard_normal((nb, hkv, BLOCK, d)).astype(np.float32)
    k = rng.standard_normal((T, hkv, d)).astype(np.float32)
    v = rng.standard_normal((T, hkv, d)).astype(np.float32)
    slots = rng.permutation(nb * BLOCK)[:T].astype(np.int64)
    slots[[3, 17]] = -1
    ek, ev = kc.copy(), vc.copy()
    for t in range(T):
        if slots[t] >= 0:
            ek[slots[t] // BLOCK, :, slots[t] % BLOCK] = k[t]
            ev[slots[t] // BLOCK, :, slots[t] % BLOCK] = v[t]
    oracle.write(k, v, slots, kc, vc)
    assert kc.tobytes() == ek.tobytes() and vc.tobytes() == ev.tobytes()


def test_copy_blocks_snapshot_semantics():
    rng = np.random.default_rng(2)
    nb, hkv, d = 12, 2, 8
    kc = rng.integers(-30000, 30000, size=(nb, hkv, BLOCK, d)).astype(np.int16)
    vc = rng.integers(-30000, 30000, size=(nb, hkv, BLOCK, d)).astype(np.int16)
    src = np.array([1, 5, 5, 7], np.int32)
    dst = np.array([5, 2, 9, 1], np.int32)     # dst 5 is also a source: must read the old block 5
    ek, ev = kc.copy(), vc.copy()
    ek[dst] = kc[src]
    ev[dst] = vc[src]
    oracle.copy_blocks(src, dst, kc, vc)
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_bad_block_id_is_rejected():
    w, q, dk, dv = random_dense_case(41, num_seqs=3, max_ctx=40, max_q=5, group=1, hkv=1, d=8)
    kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks)
    bt = w.block_tables.copy()
    bt[0, 0] = w.num_blocks
    with pytest.raises(oracle.OracleError):
        run_oracle(w, q, kc, vc, bt=bt)


# --------------------------------------------------------------------------- mutation check

_MUTANTS = {
    # (description, original, replacement)
    "offset-in-block": ("u % ORC_BLOCK) * head_dim;\n        double dot", "(u + 1) % ORC_BLOCK) * head_dim;\n        double dot"),
    "kv-head-index": ("int32_t g = h / group;", "int32_t g = h % num_kv_heads;"),
    "causal-offset": ("int64_t n_keys = p + 1;", "int64_t n_keys = p;"),
    "scale-dropped": ("s[u] = dscale * dot;", "s[u] = dot;"),
    "max-sign": ("double w = exp(s[u] - m);", "double w = exp(m - s[u]);"),
    "value-from-key": ("o[c] += w * orc_load(v_cache, v_base + c, dtype);", "o[c] += w * orc_load(k_cache, v_base + c, dtype);"),
    "transposed-q-index": ("const int64_t q_base = (t * num_q_heads + h) * head_dim;", "const int64_t q_base = (h * (query_start_loc[num_seqs]) + t) * head_dim;"),
    "kv-head-order-in-block": ("int64_t k_base = ((phys * num_kv_heads + g)", "int64_t k_base = ((phys * num_kv_heads + (num_kv_heads - 1 - g))"),
}


@pytest.mark.parametrize("mutant", sorted(_MUTANTS))
def test_planted_mistakes_are_caught(mutant, tmp_path):
    """Compile a copy of the oracle with one planted mistake; the dense-SDPA pin must fail."""
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()
    old, new = _MUTANTS[mutant]
    assert src.count(old) == 1, mutant
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.orc_attention.argtypes = [P, i32, P, P, i64, i32, i32, P, i32, P, P, i32, i32, f32, P, i64, P, i32]
    caught = False
    for seed in (51, 52):
        w, q, dk, dv = random_dense_case(seed, num_seqs=5, max_ctx=60, max_q=25, group=2, hkv=2, d=8)
        kc, vc = place_dense(dk, dv, w.block_tables, w.num_blocks)
        ref = sdpa_reference(q, dk, dv, w.seq_lens, w.query_start_loc, w.scale, 2)
        qa, ka, va = (np.ascontiguousarray(to_bits(x)) for x in (q, kc, vc))
        bt = np.ascontiguousarray(w.block_tables)
        out = np.empty((w.num_tokens, w.num_q_heads, 8))
        rc = lib.orc_attention(qa.ctypes.data, 0, ka.ctypes.data, va.ctypes.data, w.num_blocks, 2, 8,
                               bt.ctypes.data, bt.shape[1], w.seq_lens.ctypes.data,
                               w.query_start_loc.ctypes.data, w.num_seqs, w.num_q_heads, w.scale, None,
                               w.num_tokens, out.ctypes.data, 1)
        if rc != 0 or not np.allclose(out, ref, rtol=1e-12, atol=1e-13, equal_nan=False):
            caught = True
    assert caught, f"mutant {mutant} was not caught by the dense-SDPA pin"
