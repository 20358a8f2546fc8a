"""The benchmark's work accounting, checked by brute force on small batches (CPU).

bench.py divides algorithmic bytes and flops by measured times, and extrapolates the
one-core oracle time by multiply-adds; these must count exactly the visible
(query, key) pairs of the causal definition (a query at position p sees keys 0..p)
and each visible token's K and V once.
"""
import numpy as np
import pytest

import bench
import workloads as wl


def brute_pairs(w):
    """Visible (query row, key) pairs, one row at a time."""
    qsl, L = w.query_start_loc, w.seq_lens
    per_row = []
    for i in range(w.num_seqs):
        q = qsl[i + 1] - qsl[i]
        for j in range(q):
            pos = int(L[i]) - int(q) + j
            per_row.append(pos + 1)
    return np.array(per_row, np.int64)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_row_macs_and_flops_count_the_visible_pairs(seed):
    w = wl.random_case(seed, num_seqs=9, max_ctx=300, max_q=70, group=4, num_kv_heads=2, head_dim=64)
    pairs = brute_pairs(w)
    per_pair = 2 * w.head_dim * w.num_q_heads
    assert bench.row_macs(w) == int(pairs.sum()) * per_pair
    rows = np.array([0, 3, len(pairs) - 1])
    assert bench.row_macs(w, rows) == int(pairs[rows].sum()) * per_pair
    f = bench.algorithmic_flops(w)
    ql = w.q_lens
    is_pre = np.repeat(ql > 1, ql)
    assert f["prefill"] == 2 * int(pairs[is_pre].sum()) * per_pair
    assert f["decode"] == 2 * int(pairs[~is_pre].sum()) * per_pair


def test_algorithmic_bytes_count_each_visible_token_once():
    w = wl.random_case(4, num_seqs=7, max_ctx=200, max_q=40, group=2, num_kv_heads=2, head_dim=64)
    b = bench.algorithmic_bytes(w)
    kv_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    ql, L = w.q_lens, w.seq_lens.astype(np.int64)
    assert b["decode_kv"] == int(L[ql == 1].sum()) * kv_tok
    q_bytes = w.num_q_heads * w.head_dim * w.elem_bytes
    tables = int(((L + 15) // 16 * 4).sum())
    assert b["total"] == int(L.sum()) * kv_tok + 2 * w.num_tokens * q_bytes + tables


def test_prefix_workload_counts_the_shared_prefix_once():
    w = wl.make("prefix")
    b = bench.algorithmic_bytes(w)
    kv_tok = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    P = w.notes["prefix_blocks"] * 16
    assert b["decode_kv"] == (P + int((w.seq_lens.astype(np.int64) - P).sum())) * kv_tok
