"""Input-generator checks and the golden fixtures (CPU only)."""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
BLOCK = 16


@pytest.mark.parametrize("name", wl.NAMES)
def test_tables_hold_ceil_len_over_16_valid_entries(name):
    # allocate_slots hands out ceil(new_tokens / 16) blocks (teardown, "PagedAttention")
    w = wl.make(name)
    for i in range(w.num_seqs):
        n = (int(w.seq_lens[i]) + BLOCK - 1) // BLOCK
        row = w.block_tables[i]
        assert np.all(row[:n] >= 0) and np.all(row[:n] < w.num_blocks)
        assert np.all(row[n:] == -1)


@pytest.mark.parametrize("name", ["tiny", "decode", "mixed", "long"])
def test_blocks_are_private_when_not_shared(name):
    w = wl.make(name)
    ids = w.block_tables[w.block_tables >= 0]
    assert len(np.unique(ids)) == len(ids)


def test_workload_shapes():
    t = wl.make("tiny")
    assert t.seq_lens.tolist() == [5, 16, 17, 40] and t.num_tokens == 4 and t.num_blocks == 16
    assert (t.num_q_heads, t.num_kv_heads, t.head_dim, t.dtype) == (2, 1, 64, "f32")
    d = wl.make("decode")
    assert d.num_seqs == 64 and d.seq_lens.min() >= 128 and d.seq_lens.max() <= 4096
    m = wl.make("mixed")
    assert m.num_tokens == 8192 and m.num_seqs == 8 + 4096
    assert np.all(m.q_lens[:8] == 512) and np.all(m.q_lens[8:] == 1)
    assert np.all(m.seq_lens[:8] >= 512) and np.all(m.seq_lens[:8] <= 3072 + 512)
    assert m.seq_lens[8:].min() >= 256 and m.seq_lens[8:].max() <= 2048
    lg = wl.make("long")
    assert np.all(lg.seq_lens == 32768) and lg.block_tables.shape == (32, 2048)
    assert (lg.num_q_heads, lg.num_kv_heads) == (64, 8)


def test_prefix_workload_shares_and_copies():
    w = wl.make("prefix")
    shared = w.notes["shared_prefix_ids"]
    assert len(shared) == 64
    before = w.block_tables_before_cow
    assert np.all(before[:, :64] == shared[None, :])          # one set of physical ids for all
    assert np.all(w.block_tables[:, :64] == shared[None, :])
    last = (w.seq_lens - 1) // BLOCK
    assert np.array_equal(before[np.arange(w.num_seqs), last], w.cow_src)
    assert np.array_equal(w.block_tables[np.arange(w.num_seqs), last], w.cow_dst)
    # copies land in fresh blocks, distinct and never a source
    assert len(np.unique(w.cow_dst)) == w.num_seqs
    assert not set(w.cow_dst.tolist()) & set(before[before >= 0].tolist())


def test_same_seed_same_inputs():
    a = wl.make("tiny").make_tensors("cpu")
    b = wl.make("tiny").make_tensors("cpu")
    for k in a:
        assert a[k].equal(b[k])


def test_page_fact_block_counts_via_slot_mapping():
    # the teardown's two examples: a 2,000-token prompt and a 500th generated token;
    # writing all their positions touches ceil(tokens / 16) distinct blocks
    facts = json.load(open(os.path.join(HERE, "golden", "page_facts.json")))
    assert facts["block_size"] == BLOCK
    for ex in facts["examples"]:
        n = ex["tokens"]
        w = wl.sized_case(3, [n], [n], 1, 1, 8, "f32")
        slots = oracle.slot_mapping(w.block_tables, w.seq_lens, w.query_start_loc)
        assert len(np.unique(slots // BLOCK)) == ex["blocks"]
        assert len(np.unique(slots)) == n


def test_golden_tiny_decode():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    ref = np.load(os.path.join(HERE, "golden", "tiny_decode.npz"))
    now = mg.compute()
    for k in ref.files:
        assert np.array_equal(ref[k], now[k]), k
