"""Host side of the serving loop, on the CPU: block tables, prefix reuse, fork and
copy-on-write from the block manager, applied to the oracle's pool, must leave every
live request able to read exactly its own tokens' K/V rows through its table."""
import numpy as np
import pytest

import oracle
import serving_sim as sim
from helpers import bits


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_248_gb300 import _build
    _build.build()
    import paged_kv_cache_248_gb300 as m
    return m


@pytest.mark.parametrize("budget", [160, 37])
def test_every_request_reads_its_own_rows(pkv, budget):
    hkv, d, nb = 2, 16, 96
    bm = pkv.BlockManager(nb)
    kc = np.zeros((nb, hkv, sim.BLOCK, d), np.int16)      # bf16 bit patterns
    vc = np.zeros_like(kc)
    ev = {}
    steps = 0
    for st in sim.run(bm, hkv, d, steps=16, budget=budget, events=ev):
        if st.cow_src.size:
            oracle.copy_blocks(st.cow_src, st.cow_dst, kc, vc)
        slots = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
        assert len(set(slots.tolist())) == slots.size     # no two new tokens share a slot
        oracle.write(bits(st.k_new), bits(st.v_new), slots, kc, vc)
        for rid, (table, toks) in st.live.items():
            want_k, want_v = sim.kv_rows(toks, range(len(toks)), hkv, d)
            assert np.array_equal(sim.gather(kc, table, len(toks)), bits(want_k)), (st.index, rid)
            assert np.array_equal(sim.gather(vc, table, len(toks)), bits(want_v)), (st.index, rid)
        steps += 1
    assert steps >= 10
    assert ev["prefix_hit"] == 3 and ev["shared_with_a"]  # the system prompt's full blocks
    assert ev["forked"] and ev["cow"] >= 1                # the sample diverged by copy-on-write
    assert ev["finished"] >= 1


def test_without_copy_on_write_the_sibling_is_corrupted(pkv):
    """The same loop with the block copies skipped (a planted mistake, on the host):
    the parent and its sample write into one shared block and one of them reads the
    other's row, which the invariant above must catch."""
    hkv, d, nb = 2, 16, 96
    bm = pkv.BlockManager(nb)
    kc = np.zeros((nb, hkv, sim.BLOCK, d), np.int16)
    vc = np.zeros_like(kc)
    caught = False
    for st in sim.run(bm, hkv, d):
        if st.cow_src.size:
            # skip the copy and point the writer back at the shared block
            for s, dd in zip(st.cow_src, st.cow_dst):
                st.block_tables[st.block_tables == dd] = s
                for rid, (table, toks) in st.live.items():
                    st.live[rid] = ([int(s) if b == dd else b for b in table], toks)
        slots = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
        oracle.write(bits(st.k_new), bits(st.v_new), slots, kc, vc)
        for rid, (table, toks) in st.live.items():
            want_k, _ = sim.kv_rows(toks, range(len(toks)), hkv, d)
            if not np.array_equal(sim.gather(kc, table, len(toks)), bits(want_k)):
                caught = True
    assert caught
