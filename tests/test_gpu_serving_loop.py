"""The serving loop of tests/serving_sim.py on the GPU path.

The host block manager produces each step's block tables, with a shared system
prompt found by chained hashes, chunked prefills and decodes in one batch, and a
forked parallel sample diverging by copy-on-write.  Every step runs the block copies,
slot mapping, KV scatter and attention through the C ABI; the oracle replays the
same copies and writes on its own copy of the pool.  The pools must stay bit-equal
and the attention output must match the oracle's on every row.
"""
import numpy as np
import pytest
import torch

import oracle
import serving_sim as sim
from helpers import bits, compare

pytestmark = pytest.mark.gpu
HQ, HKV, D = 16, 4, 128


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


@pytest.mark.parametrize("budget,mode", [(160, "calls"), (37, "calls"), (160, "step"), (37, "step")])
def test_serving_loop(pkv, budget, mode):
    """mode "calls": slot mapping, write and attention as separate calls; "step": one
    paged_attention_step per step with the shared-prefix groups the block manager finds
    in the batch (the system prompt's blocks, and a forked sample's)."""
    nb = 256
    bm = pkv.BlockManager(nb)
    kc = torch.zeros((nb, HKV, sim.BLOCK, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ok, ov = bits(kc), bits(vc)                           # the oracle's own pool
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    scale = 1 / np.sqrt(D)
    ev = {}
    n_groups = 0
    for st in sim.run(bm, HKV, D, steps=16, budget=budget, events=ev):
        if st.cow_src.size:
            pkv.pkv_copy_blocks(dev(st.cow_src), dev(st.cow_dst), kc, vc)
            oracle.copy_blocks(st.cow_src, st.cow_dst, ok, ov)
        q = torch.randn((st.num_tokens, HQ, D), generator=torch.Generator().manual_seed(st.index)).bfloat16()
        bt, sl, qsl = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
        max_q, max_l = int(np.diff(st.query_start_loc).max()), int(st.seq_lens.max())
        if mode == "calls":
            slots = pkv.pkv_slot_mapping(bt, sl, qsl, st.num_tokens)
            pkv.pkv_write(st.k_new.cuda(), st.v_new.cuda(), slots, kc, vc)
            out = pkv.paged_attention(q.cuda(), kc, vc, bt, sl, qsl, scale, max_q, max_l)
        else:
            groups = bm.prefix_groups(st.rids, max_prefix_blocks=st.block_tables.shape[1])
            n_groups += len(groups[1])
            slots = torch.empty(st.num_tokens, dtype=torch.int64, device="cuda")
            out = pkv.paged_attention_step(q.cuda(), st.k_new.cuda(), st.v_new.cuda(), kc, vc, bt, sl, qsl, scale,
                                           max_q, max_l, prefix_groups=tuple(dev(g) for g in groups),
                                           slot_mapping=slots)
        assert pkv.pkv_get_last_error() == 0
        ref_slots = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
        assert np.array_equal(slots.cpu().numpy(), ref_slots)
        oracle.write(bits(st.k_new), bits(st.v_new), ref_slots, ok, ov)
        assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov), f"pool differs at step {st.index}"
        ref = oracle.attention(bits(q), ok, ov, st.block_tables, st.seq_lens, st.query_start_loc, scale)
        compare(out, ref, "bf16", f"step {st.index}")
    assert ev["prefix_hit"] == 3 and ev["forked"] and ev["cow"] >= 1
    if mode == "step":
        assert n_groups >= 4  # steps whose batch shared prefix blocks
