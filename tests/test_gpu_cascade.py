"""paged_attention_cascade: shared-prefix groups change how the work is done, never
the result.  Every case is checked against the oracle's plain attention (the
definition of paged_attention), and against paged_attention itself.

Shared prefixes come from the "vLLM's PagedAttention" teardown, section
"PagedAttention": requests whose prompt prefix hashes match point at the same
physical blocks.  The cascade attends those blocks once per (group, kv head) for all
members and merges the partial softmax states with each member's own keys.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import bits, compare, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_both(pkv, w, hints, t):
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    args = (t["q"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale, max(1, w.max_query_len), w.max_seq_len)
    plain = pkv.paged_attention(*args)
    cas = pkv.paged_attention_cascade(*args, dev(hints["prefix_block_tables"]), dev(hints["prefix_num_blocks"]),
                                      dev(hints["member_start"]), dev(hints["member_seqs"]))
    st = pkv.pkv_get_last_error()
    return plain, cas, st


@pytest.mark.parametrize("seed,group,hkv", [(1, 4, 2), (2, 8, 1), (3, 16, 1), (4, 6, 2), (5, 1, 4)])
def test_groups_match_the_oracle(pkv, seed, group, hkv):
    w, hints = wl.shared_prefix_case(seed, group=group, num_kv_heads=hkv)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    plain, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)
    compare(plain, ref, "bf16", w.name + " (no groups)")
    # fp32 rounding order differs between the two ways of splitting the keys: close, not equal
    assert (cas.float() - plain.float()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("long_suffix", [2049, 5000])
def test_member_with_split_suffix(pkv, long_suffix):
    # a member whose own keys are cut into several decode splits, merged after the prefix
    w, hints = wl.shared_prefix_case(11, prefix_blocks=(40, 9), members=(7, 5), long_suffix=long_suffix,
                                     bystanders=2, bad_hints=False)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    _, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)


def test_suffix_of_one_key_and_exact_split_boundaries(pkv):
    # prefixes of exactly 32 and 64 blocks (one and two 512-key prefix splits) and
    # members whose context is the prefix plus a single key
    w, hints = wl.shared_prefix_case(12, prefix_blocks=(32, 64), members=(5, 4), max_suffix=1, bystanders=0,
                                     bad_hints=False)
    assert set(w.seq_lens.tolist()) == {32 * 16 + 1, 64 * 16 + 1}
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    _, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)


@pytest.mark.parametrize("group", [4, 8, 16])
def test_long_prefixes_fold_every_prefix_split(pkv, group):
    # prefixes of 5 and 10 prefix splits (2400 and 4800 keys): a member's decode item
    # folds more prefix partials than it stages in shared memory at its start (four
    # for a padded group of 4, two for 8, one for 16), the rest straight from global
    w, hints = wl.shared_prefix_case(17, prefix_blocks=(150, 300), members=(9, 6), group=group, num_kv_heads=1,
                                     bystanders=3, bad_hints=False)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    _, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)


@pytest.mark.parametrize("group,hkv,members", [(4, 8, 70), (8, 4, 100), (16, 2, 120)])
def test_enough_members_for_paired_member_tiles(pkv, group, hkv, members):
    # A 4800-key prefix (10 prefix splits) with enough members that the items of two
    # member tiles each (128 / GP members per tile) are at least one per SM on a 152-SM
    # part -- e.g. 70 members, group 4, 8 kv heads: 2 x 8 x 10 -- so the cascade pairs
    # its member tiles (fewer items would leave SMs idle and use one tile)
    w, hints = wl.shared_prefix_case(18, prefix_blocks=(300,), members=(members,), group=group, num_kv_heads=hkv,
                                     max_suffix=40, bystanders=2, bad_hints=False)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    _, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)


def test_malformed_hints_fall_back(pkv):
    w, hints = wl.shared_prefix_case(13, bad_hints=True)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    G = hints["prefix_num_blocks"].shape[0]
    M = hints["member_seqs"].shape[0]
    assert G == 3
    variants = {
        "decreasing offsets": dict(hints, member_start=np.array([0, M, 2, M], np.int32)),
        "shorter prefix than shared": dict(hints, prefix_num_blocks=np.maximum(1, hints["prefix_num_blocks"] // 2)
                                           .astype(np.int32)),
        "offsets past the list": dict(hints, member_start=np.concatenate([hints["member_start"][:-1], [M + 5]])
                                      .astype(np.int32)),
        "prefix longer than its table": dict(hints, prefix_num_blocks=hints["prefix_num_blocks"] + 500),
        "zero-length prefix": dict(hints, prefix_num_blocks=np.zeros(G, np.int32)),
        "request index out of range": dict(hints, member_seqs=np.where(np.arange(M) % 3 == 0, 10 ** 6, -1 - np.arange(M))
                                           .astype(np.int32)),
    }
    for name, h in variants.items():
        _, cas, st = run_both(pkv, w, h, t)
        assert st == 0, name
        compare(cas, ref, "bf16", name)


def test_bad_prefix_block_zeroes_members_like_paged_attention(pkv):
    w, hints = wl.shared_prefix_case(14, prefix_blocks=(20,), members=(6,), bystanders=2, bad_hints=False)
    bad = w.num_blocks + 7
    pid = hints["prefix_block_tables"][0, 3]
    w.block_tables[w.block_tables == pid] = bad          # every member's table, and the prefix's
    hints["prefix_block_tables"][0, 3] = bad
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    plain, cas, st = run_both(pkv, w, hints, t)
    assert st == pkv.PKV_ERR_INDEX
    members = hints["member_seqs"]
    rows = w.query_start_loc[members]
    assert torch.equal(cas[rows].float(), torch.zeros_like(cas[rows].float()))
    assert torch.equal(plain[rows].float(), torch.zeros_like(plain[rows].float()))
    others = np.setdiff1d(np.arange(w.num_tokens), rows)
    assert (cas[others].float() - plain[others].float()).abs().max().item() <= 2e-2


def test_repeated_calls_are_bitwise_equal(pkv):
    w, hints = wl.shared_prefix_case(15, prefix_blocks=(64, 17), members=(70, 33), bystanders=8)
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    _, a, st = run_both(pkv, w, hints, t)
    _, b, st2 = run_both(pkv, w, hints, t)
    assert st == 0 and st2 == 0
    assert torch.equal(a, b)


def test_prefix_workload_with_its_group(pkv):
    """The prefix-shared workload at full size: 256 decodes, one 64-block prefix, CoW
    copies and writes first; every output row checked against the oracle."""
    w = wl.make("prefix")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    pkv.pkv_copy_blocks(dev(w.cow_src), dev(w.cow_dst), t["k_cache"], t["v_cache"])
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    slots = pkv.pkv_slot_mapping(bt, sl, qsl, w.num_tokens)
    pkv.pkv_write(t["k_new"], t["v_new"], slots, t["k_cache"], t["v_cache"])
    pid = w.notes["shared_prefix_ids"]
    out = pkv.paged_attention_cascade(t["q"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale, 1, w.max_seq_len,
                                      dev(pid[None, :]), dev(np.array([pid.size], np.int32)),
                                      dev(np.array([0, w.num_seqs], np.int32)),
                                      dev(np.arange(w.num_seqs, dtype=np.int32)))
    assert pkv.pkv_get_last_error() == 0
    ref, _, _, _ = oracle_step(w, t_cpu, cow=True)
    compare(out, ref, "bf16", "prefix")


def test_cascade_step_replays_from_a_cuda_graph(pkv):
    w, hints = wl.shared_prefix_case(16, prefix_blocks=(48,), members=(40,), bystanders=4)
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    h = {k: dev(v) for k, v in hints.items()}
    out_e = torch.empty_like(t["q"])
    out_g = torch.full_like(t["q"], float("nan"))

    def call(out):
        pkv.paged_attention_cascade(t["q"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale,
                                    max(1, w.max_query_len), w.max_seq_len, h["prefix_block_tables"],
                                    h["prefix_num_blocks"], h["member_start"], h["member_seqs"], out=out)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(out_e)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(out_g)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(out_g, out_e)


@pytest.mark.parametrize("prefix_blocks", [(520, 7), (513, 513)])
def test_long_prefixes_take_the_global_membership_checks(pkv, prefix_blocks):
    # a prefix table longer than 512 blocks makes the planner check membership in
    # global memory instead of shared memory; with the bad hints of
    # shared_prefix_case (a chunk, a context inside the prefix, a request listed
    # twice, a table of its own) the result is the same as without groups
    w, hints = wl.shared_prefix_case(13, prefix_blocks=prefix_blocks, members=(4, 3), max_suffix=200, bystanders=3)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    plain, cas, st = run_both(pkv, w, hints, t)
    assert st == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(cas, ref, "bf16", w.name)
    compare(plain, ref, "bf16", w.name + " (no groups)")
