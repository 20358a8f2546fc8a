"""paged_attention_step: slot mapping, K/V scatter and attention in one call must
give exactly what pkv_slot_mapping + pkv_write + paged_attention(_cascade) give --
the same caches, slots and outputs, bit for bit -- and match the oracle.

The step appends every running request's new tokens to its blocks and attends
over them ("vLLM's PagedAttention" teardown, section "Continuous batching").
"""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import bits, compare, oracle_step, sub_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def both_ways(pkv, w, t, groups=None):
    """(separate: out, slots, k, v, status), (fused: ...) on two copies of the caches."""
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    mq, ms = max(1, w.max_query_len), max(1, w.max_seq_len)
    res = []
    for fused in (False, True):
        kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
        slots = torch.full((w.num_tokens,), -7, dtype=torch.int64, device="cuda")
        if fused:
            out = pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], kc, vc, bt, sl, qsl, w.scale, mq, ms,
                                           prefix_groups=groups, slot_mapping=slots)
        else:
            pkv.pkv_slot_mapping(bt, sl, qsl, w.num_tokens, out=slots)
            pkv.pkv_write(t["k_new"], t["v_new"], slots, kc, vc)
            if groups is None:
                out = pkv.paged_attention(t["q"], kc, vc, bt, sl, qsl, w.scale, mq, ms)
            else:
                out = pkv.paged_attention_cascade(t["q"], kc, vc, bt, sl, qsl, w.scale, mq, ms, *groups)
        res.append((out, slots, kc, vc, pkv.pkv_get_last_error()))
    return res


def assert_same(a, b):
    for x, y, name in zip(a, b, ("out", "slots", "k_cache", "v_cache", "status")):
        if isinstance(x, torch.Tensor):
            assert torch.equal(x, y), name
        else:
            assert x == y, name


@pytest.mark.parametrize("seed,group,hkv,dtype", [(21, 4, 2, "bf16"), (22, 8, 2, "bf16"), (23, 16, 1, "bf16"),
                                                  (24, 6, 2, "bf16"), (25, 2, 2, "f32")])
def test_step_equals_the_separate_calls_and_the_oracle(pkv, seed, group, hkv, dtype):
    d = 128 if dtype == "bf16" else 64
    w = wl.random_case(seed, num_seqs=14, max_ctx=1400, max_q=260, group=group, num_kv_heads=hkv, head_dim=d,
                       dtype=dtype)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways(pkv, w, t)
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, ref_slots, ref_k, ref_v = oracle_step(w, t_cpu)
    assert np.array_equal(fus[1].cpu().numpy(), ref_slots)
    compare(fus[0], ref, dtype, w.name)


def hint_tensors(hints):
    return tuple(dev(hints[k]) for k in ("prefix_block_tables", "prefix_num_blocks", "member_start", "member_seqs"))


def test_step_with_prefix_groups(pkv):
    # no new token lands in a prefix block: the fused step admits the same members as
    # the separate calls and gives the same bits
    w, hints = wl.shared_prefix_case(26, prefix_blocks=(24, 40), members=(20, 9), bystanders=6, bad_hints=False)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways(pkv, w, t, hint_tensors(hints))
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, _, _, _ = oracle_step(w, t_cpu)
    compare(fus[0], ref, "bf16", w.name)


def caches_same_outputs_match(sep, fus, ref, name):
    assert sep[4] == 0 and fus[4] == 0
    for x, y, what in zip(sep[1:4], fus[1:4], ("slots", "k_cache", "v_cache")):
        assert torch.equal(x, y), what
    compare(sep[0], ref, "bf16", name + " (separate calls)")
    compare(fus[0], ref, "bf16", name + " (fused step)")


def test_step_with_a_new_token_in_a_prefix_block(pkv):
    # the bad hints list a decode whose context ends inside prefix 0, so its new token
    # is written into one of the shared prefix blocks.  The fused step's cascade reads
    # the prefix while the tokens are being written, so the step then lets every member
    # attend its whole context in the decode kernel: the caches and slots are the
    # separate calls' bit for bit, and both outputs match the oracle
    w, hints = wl.shared_prefix_case(26, prefix_blocks=(24, 40), members=(20, 9), bystanders=6)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    inside = [i for i in range(w.num_seqs) if w.q_lens[i] == 1 and w.seq_lens[i] < 24 * 16
              and w.block_tables[i, 0] == hints["prefix_block_tables"][0, 0]]
    assert inside, "the case has a decode that writes into prefix 0"
    sep, fus = both_ways(pkv, w, t, hint_tensors(hints))
    ref, _, _, _ = oracle_step(w, t_cpu)
    caches_same_outputs_match(sep, fus, ref, w.name)


def test_step_with_a_bystander_writing_into_a_prefix(pkv):
    # a decode that is no member has its newest block pointed at a block of the
    # shared prefix: its new token overwrites a row every member attends
    w, hints = wl.shared_prefix_case(29, prefix_blocks=(30,), members=(25,), bystanders=6, bad_hints=False)
    members = set(hints["member_seqs"].tolist())
    i = next(i for i in range(w.num_seqs) if i not in members and w.q_lens[i] == 1)
    last = (int(w.seq_lens[i]) - 1) // 16
    w.block_tables[i, last] = hints["prefix_block_tables"][0, 7]
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways(pkv, w, t, hint_tensors(hints))
    ref, _, _, _ = oracle_step(w, t_cpu)
    caches_same_outputs_match(sep, fus, ref, w.name)


def test_step_errors_match_the_separate_calls(pkv):
    # a new token whose block id is past the pool: the write is skipped and flagged,
    # attention zeroes the request's rows -- the same on both paths
    w = wl.random_case(27, num_seqs=6, max_ctx=300, max_q=40, group=4, num_kv_heads=2, head_dim=128, dtype="bf16")
    i = int(np.argmax(w.q_lens))
    last = (int(w.seq_lens[i]) - 1) // 16
    w.block_tables[i, last] = w.num_blocks + 3
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    sep, fus = both_ways(pkv, w, t)
    assert sep[4] == pkv.PKV_ERR_INDEX
    assert_same(sep, fus)


def test_mixed_workload_full_size(pkv):
    """The 8192-token mixed step (21 GB pool, two copies): fused and separate agree bit
    for bit; two chunks and 64 decodes, with only their blocks, match the oracle."""
    w = wl.make("mixed")
    t = w.make_tensors("cuda")
    seq_ids = np.concatenate([[1, 6], 8 + np.random.default_rng(5).choice(4096, size=64, replace=False)])
    w2, t_sub, rows = sub_batch(w, t, seq_ids)  # host copies taken before the step writes
    sep, fus = both_ways(pkv, w, t)
    assert sep[4] == 0
    assert_same(sep, fus)
    del sep, t
    ref, _, _, _ = oracle_step(w2, t_sub)
    compare(fus[0][torch.from_numpy(rows).cuda()], ref, "bf16", "mixed sub-batch")


def test_step_replays_from_a_cuda_graph(pkv):
    w = wl.random_case(28, num_seqs=20, max_ctx=2500, max_q=300, group=4, num_kv_heads=8, head_dim=128,
                       dtype="bf16")
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    kc0, vc0 = t["k_cache"].clone(), t["v_cache"].clone()
    out_e, out_g = torch.empty_like(t["q"]), torch.full_like(t["q"], float("nan"))

    def call(out):
        pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale,
                                 w.max_query_len, w.max_seq_len, out=out)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(out_e)
    s.synchronize()
    k_after, v_after = t["k_cache"].clone(), t["v_cache"].clone()
    t["k_cache"].copy_(kc0)
    t["v_cache"].copy_(vc0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(out_g)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(out_g, out_e)
    assert torch.equal(t["k_cache"], k_after) and torch.equal(t["v_cache"], v_after)


def both_ways_cow(pkv, w, t, src, dst, groups=None):
    """pkv_copy_blocks then paged_attention_step, and paged_attention_step with the
    copies in the same call, on two copies of the caches: (out, slots, k, v, status) each."""
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    s, d = dev(np.asarray(src, np.int32)), dev(np.asarray(dst, np.int32))
    mq, ms = max(1, w.max_query_len), max(1, w.max_seq_len)
    res = []
    for fused in (False, True):
        kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
        slots = torch.full((w.num_tokens,), -7, dtype=torch.int64, device="cuda")
        if not fused:
            pkv.pkv_copy_blocks(s, d, kc, vc)
        out = pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], kc, vc, bt, sl, qsl, w.scale, mq, ms,
                                       prefix_groups=groups, slot_mapping=slots, cow=(s, d) if fused else None)
        res.append((out, slots, kc, vc, pkv.pkv_get_last_error()))
    return res


def test_step_with_copies_on_the_prefix_workload(pkv):
    """The prefix-shared workload with its copy-on-write pairs handed to the step:
    bit-equal to pkv_copy_blocks followed by the step, and every row matches the oracle."""
    w = wl.make("prefix")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    pid = w.notes["shared_prefix_ids"]
    groups = (dev(pid[None, :]), dev(np.array([pid.size], np.int32)), dev(np.array([0, w.num_seqs], np.int32)),
              dev(np.arange(w.num_seqs, dtype=np.int32)))
    sep, fus = both_ways_cow(pkv, w, t, w.cow_src, w.cow_dst, groups)
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, ref_slots, _, _ = oracle_step(w, t_cpu, cow=True)
    assert np.array_equal(fus[1].cpu().numpy(), ref_slots)
    compare(fus[0], ref, "bf16", "prefix with copies in the step")


def test_step_with_a_copy_into_a_prefix_block(pkv):
    # a copy whose destination is one of the shared prefix blocks (the copy rewrites a
    # block every member attends): the step's cascade could read it mid-copy, so the
    # step lets every member attend its whole context itself; caches equal the separate
    # calls' bit for bit and both outputs match the oracle
    w, hints = wl.shared_prefix_case(31, prefix_blocks=(20,), members=(30,), bystanders=6, bad_hints=False)
    members = set(hints["member_seqs"].tolist())
    i = next(i for i in range(w.num_seqs) if i not in members)
    src = np.array([w.block_tables[i, 0]], np.int32)
    dst = np.array([hints["prefix_block_tables"][0, 4]], np.int32)
    w.cow_src, w.cow_dst = src, dst
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways_cow(pkv, w, t, src, dst, hint_tensors(hints))
    ref, _, _, _ = oracle_step(w, t_cpu, cow=True)
    caches_same_outputs_match(sep, fus, ref, w.name)


@pytest.mark.parametrize("seed,dtype", [(32, "bf16"), (33, "f32")])
def test_step_with_copies_equals_the_separate_calls(pkv, seed, dtype):
    # copies into blocks no table names yet: the caches show them, the outputs do not
    d = 128 if dtype == "bf16" else 64
    w = wl.random_case(seed, num_seqs=12, max_ctx=900, max_q=200, group=4, num_kv_heads=2, head_dim=d, dtype=dtype,
                       pool_slack=9)
    used = np.unique(w.block_tables[w.block_tables >= 0])
    free = np.setdiff1d(np.arange(w.num_blocks), used)
    assert free.size >= 4
    src, dst = used[:4].astype(np.int32), free[:4].astype(np.int32)
    w.cow_src, w.cow_dst = src, dst
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways_cow(pkv, w, t, src, dst)
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, _, ref_k, ref_v = oracle_step(w, t_cpu, cow=True)
    compare(fus[0], ref, dtype, w.name)
    # the pools after the copies and the writes (the writes may land in a copy's source)
    for got, want, name in ((fus[2], ref_k, "k_cache"), (fus[3], ref_v, "v_cache")):
        assert np.array_equal(bits(got), want), name


def test_step_with_copies_replays_from_a_cuda_graph(pkv):
    # the copy launch, the planner that overlaps it and the cascade pass beside the
    # planner, captured once and replayed: the same bits as the eager call
    w, hints = wl.shared_prefix_case(34, prefix_blocks=(24,), members=(40,), bystanders=4, bad_hints=False)
    used = np.unique(w.block_tables[w.block_tables >= 0])
    free = np.setdiff1d(np.arange(w.num_blocks), used)
    src, dst = dev(used[-3:].astype(np.int32)), dev(free[:3].astype(np.int32))
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    groups = hint_tensors(hints)
    kc0, vc0 = t["k_cache"].clone(), t["v_cache"].clone()
    out_e, out_g = torch.empty_like(t["q"]), torch.full_like(t["q"], float("nan"))

    def call(out):
        pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale,
                                 max(1, w.max_query_len), w.max_seq_len, prefix_groups=groups, out=out,
                                 cow=(src, dst))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(out_e)
    s.synchronize()
    k_after, v_after = t["k_cache"].clone(), t["v_cache"].clone()
    t["k_cache"].copy_(kc0)
    t["v_cache"].copy_(vc0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(out_g)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(out_g, out_e)
    assert torch.equal(t["k_cache"], k_after) and torch.equal(t["v_cache"], v_after)


@pytest.mark.parametrize("seed,group,hkv,d", [(41, 2, 2, 64), (42, 12, 1, 64), (43, 4, 2, 128)])
def test_fp32_one_token_step_writes_in_the_attention_launch(pkv, seed, group, hkv, d):
    """An fp32 step whose requests each bring one token stores the rows in the attention
    launch itself (each CTA its own token's rows; a group of 12 gives two head chunks
    that both write them): bit-equal to the separate calls, and the oracle's slots,
    caches and outputs."""
    w = wl.random_case(seed, num_seqs=12, max_ctx=700, group=group, num_kv_heads=hkv, head_dim=d, dtype="f32",
                       decode_frac=1.0)
    assert w.max_query_len == 1
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways(pkv, w, t)
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, ref_slots, ref_k, ref_v = oracle_step(w, t_cpu)
    assert np.array_equal(fus[1].cpu().numpy(), ref_slots)
    compare(fus[0], ref, "f32", w.name)
    for got, want, name in ((fus[2], ref_k, "k_cache"), (fus[3], ref_v, "v_cache")):
        assert np.array_equal(bits(got), want), name


def test_fp32_one_token_step_with_copies(pkv):
    w = wl.random_case(44, num_seqs=10, max_ctx=600, group=4, num_kv_heads=2, head_dim=64, dtype="f32",
                       decode_frac=1.0, pool_slack=9)
    used = np.unique(w.block_tables[w.block_tables >= 0])
    free = np.setdiff1d(np.arange(w.num_blocks), used)
    src, dst = used[:4].astype(np.int32), free[:4].astype(np.int32)
    w.cow_src, w.cow_dst = src, dst
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    sep, fus = both_ways_cow(pkv, w, t, src, dst)
    assert sep[4] == 0
    assert_same(sep, fus)
    ref, _, ref_k, ref_v = oracle_step(w, t_cpu, cow=True)
    compare(fus[0], ref, "f32", w.name)
    for got, want, name in ((fus[2], ref_k, "k_cache"), (fus[3], ref_v, "v_cache")):
        assert np.array_equal(bits(got), want), name


def test_fp32_one_token_step_errors_match_the_separate_calls(pkv):
    # a new token whose block id is past the pool: the slot is reported, the write
    # skipped and flagged, and attention zeroes the request's row -- as the separate calls
    w = wl.random_case(45, num_seqs=6, max_ctx=300, group=2, num_kv_heads=2, head_dim=64, dtype="f32",
                       decode_frac=1.0)
    i = 3
    w.block_tables[i, (int(w.seq_lens[i]) - 1) // 16] = w.num_blocks + 3
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    sep, fus = both_ways(pkv, w, t)
    assert sep[4] == pkv.PKV_ERR_INDEX
    assert_same(sep, fus)


def test_fp32_step_flags_a_request_past_the_one_token_bound(pkv):
    # max_query_len 1 with a two-token request: that request is flagged, its rows are
    # zeroed and its tokens not written; the other requests are attended as usual
    w = wl.sized_case(46, seq_lens=[20, 33, 7], q_lens=[1, 2, 1], num_q_heads=2, num_kv_heads=1, head_dim=64,
                      dtype="f32")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    out = pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], kc, vc, bt, sl, qsl, w.scale, 1, w.max_seq_len)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    ref, ref_slots, _, _ = oracle_step(w, t_cpu)
    got = out.cpu().numpy()
    assert not got[1:3].any()
    compare(out[[0, 3]], ref[[0, 3]], "f32", w.name)
    kb, vb = bits(kc), bits(vc)
    k0, v0 = bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"])
    for tok in (1, 2):  # the two-token request's slots keep what they held
        b, off = divmod(int(ref_slots[tok]), 16)
        assert np.array_equal(kb[b, :, off], k0[b, :, off]) and np.array_equal(vb[b, :, off], v0[b, :, off])
