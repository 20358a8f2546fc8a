"""paged_attention on the GPU against the fp64 oracle.

Small seeded batches (oracle runs in seconds) span several 128-key tiles, several
query tiles and ragged tails; the five named workloads run at full size, checked
on every output row where the oracle is quick (tiny, decode, prefix) and on
sampled requests where it is not (mixed, long).  Bitwise invariances (block-id
permutation, shared vs duplicated prefix, mixed batch vs separate calls) compare
the GPU with itself.  Tolerances: bf16 max-abs 2e-2 and mean-abs 2e-3, fp32 1e-4.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import bits, compare, gpu_step, oracle_step, sub_batch, to_gpu_meta

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def run_pair(pkv, w, rows=None, cow=False):
    t_cpu = w.make_tensors("cpu")
    t_gpu = {k: v.cuda() for k, v in t_cpu.items()}
    out, slots, st = gpu_step(pkv, w, t_gpu, cow=cow)
    assert st == 0, pkv.status_string(st)
    ref, ref_slots, _, _ = oracle_step(w, t_cpu, rows=rows, cow=cow)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    got = out if rows is None else out[torch.from_numpy(np.asarray(rows)).cuda()]
    return compare(got, ref, w.dtype, w.name)


def test_tiny_decode_f32(pkv):
    run_pair(pkv, wl.make("tiny"))


@pytest.mark.parametrize("seed,group,hkv,d", [(1, 2, 1, 64), (2, 1, 2, 64), (3, 4, 2, 128), (4, 8, 1, 64),
                                              (5, 16, 1, 128), (6, 3, 2, 64)])
def test_random_mixed_f32(pkv, seed, group, hkv, d):
    w = wl.random_case(seed, num_seqs=9, max_ctx=300, max_q=70, group=group, num_kv_heads=hkv, head_dim=d)
    run_pair(pkv, w)


@pytest.mark.parametrize("seed,group,hkv", [(11, 4, 2), (12, 8, 1), (13, 1, 4), (14, 2, 2), (15, 16, 1),
                                            (16, 4, 8)])
def test_random_mixed_bf16(pkv, seed, group, hkv):
    # contexts up to 700 keys (several 128-key tiles), chunks up to 300 queries (several
    # query tiles), ragged everywhere
    w = wl.random_case(seed, num_seqs=8, max_ctx=700, max_q=300, group=group, num_kv_heads=hkv,
                       head_dim=128, dtype="bf16")
    run_pair(pkv, w)


@pytest.mark.parametrize("lens", [[1], [16], [17], [128], [129], [255, 256, 257], [1024, 1, 2049],
                                  [2047, 2048, 4097, 3073]])
def test_decode_edge_lengths_bf16(pkv, lens):
    w = wl.sized_case(21, lens, [1] * len(lens), 32, 8, 128, "bf16")
    run_pair(pkv, w)


@pytest.mark.parametrize("lens,qs", [([16], [16]), ([1], [1]), ([300], [300]), ([129, 40], [128, 40]),
                                     ([500, 33], [257, 2])])
def test_prefill_edge_lengths_bf16(pkv, lens, qs):
    w = wl.sized_case(22, lens, qs, 32, 8, 128, "bf16")
    run_pair(pkv, w)


@pytest.mark.parametrize("scale", [-0.0884, -0.5])
def test_negative_scale_bf16(pkv, scale):
    # a negative scale flips which key is each row's largest logit; the kernels take the
    # tile minimum of the raw scores then (the API accepts any finite scale)
    w = dataclasses.replace(wl.random_case(41, num_seqs=10, max_ctx=900, max_q=300, group=4, num_kv_heads=2,
                                           head_dim=128, dtype="bf16"), scale=scale)
    run_pair(pkv, w)


@pytest.mark.parametrize("scale", [0.3, 1.0])
def test_prefill_rescale_path_bf16(pkv, scale):
    # a large logit scale makes row maxima jump between key tiles, so the prefill
    # kernel's conditional rescale of the TMEM accumulator runs many times
    w = wl.sized_case(24, [900, 700, 130], [300, 200, 129], 32, 8, 128, "bf16", scale=scale)
    run_pair(pkv, w)


@pytest.mark.parametrize("group,hkv", [(1, 8), (2, 4), (3, 2), (4, 8), (5, 1), (8, 2), (16, 1)])
def test_prefill_head_folding_bf16(pkv, group, hkv):
    # G heads folded into the 128 tile rows (R = 128 / GP queries); G below GP leaves padding rows
    w = wl.sized_case(25, [777, 64, 300], [333, 17, 300], group * hkv, hkv, 128, "bf16")
    run_pair(pkv, w)


def test_many_prefill_chunks_heaviest_first(pkv):
    # 1200 chunks of 2..40 queries after 0..200 cached tokens, mixed with decodes: the
    # planner orders ~1200 query-tile pairs over more requests than its block holds
    # threads; every row matches the oracle whichever CTA ran its pair
    rng = np.random.default_rng(27)
    n = 1500
    q = np.where(np.arange(n) % 5 == 4, 1, rng.integers(2, 40, size=n, endpoint=True)).astype(np.int32)
    L = (q + rng.integers(0, 200, size=n, endpoint=True)).astype(np.int32)
    w = wl.sized_case(28, L, q, 8, 2, 128, "bf16")
    run_pair(pkv, w)


def test_decode_large_scale_bf16(pkv):
    w = wl.sized_case(26, [3000, 2049, 77], [1, 1, 1], 64, 8, 128, "bf16", scale=0.5)
    run_pair(pkv, w)


def test_request_without_query_tokens(pkv):
    # a request that contributes no tokens this step is skipped; its neighbours are not disturbed
    w = wl.sized_case(23, [50, 70, 90], [3, 0, 1], 8, 2, 128, "bf16")
    run_pair(pkv, w)


@pytest.mark.parametrize("group,hkv,n", [(4, 8, 3000), (8, 4, 3000), (16, 2, 3000), (4, 1, 2000)])
def test_many_short_decodes_with_invalid_items(pkv, group, hkv, n):
    """n decodes of 1..400 keys: every CTA takes many items, so the item ring wraps
    many times; every 97th request has seq_len 0 (an invalid item: flagged, its rows
    zeroed).  With one kv head, 2000 items are few enough per SM for the planner to hand
    them out largest first, over more requests than its block holds threads.  Valid
    rows match the oracle."""
    rng = np.random.default_rng(31)
    L = rng.integers(1, 400, size=n, endpoint=True).astype(np.int32)
    w = wl.sized_case(32, L, np.ones(n, np.int32), group * hkv, hkv, 128, "bf16")
    bad = np.arange(5, n, 97)
    L_run = L.copy()
    L_run[bad] = 0
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], dev(w.block_tables), dev(L_run),
                              dev(w.query_start_loc), w.scale, 1, int(L.max()))
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    good = np.setdiff1d(np.arange(n), bad)
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables, L,
                           w.query_start_loc, w.scale, rows=good)
    compare(out[torch.from_numpy(good).cuda()], ref, "bf16", "valid rows")
    zero = out[torch.from_numpy(bad).cuda()].float()
    assert torch.equal(zero, torch.zeros_like(zero))


def test_decode_workload_full(pkv):
    run_pair(pkv, wl.make("decode"))


def test_prefix_workload_full_with_cow(pkv):
    run_pair(pkv, wl.make("prefix"), cow=True)


def _sampled(pkv, name, seq_ids, row_pick=None):
    w = wl.make(name)
    t = w.make_tensors("cuda")
    w2, t_sub, rows = sub_batch(w, t, seq_ids)
    out, slots, st = gpu_step(pkv, w, t)
    assert st == 0, pkv.status_string(st)
    sub_rows = np.arange(len(rows)) if row_pick is None else row_pick(w2)
    ref, _, _, _ = oracle_step(w2, t_sub, rows=sub_rows)
    got = out[torch.from_numpy(rows[sub_rows]).cuda()]
    del t
    torch.cuda.empty_cache()
    return compare(got, ref, w.dtype, name)


def test_long_workload_sampled(pkv):
    _sampled(pkv, "long", [0, 13, 31])


def test_mixed_workload_sampled(pkv):
    rng = np.random.default_rng(3)
    decodes = 8 + rng.choice(4096, size=48, replace=False)
    seq_ids = np.concatenate([[0, 3, 7], decodes])

    def pick(w2):
        # every decode row, and the first, last and 30 random rows of each chunk
        qsl = w2.query_start_loc
        r = []
        for i in range(w2.num_seqs):
            n = qsl[i + 1] - qsl[i]
            if n == 1:
                r.append(qsl[i])
            else:
                sel = np.unique(np.concatenate([[0, n - 1], rng.choice(n, size=30, replace=False)]))
                r.extend(qsl[i] + sel)
        return np.asarray(r, np.int64)

    _sampled(pkv, "mixed", seq_ids, pick)


# --------------------------------------------------------------------------- bitwise invariances

def _attention_only(pkv, w, t, bt=None):
    m = to_gpu_meta(w, bt)
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"],
                              m["query_start_loc"], w.scale, w.max_query_len, w.max_seq_len)
    assert pkv.pkv_get_last_error() == 0
    return out


def test_permuted_block_ids_bitwise(pkv):
    w = wl.random_case(31, num_seqs=10, max_ctx=900, max_q=200, group=4, num_kv_heads=2, head_dim=128,
                       dtype="bf16")
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    a = _attention_only(pkv, w, t)
    perm = torch.from_numpy(np.random.default_rng(2).permutation(w.num_blocks)).cuda()
    k2, v2 = torch.empty_like(t["k_cache"]), torch.empty_like(t["v_cache"])
    k2[perm] = t["k_cache"]
    v2[perm] = t["v_cache"]
    permc = perm.cpu().numpy().astype(np.int32)
    bt2 = np.where(w.block_tables >= 0, permc[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    b = _attention_only(pkv, w, dict(t, k_cache=k2, v_cache=v2), bt=bt2)
    assert torch.equal(a, b)


def test_shared_prefix_vs_duplicated_bitwise(pkv):
    w = wl.make("prefix")
    t = w.make_tensors("cuda")
    shared = _attention_only(pkv, w, t, bt=w.block_tables_before_cow)
    # give every request private copies of the 64 prefix blocks
    n = w.num_seqs
    prefix = w.notes["shared_prefix_ids"]
    used = set(w.block_tables_before_cow[w.block_tables_before_cow >= 0].tolist())
    free = np.array(sorted(set(range(w.num_blocks)) - used - set(w.cow_dst.tolist())), np.int32)
    needed = n * len(prefix)
    extra = needed - len(free) + 8
    kc, vc = t["k_cache"], t["v_cache"]
    if extra > 0:
        kc = torch.cat([kc, torch.empty((extra,) + kc.shape[1:], dtype=kc.dtype, device="cuda")])
        vc = torch.cat([vc, torch.empty((extra,) + vc.shape[1:], dtype=vc.dtype, device="cuda")])
        free = np.concatenate([free, np.arange(w.num_blocks, w.num_blocks + extra, dtype=np.int32)])
    dup = w.block_tables_before_cow.copy()
    copies = free[:needed].reshape(n, len(prefix))
    dup[:, :len(prefix)] = copies
    src = torch.from_numpy(np.tile(prefix, n).astype(np.int32)).cuda()
    dst = torch.from_numpy(copies.reshape(-1).astype(np.int32)).cuda()
    pkv.pkv_copy_blocks(src, dst, kc, vc)
    w_dup = dataclasses.replace(w, num_blocks=kc.shape[0])
    duplicated = _attention_only(pkv, w_dup, dict(t, k_cache=kc, v_cache=vc), bt=dup)
    assert torch.equal(shared, duplicated)


def test_mixed_batch_equals_separate_calls_bitwise(pkv):
    w = wl.random_case(32, num_seqs=12, max_ctx=800, max_q=150, group=4, num_kv_heads=2, head_dim=128,
                       dtype="bf16")
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    whole = _attention_only(pkv, w, t)
    qsl = w.query_start_loc
    for i in range(w.num_seqs):
        wi = dataclasses.replace(w, seq_lens=w.seq_lens[i:i + 1].copy(),
                                 query_start_loc=np.array([0, qsl[i + 1] - qsl[i]], np.int32),
                                 block_tables=w.block_tables[i:i + 1].copy())
        ti = dict(t, q=t["q"][qsl[i]:qsl[i + 1]].contiguous())
        one = _attention_only(pkv, wi, ti)
        assert torch.equal(one, whole[qsl[i]:qsl[i + 1]]), i


def test_output_aligned_to_16_bytes_only(pkv):
    # The C ABI asks only 16-byte alignment of out; the prefill epilogue stores whole
    # 32-byte sectors when out allows it and 16-byte pieces otherwise.  An out that
    # starts 16 bytes past a 32-byte boundary takes the narrow stores; the values must
    # be the same bits as with an aligned out, and the bytes around out untouched.
    w = wl.random_case(41, num_seqs=8, max_ctx=900, max_q=300, group=4, num_kv_heads=2, head_dim=128,
                       dtype="bf16", decode_frac=0.3)
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    m = to_gpu_meta(w)
    args = (t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"], m["query_start_loc"], w.scale,
            w.max_query_len, w.max_seq_len)
    aligned = pkv.paged_attention(*args)
    assert pkv.pkv_get_last_error() == 0
    n = t["q"].numel()
    flat = torch.full((n + 32,), 7.0, dtype=torch.bfloat16, device="cuda")
    assert flat.data_ptr() % 32 == 0
    shifted = flat[8:8 + n].view(t["q"].shape)  # 8 bf16 = 16 bytes past the boundary
    assert shifted.data_ptr() % 32 == 16
    pkv.paged_attention(*args, out=shifted)
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(shifted, aligned)
    assert torch.all(flat[:8] == 7.0) and torch.all(flat[8 + n:] == 7.0)
    # attention alone read the pool as drawn (no new tokens were written)
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    compare(shifted, ref, "bf16", w.name)


@pytest.mark.parametrize("seed,group,hkv", [(13, 1, 4), (14, 2, 2), (16, 4, 8), (17, 8, 2)])
def test_repeated_calls_match_oracle_and_each_other(pkv, seed, group, hkv):
    # Which CTA runs which item, and when, changes from call to call; the results must
    # not.  Repetition also exposes ordering races inside a CTA's pipeline.
    w = wl.random_case(seed, num_seqs=10, max_ctx=1500, max_q=300, group=group, num_kv_heads=hkv,
                       head_dim=128, dtype="bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    _, slots, st = gpu_step(pkv, w, t)
    assert st == 0
    ref, _, kc, vc = oracle_step(w, t_cpu)
    outs = [_attention_only(pkv, w, t) for _ in range(6)]
    for o in outs:
        compare(o, ref, "bf16", w.name)
        assert torch.equal(o, outs[0])


def test_split_decodes_repeat_bitwise(pkv):
    # Requests of 2 to 9 key splits next to unsplit ones: which split finishes last
    # changes from call to call; the merge runs in split order all the same, so the
    # rows must be identical.
    lens = [2049, 3000, 4096, 5121, 9000, 300, 2048, 7777, 18000]
    w = wl.sized_case(43, lens, [1] * len(lens), 16, 4, 128, "bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    outs = [_attention_only(pkv, w, t) for _ in range(6)]
    assert pkv.pkv_get_last_error() == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale)
    for o in outs:
        compare(o, ref, "bf16", w.name)
        assert torch.equal(o, outs[0])


def test_bad_block_in_one_split_zeroes_the_merged_row(pkv):
    # a bad block id in the second split of a 5121-key request: that request's merged
    # rows are zero, every other request is unaffected
    w = wl.sized_case(44, [5121, 3000, 600], [1, 1, 1], 8, 2, 128, "bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    bt = w.block_tables.copy()
    bt[0, 2100 // 16] = w.num_blocks + 3
    m = to_gpu_meta(w, bt)
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"],
                              m["query_start_loc"], w.scale, w.max_query_len, w.max_seq_len)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    assert torch.count_nonzero(out[0]) == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale, rows=np.array([1, 2], np.int64))
    compare(out[1:3], ref, "bf16")


# --------------------------------------------------------------------------- device errors

def test_bad_block_id_zeroes_only_that_request(pkv):
    w = wl.sized_case(41, [300, 200, 150], [1, 40, 1], 8, 2, 128, "bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    bt = w.block_tables.copy()
    bt[1, 3] = w.num_blocks + 5              # request 1 (a 40-token chunk) points past the pool
    m = to_gpu_meta(w, bt)
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"],
                              m["query_start_loc"], w.scale, w.max_query_len, w.max_seq_len)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    qsl = w.query_start_loc
    # rows of request 1 that would read logical block 3 (positions >= 48) are zero
    pos = w.seq_lens[1] - 40 + np.arange(40)
    bad_rows = qsl[1] + np.nonzero(pos >= 48)[0]
    assert torch.count_nonzero(out[torch.from_numpy(bad_rows).cuda()]) == 0
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                           w.seq_lens, w.query_start_loc, w.scale, rows=np.array([0, qsl[2]], np.int64))
    compare(out[torch.tensor([0, int(qsl[2])], device="cuda")], ref, "bf16")


def test_seq_len_shorter_than_query_is_flagged(pkv):
    w = wl.sized_case(42, [64, 64], [1, 1], 8, 2, 128, "bf16")
    t = {k: v.cuda() for k, v in w.make_tensors("cpu").items()}
    m = to_gpu_meta(w)
    m["query_start_loc"] = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    m["seq_lens"] = torch.tensor([64, 0], dtype=torch.int32, device="cuda")
    out = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["block_tables"], m["seq_lens"],
                              m["query_start_loc"], w.scale, 1, 64)
    assert pkv.pkv_get_last_error() == pkv.PKV_ERR_INDEX
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[0]) > 0


def test_both_merge_launches_give_the_same_bits(pkv):
    # Requests of 3 to 8 key splits are merged by one thread per column when no request
    # of the batch folds more partials than that, and by four 128-thread runs otherwise;
    # both fold in the same order.  The same requests in a batch with a 9-split request
    # (the general merge) and without it (the per-thread merge) give identical rows,
    # and both match the oracle.
    lens = [2049, 3000, 4096, 5121, 8000, 300]
    w_small = wl.sized_case(45, lens, [1] * len(lens), 32, 8, 128, "bf16")
    w_big = wl.sized_case(45, lens + [9000], [1] * (len(lens) + 1), 32, 8, 128, "bf16")
    t_cpu = w_big.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    # the small batch's tables are the big batch's first rows, so both read the same keys
    w_small = dataclasses.replace(w_small, num_blocks=w_big.num_blocks,
                                  block_tables=w_big.block_tables[:len(lens), :w_big.block_tables.shape[1]].copy())
    t_small = dict(t, q=t["q"][:len(lens)].contiguous())
    small = _attention_only(pkv, w_small, t_small)
    big = _attention_only(pkv, w_big, t)
    assert torch.equal(small, big[:len(lens)])
    ref = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w_big.block_tables,
                           w_big.seq_lens, w_big.query_start_loc, w_big.scale)
    compare(big, ref, "bf16", w_big.name)


def test_zero_scale_averages_the_visible_values(pkv):
    # scale 0: every visible key weighs the same, so each row is the mean of its
    # visible V rows (the oracle computes that exactly); masked keys of diagonal and
    # partial tiles must weigh nothing rather than turn into NaN
    w = dataclasses.replace(wl.random_case(46, num_seqs=10, max_ctx=900, max_q=300, group=4, num_kv_heads=2,
                                           head_dim=128, dtype="bf16"), scale=0.0)
    run_pair(pkv, w)
