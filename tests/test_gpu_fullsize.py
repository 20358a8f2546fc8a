"""Every output row of every named workload, at full size, against the fp64 oracle,
through the very calls the benchmark times.

``bench.Step`` runs one step as ``bench.py`` does: the copy-on-write copies where
the workload has them, then ``paged_attention_step`` (slot mapping, K/V scatter
and attention in one call), with the shared prefix handed over as a group hint
where the workload has one.  The oracle starts from a device copy of the pool
taken before the step, performs the copy-on-write, the slot mapping and the
scatter itself, and attends every query row ("vLLM's PagedAttention" teardown,
sections "PagedAttention: the KV cache is paged, like virtual memory" and
"Continuous batching: rebuild the batch every step"; the copy-on-write step
follows the OS-trick article, Technical Details).

Large pools go to the host a group of requests at a time: only the blocks a
group references, renumbered (the oracle's result does not depend on physical
ids).  Every group's written blocks are compared bit for bit with the oracle's
scatter and copies; every output row within bf16 max-abs 2e-2 and mean-abs 2e-3
(fp32: 1e-4).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from bench import Step
from helpers import compare, host_requests, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def _groups_of(w, kv_bytes_per_group=3 << 30):
    """Request groups whose referenced blocks take about ``kv_bytes_per_group`` on the host."""
    blk_bytes = 2 * w.num_kv_heads * 16 * w.head_dim * w.elem_bytes
    nblk = (w.seq_lens.astype(np.int64) + 15) // 16
    groups, cur, acc = [], [], 0
    for i in range(w.num_seqs):
        cur.append(i)
        acc += int(nblk[i]) * blk_bytes
        if acc >= kv_bytes_per_group:
            groups.append(cur)
            cur, acc = [], 0
    if cur:
        groups.append(cur)
    return groups


def _every_row(pkv, name, cascade=True):
    w = wl.make(name)
    step = Step(pkv, w, torch.device("cuda"), cascade=cascade, fused=True)
    t = step.t
    k0, v0 = t["k_cache"].clone(), t["v_cache"].clone()   # the pool as drawn: the oracle's input
    step.run()
    assert pkv.pkv_get_last_error() == 0
    torch.cuda.synchronize()
    n_rows, worst_max, sum_err = 0, 0.0, 0.0
    for seq_ids in _groups_of(w):
        w2, t_sub, rows, used = host_requests(w, k0, v0, t, seq_ids)
        ref, _, kc_ref, vc_ref = oracle_step(w2, t_sub, cow=w2.cow_src is not None)
        got = step.out.index_select(0, torch.from_numpy(rows).cuda())
        mx, mean = compare(got, ref, w.dtype, f"{name} requests {seq_ids[0]}..{seq_ids[-1]}")
        worst_max = max(worst_max, mx)
        sum_err += mean * ref.size
        n_rows += len(rows)
        # the written pool, bit for bit, on every block these requests reference
        idx = torch.from_numpy(used).cuda()
        for pool, ref_pool in ((t["k_cache"], kc_ref), (t["v_cache"], vc_ref)):
            g = pool.index_select(0, idx)
            g = g.view(torch.int16) if g.dtype == torch.bfloat16 else g
            assert torch.equal(g.cpu(), torch.from_numpy(ref_pool)), f"{name}: written pool differs"
    assert n_rows == w.num_tokens
    del step, t, k0, v0
    torch.cuda.empty_cache()
    return worst_max, sum_err


@pytest.mark.parametrize("name", ["tiny", "decode", "prefix", "prefill", "long", "mixed"])
def test_every_row_of_the_benchmarked_step(pkv, name):
    _every_row(pkv, name)


def test_every_row_of_the_prefix_step_without_the_group_hint(pkv):
    # bench.py --no-cascade: each member attends its shared prefix itself
    _every_row(pkv, "prefix", cascade=False)
