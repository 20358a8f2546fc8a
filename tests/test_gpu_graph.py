"""The whole step -- slot mapping, KV scatter, attention -- captured into a CUDA graph
and replayed.  The library does no allocation inside a capture (its workspace is
sized by an eager call first), so the step is one graph launch per iteration, as a
serving loop would run it."""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import bits, compare, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_248_gb300 as m
    m.lib()
    assert m.pkv_get_last_error() == 0
    return m


def _step_fn(pkv, w, t, m, slots, out):
    def run():
        pkv.pkv_slot_mapping(m["bt"], m["sl"], m["qsl"], w.num_tokens, out=slots)
        pkv.pkv_write(t["k_new"], t["v_new"], slots, t["k_cache"], t["v_cache"])
        pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], m["bt"], m["sl"], m["qsl"], w.scale,
                            w.max_query_len, w.max_seq_len, out=out)
    return run


@pytest.mark.parametrize("case", ["mixed_small", "decode"])
def test_step_replays_from_a_cuda_graph(pkv, case):
    if case == "decode":
        w = wl.make("decode")
    else:
        w = wl.random_case(3, num_seqs=12, max_ctx=1800, max_q=300, group=4, num_kv_heads=8, head_dim=128,
                           dtype="bf16")
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    m = {"bt": dev(w.block_tables), "sl": dev(w.seq_lens), "qsl": dev(w.query_start_loc)}
    slots = torch.empty(w.num_tokens, dtype=torch.int64, device="cuda")
    out_eager = torch.empty_like(t["q"])
    out_graph = torch.full_like(t["q"], float("nan"))
    step = _step_fn(pkv, w, t, m, slots, out_eager)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()                                   # eager: sizes the workspace
    s.synchronize()
    assert pkv.pkv_get_last_error(s) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step_fn(pkv, w, t, m, slots, out_graph)()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(out_graph, out_eager)     # same kernels, same inputs: bitwise
    ref, _, _, _ = oracle_step(w, t_cpu)
    compare(out_graph, ref, "bf16", w.name)
