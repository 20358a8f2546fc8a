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


def test_fp32_one_token_step_replays_from_a_cuda_graph(pkv):
    """The tiny fp32 workload's step (every request one token: the new rows are stored by
    the attention launch itself) captured and replayed: the same bits as the eager call,
    and the oracle's outputs.  The step rewrites the same rows on every replay."""
    w = wl.make("tiny")
    assert w.max_query_len == 1 and w.dtype == "f32"
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    bt, sl, qsl = dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)
    slots = torch.empty(w.num_tokens, dtype=torch.int64, device="cuda")
    out_eager = torch.empty_like(t["q"])
    out_graph = torch.full_like(t["q"], float("nan"))

    def step(out):
        pkv.paged_attention_step(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale,
                                 w.max_query_len, w.max_seq_len, slot_mapping=slots, out=out)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(out_eager)
    s.synchronize()
    assert pkv.pkv_get_last_error(s) == 0
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(out_graph)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_get_last_error() == 0
    assert torch.equal(out_graph, out_eager)
    ref, ref_slots, ref_k, ref_v = oracle_step(w, t_cpu)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    compare(out_graph, ref, "f32", w.name)
    for got, want, name in ((t["k_cache"], ref_k, "k_cache"), (t["v_cache"], ref_v, "v_cache")):
        assert np.array_equal(bits(got), want), name
