"""paged_attention_noalloc: the attention entry point for callers that cannot let a
library allocate device memory (their allocator must account for every byte, or
their service forbids allocation after start-up).  It keeps its split-KV scratch
in a fixed static device array.

Checked through the C ABI, for two calls in a row (the array keeps the previous
call's contents), against the fp64 oracle and against paged_attention on the same
inputs, within the bf16 tolerance the other parity tests use.  This file is collected last so that a
failure here cannot hide the result of any other test; it also passes when run
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import TOL, bits, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import paged_kv_cache_248_gb300 as pkv
    lib = pkv.lib()
    fn = lib.paged_attention_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, P, P, ctypes.POINTER(pkv._CacheDesc), P, i32, P, P, i32, i32, i64, i32, i32,
                   ctypes.c_float, P, P, P]
    fn.restype = ctypes.c_int
    assert pkv.pkv_get_last_error() == 0
    return pkv, fn


def _inputs(w):
    t_cpu = w.make_tensors("cpu")
    t = {k: v.cuda() for k, v in t_cpu.items()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return t_cpu, t, dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc)


def _call_noalloc(pkv, fn, w, t, bt, sl, qsl, out, err_word):
    desc = pkv._cache_desc(t["k_cache"], t["v_cache"])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = ctypes.c_void_p
    return fn(P(t["q"].data_ptr()), P(t["k_cache"].data_ptr()), P(t["v_cache"].data_ptr()), ctypes.byref(desc),
              P(bt.data_ptr()), bt.shape[1], P(sl.data_ptr()), P(qsl.data_ptr()), w.num_seqs, w.num_q_heads,
              w.num_tokens, w.max_query_len, w.max_seq_len, ctypes.c_float(w.scale), P(out.data_ptr()),
              P(err_word.data_ptr()) if err_word is not None else None, stream)


def _close(a: torch.Tensor, b: torch.Tensor):
    d = (a.double() - b.double()).abs()
    max_tol, mean_tol = TOL["bf16"]
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= max_tol and d.mean().item() <= mean_tol


@pytest.mark.parametrize("case", ["decode", "mixed_small"])
def test_noalloc_matches_the_oracle_and_paged_attention_twice(api, case):
    pkv, fn = api
    if case == "decode":
        w = wl.make("decode")                 # 64 requests up to 4096 tokens: multi-split decode
    else:
        w = wl.random_case(5, num_seqs=10, max_ctx=2500, max_q=300, group=4, num_kv_heads=8, head_dim=128,
                           dtype="bf16")       # chunked prefills and decodes in one batch
    t_cpu, t, bt, sl, qsl = _inputs(w)
    exact = oracle.attention(bits(t_cpu["q"]), bits(t_cpu["k_cache"]), bits(t_cpu["v_cache"]), w.block_tables,
                             w.seq_lens, w.query_start_loc, w.scale)
    ref = pkv.paged_attention(t["q"], t["k_cache"], t["v_cache"], bt, sl, qsl, w.scale, w.max_query_len,
                              w.max_seq_len)
    assert pkv.pkv_get_last_error() == 0
    err_word = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(t["q"], float("nan"))
        st = _call_noalloc(pkv, fn, w, t, bt, sl, qsl, out, err_word if call == 0 else None)
        assert st == 0, pkv.status_string(st)
        torch.cuda.synchronize()
        compare(out, exact, "bf16", f"{case}, call {call}")
        _close(out, ref)
    assert int(err_word.item()) == 0


def test_noalloc_rejects_batches_beyond_its_scratch(api):
    pkv, fn = api
    w = wl.make("long")                        # 32 x 32768 tokens, 64/8 heads: ~34 MB of partials
    k = torch.empty((16, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((w.num_tokens, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    t = {"q": q, "k_cache": k, "v_cache": k.clone()}
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    out = torch.empty_like(q)
    st = _call_noalloc(pkv, fn, w, t, dev(w.block_tables), dev(w.seq_lens), dev(w.query_start_loc), out, None)
    assert st == pkv.PKV_ERR_NO_MEMORY
