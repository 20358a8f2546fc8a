"""PagedAttention hot path for GB300 (sm_103a): thin Python binding over libpkv.

The library (``libpkv.so``, built in-tree from ``csrc/`` by ``_build.py``) exports
a C ABI declared in ``include/pkv.h``.  This module only marshals arguments:
it checks tensor placement, dtype and contiguity, passes raw device pointers and
the current CUDA stream, and turns a non-zero status into :class:`PkvError`.
Every computation runs in the library's CUDA kernels; there is no CPU path.
If the library has not been built, importing a function raises immediately.

Functions carry the C names:
  pkv_slot_mapping, pkv_write, pkv_copy_blocks, paged_attention,
  pkv_get_last_error, pkv_peek_error_bits, pkv_trace_enable, pkv_trace_read,
  pkv_num_workers, pkv_shutdown, pkv_umma_selftest, pkv_tma_selftest.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_INDEX = 0, 1, 2, 3
PKV_ERR_CUDA, PKV_ERR_NO_MEMORY, PKV_ERR_TIMEOUT = 4, 5, 6
PKV_F32, PKV_BF16 = 0, 1
BLOCK_SIZE = 16
TRACE_KINDS = 8

_lib = None
_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def lib():
    """The loaded libpkv (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libpkv.so not built at {LIB_PATH}; run "
                                  "`python -m paged_kv_cache_248_gb300._build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            D = ctypes.POINTER(_CacheDesc)
            sig = {
                "pkv_slot_mapping": [P, i32, P, P, i32, i64, P, P],
                "pkv_write": [P, P, P, i64, P, P, D, P],
                "pkv_copy_blocks": [P, P, i64, P, P, D, P],
                "paged_attention": [P, P, P, D, P, i32, P, P, i32, i32, i64, i32, i32, f32, P, P],
                "pkv_get_last_error": [P],
                "pkv_peek_error_bits": [P, ctypes.POINTER(ctypes.c_uint32)],
                "pkv_num_workers": [ctypes.POINTER(ctypes.c_int32)],
                "pkv_trace_enable": [ctypes.c_int],
                "pkv_trace_read": [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)],
                "pkv_umma_selftest": [P, P, P, P, P],
                "pkv_tma_selftest": [P, i64, i32, P, P],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.pkv_status_string.argtypes = [ctypes.c_int]
            L.pkv_status_string.restype = ctypes.c_char_p
            L.pkv_trace_kind_name.argtypes = [ctypes.c_int]
            L.pkv_trace_kind_name.restype = ctypes.c_char_p
            L.pkv_shutdown.argtypes = []
            L.pkv_shutdown.restype = None
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pkv_status_string(int(status)).decode()
    except ImportError:
        return str(status)


def _check(status: int, what: str):
    if status != PKV_OK:
        raise PkvError(status, what)


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _cache_desc(k_cache: torch.Tensor, v_cache: torch.Tensor) -> _CacheDesc:
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must both be [num_blocks, num_kv_heads, 16, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    if k_cache.dtype == torch.float32:
        dt = PKV_F32
    elif k_cache.dtype == torch.bfloat16:
        dt = PKV_BF16
    else:
        raise ValueError(f"unsupported cache dtype {k_cache.dtype}")
    return _CacheDesc(nb, bs, hkv, d, dt)


def pkv_slot_mapping(block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                     num_tokens: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int64 physical slot of every new token (block_tables[i][p // 16] * 16 + p % 16)."""
    if out is None:
        out = torch.empty(num_tokens, dtype=torch.int64, device=block_tables.device)
    num_seqs = seq_lens.shape[0]
    _check(lib().pkv_slot_mapping(_dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                                  _dev(seq_lens, "seq_lens", torch.int32),
                                  _dev(query_start_loc, "query_start_loc", torch.int32), num_seqs, num_tokens,
                                  _dev(out, "out", torch.int64), _stream(stream)), "pkv_slot_mapping")
    return out


def pkv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
              v_cache: torch.Tensor, stream=None) -> None:
    """Scatter new tokens' K/V rows [T, Hkv, d] into their cache slots (in place)."""
    desc = _cache_desc(k_cache, v_cache)
    _check(lib().pkv_write(_dev(k, "k", k_cache.dtype), _dev(v, "v", k_cache.dtype),
                           _dev(slot_mapping, "slot_mapping", torch.int64), k.shape[0],
                           _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                           _stream(stream)), "pkv_write")


def pkv_copy_blocks(src: torch.Tensor, dst: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    stream=None) -> None:
    """Copy-on-write: cache[dst[i]] = cache[src[i]] for K and V (in place)."""
    desc = _cache_desc(k_cache, v_cache)
    _check(lib().pkv_copy_blocks(_dev(src, "src", torch.int32), _dev(dst, "dst", torch.int32), src.shape[0],
                                 _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                 _stream(stream)), "pkv_copy_blocks")


def paged_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, query_start_loc: torch.Tensor, scale: float, max_query_len: int,
                    max_seq_len: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention of one mixed batch of chunked prefills and decodes over the paged cache."""
    desc = _cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    T, hq, d = q.shape
    _check(lib().paged_attention(_dev(q, "q", k_cache.dtype), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                 ctypes.byref(desc), _dev(block_tables, "block_tables", torch.int32),
                                 block_tables.shape[1], _dev(seq_lens, "seq_lens", torch.int32),
                                 _dev(query_start_loc, "query_start_loc", torch.int32), seq_lens.shape[0], hq, T,
                                 int(max_query_len), int(max_seq_len), float(scale),
                                 _dev(out, "out", k_cache.dtype), _stream(stream)), "paged_attention")
    return out


def pkv_get_last_error(stream=None) -> int:
    """Sync the stream; return (and clear) the device error status."""
    return int(lib().pkv_get_last_error(_stream(stream)))


def pkv_peek_error_bits(stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().pkv_peek_error_bits(_stream(stream), ctypes.byref(bits)), "pkv_peek_error_bits")
    return int(bits.value)


def pkv_num_workers() -> int:
    w = ctypes.c_int32(0)
    _check(lib().pkv_num_workers(ctypes.byref(w)), "pkv_num_workers")
    return int(w.value)


def pkv_trace_enable(on: bool = True) -> None:
    _check(lib().pkv_trace_enable(1 if on else 0), "pkv_trace_enable")


def pkv_trace_read() -> dict:
    """{kind: (launches, total_ms)} since the last read; synchronises the device."""
    n = (ctypes.c_int64 * TRACE_KINDS)()
    ms = (ctypes.c_double * TRACE_KINDS)()
    _check(lib().pkv_trace_read(n, ms), "pkv_trace_read")
    return {lib().pkv_trace_kind_name(k).decode(): (int(n[k]), float(ms[k])) for k in range(TRACE_KINDS)}


def pkv_shutdown() -> None:
    lib().pkv_shutdown()


def pkv_umma_selftest(params, a_img: torch.Tensor, b_img: torch.Tensor, d_out: torch.Tensor, stream=None) -> None:
    arr = (ctypes.c_int32 * 29)(*[int(x) for x in params])
    _check(lib().pkv_umma_selftest(arr, _dev(a_img, "a_img"), _dev(b_img, "b_img"),
                                   _dev(d_out, "d_out", torch.float32), _stream(stream)), "pkv_umma_selftest")


def pkv_tma_selftest(src: torch.Tensor, row0: int, dump: torch.Tensor, stream=None) -> None:
    _check(lib().pkv_tma_selftest(_dev(src, "src", torch.bfloat16), src.shape[0], int(row0), _dev(dump, "dump"),
                                  _stream(stream)), "pkv_tma_selftest")
