"""fp64 CPU oracle for the PagedAttention hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never does: it shares no code with
the oracle, and the product fails loudly when its CUDA extension is missing
instead of falling back here.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64).  This module compiles
it with gcc on first use and marshals numpy arrays / CPU torch tensors into it.
What each function computes, and which passage of the pages it follows, is
written in the C file's comments:

* ``slot_mapping``  -- logical position -> physical slot through the block table
  ("vLLM's PagedAttention" teardown, section "PagedAttention: the KV cache is
  paged, like virtual memory").
* ``write``         -- scatter of new tokens' K/V rows into their slots (same
  section).
* ``copy_blocks``   -- copy-on-write of whole blocks ("The 1960s Operating System
  Trick ...", Technical Details, Copy-on-Write).
* ``attention``     -- softmax(scale * q k^T) v over each request's logical
  context gathered through its block table, bottom-right causal inside prefill
  chunks ("vLLM's PagedAttention" teardown, sections "PagedAttention" and
  "Continuous batching").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
BLOCK = 16


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libpkv_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            lib.orc_slot_mapping.argtypes = [P, i32, P, P, i32, P]
            lib.orc_write.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P]
            lib.orc_copy_blocks.argtypes = [P, P, i64, i64, i64, P, P]
            lib.orc_attention.argtypes = [P, i32, P, P, i64, i32, i32, P, i32, P, P, i32,
                                          i32, f32, P, i64, P, i32]
            for f in (lib.orc_slot_mapping, lib.orc_write, lib.orc_copy_blocks, lib.orc_attention):
                f.restype = ctypes.c_int
            lib.orc_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _np(x, dtype=None):
    """CPU torch tensor or array -> C-contiguous numpy array (no copy when possible)."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach()
        if x.dtype == torch.bfloat16:
            x = x.contiguous().view(torch.int16)
        x = x.cpu().contiguous().numpy()
    a = np.ascontiguousarray(x)
    if dtype is not None and a.dtype != dtype:
        a = a.astype(dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype in (np.int16, np.uint16):  # bf16 bit patterns
        return BF16
    raise TypeError(f"oracle reads fp32 or bf16 bit patterns (int16/uint16), got {a.dtype}")


def max_threads() -> int:
    return int(_load().orc_max_threads())


def slot_mapping(block_tables, seq_lens, query_start_loc) -> np.ndarray:
    """int64 slot per query token: block_tables[i][p // 16] * 16 + p % 16."""
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    out = np.empty(int(qsl[-1]), dtype=np.int64)
    rc = _load().orc_slot_mapping(_ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl), sl.shape[0], _ptr(out))
    if rc:
        raise OracleError(f"orc_slot_mapping status {rc}")
    return out


def write(k, v, slots, k_cache: np.ndarray, v_cache: np.ndarray) -> None:
    """In place: cache[slot // 16][h][slot % 16][:] = k[t][h][:] (and v).  Negative slots skip."""
    k, v = _np(k), _np(v)
    s = _np(slots, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, hkv, d = k.shape
    rc = _load().orc_write(_ptr(k), _ptr(v), _ptr(s), T, hkv, d, k.itemsize,
                           k_cache.shape[0], _ptr(k_cache), _ptr(v_cache))
    if rc:
        raise OracleError(f"orc_write status {rc}")


def copy_blocks(src, dst, k_cache: np.ndarray, v_cache: np.ndarray) -> None:
    """In place: cache[dst[i]] = snapshot(cache)[src[i]] for K and V."""
    s, d = _np(src, np.int32), _np(dst, np.int32)
    block_bytes = k_cache[0].nbytes
    rc = _load().orc_copy_blocks(_ptr(s), _ptr(d), s.shape[0], block_bytes, k_cache.shape[0],
                                 _ptr(k_cache), _ptr(v_cache))
    if rc:
        raise OracleError(f"orc_copy_blocks status {rc}")


def attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale: float,
              rows=None, n_threads: int = 0) -> np.ndarray:
    """fp64 [n_rows, Hq, d] attention by definition (see pkv_oracle.c).

    ``q`` is [T_q, Hq, d]; caches are [num_blocks, Hkv, 16, d]; all in fp32 or as
    bf16 bit patterns.  ``rows`` selects query tokens (default: all of them).
    """
    qa, kc, vc = _np(q), _np(k_cache), _np(v_cache)
    dt = _dtype_code(qa)
    assert _dtype_code(kc) == dt and _dtype_code(vc) == dt
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    T_q, hq, d = qa.shape
    nb, hkv, bs, d2 = kc.shape
    assert bs == BLOCK and d2 == d and int(qsl[-1]) == T_q
    if rows is None:
        rows_a, n_rows, rp = None, T_q, None
    else:
        rows_a = _np(rows, np.int64)
        n_rows, rp = rows_a.shape[0], _ptr(rows_a)
    out = np.empty((n_rows, hq, d), dtype=np.float64)
    rc = _load().orc_attention(_ptr(qa), dt, _ptr(kc), _ptr(vc), nb, hkv, d, _ptr(bt), bt.shape[1],
                               _ptr(sl), _ptr(qsl), sl.shape[0], hq, ctypes.c_float(scale), rp,
                               n_rows, _ptr(out), n_threads)
    if rc:
        raise OracleError(f"orc_attention status {rc}")
    return out
