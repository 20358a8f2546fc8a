"""PagedAttention hot path for GB300 (sm_103a): thin Python binding over libpkv.

The library (``libpkv.so``, built in-tree from ``csrc/`` by ``_build.py``) exports
a C ABI declared in ``include/pkv.h``.  This module only marshals arguments:
it checks tensor placement, dtype and contiguity, passes raw device pointers and
the current CUDA stream, and turns a non-zero status into :class:`PkvError`.
Every computation runs in the library's CUDA kernels; there is no CPU path.
If the library has not been built, importing a function raises immediately.

Functions carry the C names:
  pkv_slot_mapping, pkv_write, pkv_copy_blocks, paged_attention, paged_attention_cascade,
  paged_attention_step,
  pkv_get_last_error, pkv_peek_error_bits, pkv_trace_enable, pkv_trace_read,
  pkv_num_workers, pkv_shutdown, pkv_umma_selftest, pkv_tma_selftest, pkv_wait_selftest.
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
TRACE_KINDS = 9

_lib = None
_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class _PrefixGroups(ctypes.Structure):
    _fields_ = [("prefix_block_tables", ctypes.c_void_p), ("max_prefix_blocks", ctypes.c_int32),
                ("prefix_num_blocks", ctypes.c_void_p), ("member_start", ctypes.c_void_p),
                ("member_seqs", ctypes.c_void_p), ("num_groups", ctypes.c_int32), ("num_members", ctypes.c_int32)]


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
                "paged_attention_cascade": [P, P, P, D, P, i32, P, P, i32, i32, i64, i32, i32, f32,
                                            ctypes.POINTER(_PrefixGroups), P, P],
                "paged_attention_step": [P, P, P, P, P, D, P, i32, P, P, i32, i32, i64, i32, i32, f32,
                                         ctypes.POINTER(_PrefixGroups), P, P, P],
                "paged_attention_step_cow": [P, P, P, P, P, D, P, i32, P, P, i32, i32, i64, i32, i32, f32,
                                             ctypes.POINTER(_PrefixGroups), P, P, i64, P, P, P],
                "pkv_get_last_error": [P],
                "pkv_peek_error_bits": [P, ctypes.POINTER(ctypes.c_uint32)],
                "pkv_num_workers": [ctypes.POINTER(ctypes.c_int32)],
                "pkv_trace_enable": [ctypes.c_int],
                "pkv_trace_read": [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)],
                "pkv_umma_selftest": [P, P, P, P, P],
                "pkv_tma_selftest": [P, i64, i32, P, P],
                "pkv_wait_selftest": [P],
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


def paged_attention_cascade(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                            scale: float, max_query_len: int, max_seq_len: int, prefix_block_tables: torch.Tensor,
                            prefix_num_blocks: torch.Tensor, member_start: torch.Tensor, member_seqs: torch.Tensor,
                            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """paged_attention with shared-prefix groups as a hint: group g's prefix is the
    first prefix_num_blocks[g] blocks of row g of prefix_block_tables, shared by the
    requests member_seqs[member_start[g]:member_start[g + 1]].  Same result."""
    desc = _cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    T, hq, d = q.shape
    groups = _groups((prefix_block_tables, prefix_num_blocks, member_start, member_seqs))
    _check(lib().paged_attention_cascade(_dev(q, "q", k_cache.dtype), _dev(k_cache, "k_cache"),
                                         _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                         _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                                         _dev(seq_lens, "seq_lens", torch.int32),
                                         _dev(query_start_loc, "query_start_loc", torch.int32), seq_lens.shape[0],
                                         hq, T, int(max_query_len), int(max_seq_len), float(scale),
                                         ctypes.byref(groups), _dev(out, "out", k_cache.dtype), _stream(stream)),
           "paged_attention_cascade")
    return out


def _groups(prefix_groups):
    """(prefix_block_tables, prefix_num_blocks, member_start, member_seqs) -> struct, or None."""
    if prefix_groups is None:
        return None
    tables, nblocks, start, members = prefix_groups
    if tables.dim() != 2:
        raise ValueError("prefix_block_tables must be [num_groups, max_prefix_blocks]")
    G, M = nblocks.shape[0], members.shape[0]
    if tables.shape[0] != G or start.shape[0] != G + 1:
        raise ValueError("prefix group arrays disagree on the number of groups")
    return _PrefixGroups(_dev(tables, "prefix_block_tables", torch.int32), tables.shape[1],
                         _dev(nblocks, "prefix_num_blocks", torch.int32), _dev(start, "member_start", torch.int32),
                         _dev(members, "member_seqs", torch.int32) if M else None, G, M)


def paged_attention_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                         v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor,
                         query_start_loc: torch.Tensor, scale: float, max_query_len: int, max_seq_len: int,
                         prefix_groups=None, slot_mapping: torch.Tensor | None = None,
                         out: torch.Tensor | None = None, stream=None, cow=None) -> torch.Tensor:
    """Slot mapping, K/V scatter and attention of one step in one call (same results as
    pkv_slot_mapping + pkv_write + paged_attention[_cascade]).  ``prefix_groups`` is
    None or (prefix_block_tables, prefix_num_blocks, member_start, member_seqs);
    ``slot_mapping``, if given, receives the int64 slots.  ``cow`` is None or
    (src, dst) int32 block ids: copied first, as pkv_copy_blocks (C call
    paged_attention_step_cow)."""
    desc = _cache_desc(k_cache, v_cache)
    if out is None:
        out = torch.empty_like(q)
    T, hq, d = q.shape
    if k_new.shape != (T, k_cache.shape[1], d) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [num_tokens, num_kv_heads, head_dim]")
    g = _groups(prefix_groups)
    head = (_dev(q, "q", k_cache.dtype), _dev(k_new, "k_new", k_cache.dtype), _dev(v_new, "v_new", k_cache.dtype),
            _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(seq_lens, "seq_lens", torch.int32), _dev(query_start_loc, "query_start_loc", torch.int32),
            seq_lens.shape[0], hq, T, int(max_query_len), int(max_seq_len), float(scale),
            ctypes.byref(g) if g is not None else None)
    tail = (_dev(slot_mapping, "slot_mapping", torch.int64) if slot_mapping is not None else None,
            _dev(out, "out", k_cache.dtype), _stream(stream))
    if cow is None:
        _check(lib().paged_attention_step(*head, *tail), "paged_attention_step")
    else:
        src, dst = cow
        if src.shape != dst.shape or src.dim() != 1:
            raise ValueError("cow src and dst must be int32 vectors of one length")
        _check(lib().paged_attention_step_cow(*head, _dev(src, "cow src", torch.int32),
                                              _dev(dst, "cow dst", torch.int32), src.shape[0], *tail),
               "paged_attention_step_cow")
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


def pkv_wait_selftest(stream=None) -> None:
    _check(lib().pkv_wait_selftest(_stream(stream)), "pkv_wait_selftest")


def pkv_tma_selftest(src: torch.Tensor, row0: int, dump: torch.Tensor, stream=None) -> None:
    _check(lib().pkv_tma_selftest(_dev(src, "src", torch.bfloat16), src.shape[0], int(row0), _dev(dump, "dump"),
                                  _stream(stream)), "pkv_tma_selftest")


# ----------------------------------------------------------------------------- block manager
class BlockManager:
    """Host-side KV block manager in libpkv (C ABI in include/pkv_blocks.h): a pool of
    16-token blocks with a free queue, reference counts, chained hashing of full blocks
    for prefix reuse, fork and copy-on-write.  Argument marshalling only."""

    def __init__(self, num_blocks: int, enable_prefix_cache: bool = True):
        L = lib()
        if not getattr(L, "_bm_ready", False):
            P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            I32P = ctypes.POINTER(ctypes.c_int32)
            I64P = ctypes.POINTER(ctypes.c_int64)
            L.pkv_bm_create.argtypes, L.pkv_bm_create.restype = [i64, i32], P
            L.pkv_bm_destroy.argtypes, L.pkv_bm_destroy.restype = [P], None
            L.pkv_bm_num_free.argtypes, L.pkv_bm_num_free.restype = [P], i64
            L.pkv_bm_get_computed_blocks.argtypes = [P, i64, I32P, i64]
            L.pkv_bm_allocate_slots.argtypes = [P, i64, i64]
            L.pkv_bm_cache_full_blocks.argtypes = [P, i64, I32P, i64]
            L.pkv_bm_block_table.argtypes = [P, i64, I32P, i32]
            L.pkv_bm_free.argtypes = [P, i64]
            L.pkv_bm_fork.argtypes = [P, i64, i64]
            L.pkv_bm_cow.argtypes = [P, i64, i32, I32P, I32P]
            L.pkv_bm_usage.argtypes = [P, I64P, I64P, I64P]
            L.pkv_bm_prefix_groups.argtypes = [P, I64P, i32, i32, i32, I32P, I32P, I32P, I32P]
            L.pkv_bm_block_hash.argtypes, L.pkv_bm_block_hash.restype = [ctypes.c_uint64, I32P, ctypes.c_uint64], \
                ctypes.c_uint64
            for f in ("pkv_bm_get_computed_blocks", "pkv_bm_allocate_slots", "pkv_bm_cache_full_blocks",
                      "pkv_bm_block_table", "pkv_bm_free", "pkv_bm_fork", "pkv_bm_cow", "pkv_bm_usage"):
                getattr(L, f).restype = ctypes.c_int32
            L._bm_ready = True
        self._L = L
        self._h = L.pkv_bm_create(int(num_blocks), 1 if enable_prefix_cache else 0)
        if not self._h:
            raise ValueError("bad block manager arguments")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._L.pkv_bm_destroy(h)

    @staticmethod
    def _i32(tokens):
        import numpy as np
        a = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def _ok(self, rc: int, what: str) -> int:
        if rc in (-2, -3):
            raise ValueError(f"{what}: {'unknown or duplicate request' if rc == -2 else 'bad argument'}")
        return rc

    @property
    def num_free(self) -> int:
        return int(self._L.pkv_bm_num_free(self._h))

    def get_computed_blocks(self, req: int, tokens) -> int:
        a, p = self._i32(tokens)
        return self._ok(self._L.pkv_bm_get_computed_blocks(self._h, req, p, a.size), "get_computed_blocks")

    def allocate_slots(self, req: int, total_tokens: int):
        """Number of blocks added, or None when the pool cannot cover the tokens."""
        rc = self._ok(self._L.pkv_bm_allocate_slots(self._h, req, int(total_tokens)), "allocate_slots")
        return None if rc == -1 else rc

    def cache_full_blocks(self, req: int, tokens) -> int:
        a, p = self._i32(tokens)
        return self._ok(self._L.pkv_bm_cache_full_blocks(self._h, req, p, a.size), "cache_full_blocks")

    def block_table(self, req: int) -> list:
        n = self._ok(self._L.pkv_bm_block_table(self._h, req, None, 0), "block_table")
        out = (ctypes.c_int32 * max(n, 1))()
        self._L.pkv_bm_block_table(self._h, req, out, n)
        return list(out[:n])

    def free(self, req: int) -> None:
        self._ok(self._L.pkv_bm_free(self._h, req), "free")

    def fork(self, parent: int, child: int) -> None:
        self._ok(self._L.pkv_bm_fork(self._h, parent, child), "fork")

    def cow(self, req: int, logical_block: int):
        """(src, dst) when the block was shared and is now a private copy, () when it was
        already exclusive, None when no block is free."""
        s, d = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = self._ok(self._L.pkv_bm_cow(self._h, req, int(logical_block), ctypes.byref(s), ctypes.byref(d)), "cow")
        return None if rc == -1 else ((s.value, d.value) if rc == 1 else ())

    def usage(self) -> dict:
        b, t, u = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        self._L.pkv_bm_usage(self._h, ctypes.byref(b), ctypes.byref(t), ctypes.byref(u))
        return {"blocks_in_use": b.value, "tokens_held": t.value, "unused_slots": u.value}

    def prefix_groups(self, reqs, max_prefix_blocks: int, max_groups: int | None = None):
        """Shared-prefix groups of the batch ``reqs`` (request ids in batch order), as
        (prefix_block_tables [G, max_prefix_blocks], prefix_num_blocks [G], member_start
        [G + 1], member_seqs) int32 numpy arrays for paged_attention_cascade / _step."""
        import numpy as np
        r = np.ascontiguousarray(np.asarray(reqs, dtype=np.int64).reshape(-1))
        n = int(r.size)
        mg = max(1, n // 2) if max_groups is None else int(max_groups)
        tables = np.empty((mg, int(max_prefix_blocks)), np.int32)
        nblk = np.empty(mg, np.int32)
        start = np.zeros(mg + 1, np.int32)
        members = np.empty(max(n, 1), np.int32)
        P32 = ctypes.POINTER(ctypes.c_int32)
        g = self._ok(self._L.pkv_bm_prefix_groups(
            self._h, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, int(max_prefix_blocks), mg,
            tables.ctypes.data_as(P32), nblk.ctypes.data_as(P32), start.ctypes.data_as(P32),
            members.ctypes.data_as(P32)), "prefix_groups")
        return tables[:g].copy(), nblk[:g].copy(), start[:g + 1].copy(), members[:start[g]].copy()

    def block_hash(self, parent: int, tokens16, extra: int = 0) -> int:
        a, p = self._i32(tokens16)
        if a.size != BLOCK_SIZE:
            raise ValueError("a block holds 16 tokens")
        return int(self._L.pkv_bm_block_hash(ctypes.c_uint64(parent), p, ctypes.c_uint64(extra)))
