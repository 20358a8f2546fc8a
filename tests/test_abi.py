"""The C ABI: the library builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
BLOCKS_HEADER = os.path.join(ROOT, "include", "pkv_blocks.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_248_gb300 import _build
    _build.build()
    import paged_kv_cache_248_gb300 as pkv
    return pkv.lib()


def declared_symbols(header=HEADER, macro="PKV_API"):
    text = open(header).read()
    return sorted(set(re.findall(rf"^{macro}\s+[\w\s\*]+?\b(\w+)\(", text, flags=re.M)))


def test_header_declares_the_hot_path_calls():
    names = declared_symbols()
    for n in ("pkv_slot_mapping", "pkv_write", "pkv_copy_blocks", "paged_attention", "pkv_get_last_error",
              "pkv_status_string", "pkv_shutdown"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols() + declared_symbols(BLOCKS_HEADER, "PKV_BM_API")
    assert "pkv_bm_allocate_slots" in names and "pkv_bm_cow" in names
    for name in names:
        assert hasattr(lib, name), f"libpkv does not export {name}"


def test_status_strings(lib):
    import paged_kv_cache_248_gb300 as pkv
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(3) == "PKV_ERR_INDEX"
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"


def _desc(pkv, nb=4, bs=16, hkv=1, d=64, dt=0):
    return pkv._CacheDesc(nb, bs, hkv, d, dt)


def test_host_argument_checks_fail_without_launching(lib):
    import paged_kv_cache_248_gb300 as pkv
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails its host checks first
    bad_block = _desc(pkv, bs=15)
    assert lib.pkv_write(fake, fake, fake, 1, fake, fake, ctypes.byref(bad_block), None) == pkv.PKV_ERR_INVALID_ARG
    unsupported = _desc(pkv, d=96)
    assert lib.pkv_write(fake, fake, fake, 1, fake, fake, ctypes.byref(unsupported), None) == pkv.PKV_ERR_UNSUPPORTED
    bf16_64 = _desc(pkv, d=64, dt=1)
    assert lib.pkv_copy_blocks(fake, fake, 1, fake, fake, ctypes.byref(bf16_64), None) == pkv.PKV_ERR_UNSUPPORTED
    ok = _desc(pkv)
    assert lib.pkv_write(None, fake, fake, 1, fake, fake, ctypes.byref(ok), None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_write(fake, fake, fake, -1, fake, fake, ctypes.byref(ok), None) == pkv.PKV_ERR_INVALID_ARG
    # zero tokens / pairs: nothing to do, success without any CUDA call
    assert lib.pkv_write(fake, fake, fake, 0, fake, fake, ctypes.byref(ok), None) == pkv.PKV_OK
    assert lib.pkv_copy_blocks(fake, fake, 0, fake, fake, ctypes.byref(ok), None) == pkv.PKV_OK
    # attention: group must divide, scale finite, hints positive
    two = _desc(pkv, hkv=2)
    assert lib.paged_attention(fake, fake, fake, ctypes.byref(two), fake, 1, fake, fake, 1, 3, 1, 1, 1,
                               ctypes.c_float(1.0), fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_attention(fake, fake, fake, ctypes.byref(ok), fake, 1, fake, fake, 1, 2, 1, 1, 1,
                               ctypes.c_float(float("inf")), fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_attention(fake, fake, fake, ctypes.byref(ok), fake, 1, fake, fake, 1, 2, 1, 0, 1,
                               ctypes.c_float(1.0), fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_attention(fake, fake, fake, ctypes.byref(ok), fake, 1, fake, fake, 1, 2, 0, 1, 1,
                               ctypes.c_float(1.0), fake, None) == pkv.PKV_OK
    misaligned = P(0x1004)
    assert lib.paged_attention(misaligned, fake, fake, ctypes.byref(ok), fake, 1, fake, fake, 1, 2, 1, 1, 1,
                               ctypes.c_float(1.0), fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_slot_mapping(fake, 0, fake, fake, 1, 1, fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_slot_mapping(fake, 1, fake, fake, 1, 0, fake, None) == pkv.PKV_OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import paged_kv_cache_248_gb300 as pkv
    kc = torch.zeros(4, 1, 16, 64)
    with pytest.raises(ValueError):
        pkv.pkv_write(torch.zeros(1, 1, 64), torch.zeros(1, 1, 64), torch.zeros(1, dtype=torch.int64), kc,
                      kc.clone())


def test_cascade_host_checks_fail_without_launching(lib):
    import paged_kv_cache_248_gb300 as pkv
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: each call below fails its host checks first
    desc = _desc(pkv, d=128, dt=1)
    args = (fake, fake, fake, ctypes.byref(desc), fake, 4, fake, fake, 2, 8, 2, 1, 64, ctypes.c_float(0.1))
    g = pkv._PrefixGroups(fake, 4, fake, fake, fake, -1, 3)
    assert lib.paged_attention_cascade(*args, ctypes.byref(g), fake, None) == pkv.PKV_ERR_INVALID_ARG
    g = pkv._PrefixGroups(None, 4, fake, fake, fake, 2, 3)       # a group array missing
    assert lib.paged_attention_cascade(*args, ctypes.byref(g), fake, None) == pkv.PKV_ERR_INVALID_ARG
    g = pkv._PrefixGroups(fake, 0, fake, fake, fake, 2, 3)       # max_prefix_blocks < 1
    assert lib.paged_attention_cascade(*args, ctypes.byref(g), fake, None) == pkv.PKV_ERR_INVALID_ARG
    bad_scale = args[:-1] + (ctypes.c_float(float("nan")),)
    assert lib.paged_attention_cascade(*bad_scale, None, fake, None) == pkv.PKV_ERR_INVALID_ARG


def test_step_with_copies_host_checks_fail_without_launching(lib):
    import paged_kv_cache_248_gb300 as pkv
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: each call below fails its host checks first
    desc = _desc(pkv, d=128, dt=1)
    head = (fake, fake, fake, fake, fake, ctypes.byref(desc), fake, 4, fake, fake, 2, 8, 2, 1, 64,
            ctypes.c_float(0.1), None)
    assert lib.paged_attention_step_cow(*head, fake, fake, -1, None, fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_attention_step_cow(*head, None, fake, 3, None, fake, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_attention_step_cow(*head, fake, None, 3, None, fake, None) == pkv.PKV_ERR_INVALID_ARG
    no_new = (fake, None) + head[2:]
    assert lib.paged_attention_step_cow(*no_new, fake, fake, 3, None, fake, None) == pkv.PKV_ERR_INVALID_ARG


def test_noalloc_refuses_too_many_split_items_like_paged_attention(lib):
    # 2^20 requests x 8 kv heads x ceil(2^19 / 2048) splits = 2^31 items: both calls
    # refuse the batch as unsupported on the host, before any CUDA call
    import paged_kv_cache_248_gb300 as pkv
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn = lib.paged_attention_noalloc
    fn.argtypes = [P, P, P, ctypes.POINTER(pkv._CacheDesc), P, i32, P, P, i32, i32, i64, i32, i32,
                   ctypes.c_float, P, P, P]
    fn.restype = ctypes.c_int
    fake = P(0x1000)
    desc = _desc(pkv, nb=1 << 20, hkv=8, d=128, dt=1)
    n, max_len = 1 << 20, 1 << 19
    args = (fake, fake, fake, ctypes.byref(desc), fake, max_len // 16, fake, fake, n, 32, n, 1, max_len,
            ctypes.c_float(0.1), fake)
    assert fn(*args, None, None) == pkv.PKV_ERR_UNSUPPORTED
    assert lib.paged_attention(*args, None) == pkv.PKV_ERR_UNSUPPORTED
