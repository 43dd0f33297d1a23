"""CPU-only checks of the C ABI: the shared library loads, exports every
function include/pfkv.h declares, and its host-only paths (workspace sizing,
error strings, argument checks that return before any CUDA call) behave."""
import ctypes
import os
import re

import pytest

from paged_fp8_kv_quantize_gb300 import abi

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pfkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pfkv_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(abi.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(abi.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_entry_points():
    assert abi.lib.pfkv_abi_version() == 1
    assert abi.strerror(0) == "ok"
    assert "workspace" in abi.strerror(-5)
    d = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, 16)
    n = abi.lib.pfkv_decode_workspace_bytes(ctypes.byref(d), 64, 32, 64)
    # per-request piece index and count, (m, l) and O partials for every
    # (request, piece, head), a status word per piece and head group (at most
    # one group per query head) and an abort word per split CTA
    fixed = 64 * 64 * 32 * (8 + 4 * 128 + 4)
    assert fixed <= n < fixed + 64 * 1024


def test_argument_errors_return_before_any_cuda_call():
    f = abi.lib.pfkv_paged_decode_attention_fp8
    args_tail = [None, 32, None, None, None, 4, 8, 1.0, 0, 64, None, 0, None, None, None]
    assert f(None, *args_tail) == -1  # NULL cache
    bf16 = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_BF16, 0, 16, 16, None, None, None)
    assert f(ctypes.byref(bf16), *args_tail) == -4  # FP8 entry point, BF16 cache
    fp8 = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, None, None, None)
    assert f(ctypes.byref(fp8), *args_tail) == -1  # FP8 cache without scales
    bad = abi.CacheDesc(100, 16, 8, 128, 128, 0, 7, 0, 16, 16, 16, 16, None)
    assert f(ctypes.byref(bad), *args_tail) == -4  # unknown dtype
    unal = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 17, 16, 16, 16, None)
    assert f(ctypes.byref(unal), *args_tail) == -6  # misaligned pool
    g = abi.lib.pfkv_kv_append_quantize
    assert g(None, None, None, 0, None, None, None, None, 1, 1, 0, None, None) == -1
    # an empty batch is a valid call that enqueues nothing (no CUDA call is made)
    ok = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None)
    empty_tail = [None, 32, None, None, None, 0, 8, 1.0, 0, 64, None, 0, None, None, None]
    assert f(ctypes.byref(ok), *empty_tail) == 0
    assert g(ctypes.byref(ok), None, None, 0, None, None, None, None, 0, 1, 0, None, None) == 0
    # batch * max_pages above 2^40: the kernels' page arithmetic would leave
    # its exact range, so the call is refused (2^21 x 2^19 = 2^40 passes this
    # check and stops at the next one, the NULL buffers)
    big = [None, 32, None, None, None, 1 << 21, 1 << 20, 1.0, 0, 64, None, 0, None, None, None]
    assert f(ctypes.byref(ok), *big) == -2
    edge = [None, 32, None, None, None, 1 << 21, 1 << 19, 1.0, 0, 64, None, 0, None, None, None]
    assert f(ctypes.byref(ok), *edge) == -1


def test_workspace_size_bounds_and_huge_head_counts():
    # sizes a decode call refuses get no workspace size (SIZE_MAX), so that a
    # caller sizing a buffer from it cannot be handed a wrapped-around small
    # number; the decode itself refuses them before any CUDA call
    ok = abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None)
    size_max = ctypes.c_size_t(-1).value
    assert abi.lib.pfkv_decode_workspace_bytes(ctypes.byref(ok), 64, 1 << 30, 64) == size_max
    assert abi.lib.pfkv_decode_workspace_bytes(ctypes.byref(ok), 64, 32, 100000) == size_max
    wide = abi.CacheDesc(100, 16, 8, 128, 1 << 20, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None)
    assert abi.lib.pfkv_decode_workspace_bytes(ctypes.byref(wide), 64, 32, 64) == size_max
    f = abi.lib.pfkv_paged_decode_attention_fp8
    huge_heads = [None, 1 << 30, None, None, None, 4, 8, 1.0, 0, 64, None, 0, None, None, None]
    assert f(ctypes.byref(ok), *huge_heads) == -2


def test_noalloc_entry_point_checks_like_the_regular_one():
    # every bad argument gives the same code from both entry points, before
    # any device work (none of these calls reaches a CUDA call)
    f = abi.lib.pfkv_paged_decode_attention_fp8
    g = abi.lib.pfkv_paged_decode_attention_fp8_noalloc
    cases = [
        (None, 32, 4, 8, 64),                                                                  # NULL cache
        (abi.CacheDesc(100, 16, 8, 128, -5, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None), 32, 4, 8, 64),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_BF16, 0, 16, 16, None, None, None), 32, 4, 8, 64),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, 9, 0, 16, 16, 16, 16, None), 32, 4, 8, 64),  # unknown dtype
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 17, 16, 16, 16, None), 32, 4, 8, 64),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None), 0, 4, 8, 64),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None), 32, -1, 8, 64),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None), 32, 4, 8, 0),
        (abi.CacheDesc(100, 16, 8, 128, 128, 0, abi.DTYPE_FP8_E4M3, 0, 16, 16, 16, 16, None), 32, 4, 8, 300),
    ]
    for desc, hq, batch, mp, splits in cases:
        d = None if desc is None else ctypes.byref(desc)
        a = f(d, None, hq, None, None, None, batch, mp, 1.0, 0, splits, None, 0, None, None, None)
        b = g(d, None, hq, None, None, None, batch, mp, 1.0, 0, splits, None, None, None)
        assert a == b and a < 0, (a, b)


def test_page_allocator_host_checks():
    L = abi.lib
    n = L.pfkv_page_allocator_bytes(1000)
    # header + stack + scratch word + held flag per page + chunk counts
    assert 256 + 9 * 1000 <= n < 256 + 9 * 1000 + 4 * 256 + 64
    assert L.pfkv_page_allocator_bytes(0) == 0
    assert L.pfkv_page_allocator_init(None, n, 1000, None, 0, None) == -1
    assert L.pfkv_page_allocator_init(256, n, 0, None, 0, None) == -2
    assert L.pfkv_page_allocator_init(256, n - 1, 1000, None, 0, None) == -5
    assert L.pfkv_page_allocator_init(256, n, 1000, None, 3, None) == -1  # held ids missing
    assert L.pfkv_page_allocator_init(272, n, 1000, None, 0, None) == -6  # state not 256-byte aligned
    assert L.pfkv_page_alloc(256, 256, -1, None, None, 256, None) == -2
    assert L.pfkv_page_alloc(256, 256, 4, None, None, 256, None) == -1
    assert L.pfkv_page_free(256, None, 0, None, None) == 0  # nothing to do, nothing launched
    assert L.pfkv_page_free(256, None, 2, None, None) == -1
    assert L.pfkv_page_realloc(256, 256, None, 0, None, None, None) == 0
    assert L.pfkv_page_realloc(256, None, None, 1, None, None, None) == -1
