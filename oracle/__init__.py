"""CPU oracle for the paged FP8 KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never touches it, and it never touches the product path: the two
share no code.  The arithmetic lives in ``pfkv_oracle.c`` (plain C, fp64);
this module only compiles it and marshals numpy arrays.

Sources: "Smaller, faster, safer: running Kimi and GLM at scale" (Cloudflare),
section "Quantizing the KV cache" (FP8 e4m3 cache, converted as it is read)
and its cache-protection passage (per-page tag, compared before the read,
abort on mismatch, off by default).  Readings R1-R10 are listed in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pfkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Interface numbers (the same values as the library's header, restated).
DTYPE_BF16 = 0
DTYPE_FP8 = 1
SCALE_PER_HEAD = 0
SCALE_PER_TOKEN = 1
FLAG_TAG_CHECK = 1
ST_STALE_TAG = 1
ST_PAGE_OOB = 2
ST_BAD_LEN = 4
ST_NO_PAGES = 16
ST_NOT_HELD = 32
ST_DUPLICATE = 64


def build(force: bool = False) -> str:
    """Compile pfkv_oracle.c into liboracle.so next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cache(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("kv_shared", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("page_tags", ctypes.c_void_p),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode_nearest.restype = ctypes.c_uint8
            L.orc_e4m3_encode_nearest.argtypes = [ctypes.c_float]
            L.orc_quantize.restype = ctypes.c_uint8
            L.orc_quantize.argtypes = [ctypes.c_uint16, ctypes.c_float]
            L.orc_scale_from_amax.restype = ctypes.c_float
            L.orc_scale_from_amax.argtypes = [ctypes.c_double]
            for name in ("orc_e4m3_encode_array", "orc_e4m3_encode_nearest_array", "orc_e4m3_encode_bits"):
                getattr(L, name).restype = None
                getattr(L, name).argtypes = [P, P, i64]
            L.orc_e4m3_sweep.restype = u64
            L.orc_e4m3_sweep.argtypes = [u64, u64, ctypes.c_int, ctypes.POINTER(u64)]
            L.orc_calibrate_per_head.restype = None
            L.orc_calibrate_per_head.argtypes = [P, i64, i32, i32, P]
            L.orc_append.restype = None
            L.orc_append.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, u32, P]
            L.orc_handoff.restype = None
            L.orc_handoff.argtypes = [P, P, P, P, i32, P]
            L.orc_alloc_init.restype = None
            L.orc_alloc_init.argtypes = [P, P, P, i32, P, i32]
            L.orc_page_alloc.restype = None
            L.orc_page_alloc.argtypes = [P, P, P, P, i32, P, P, P]
            L.orc_page_free.restype = None
            L.orc_page_free.argtypes = [P, P, P, i32, P, i32, P]
            L.orc_page_realloc.restype = None
            L.orc_page_realloc.argtypes = [P, i32, P, P, i32, P, P]
            L.orc_decode.restype = None
            L.orc_decode.argtypes = [P, P, i32, P, P, P, i32, i32, ctypes.c_double, u32, P, P, i32]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codec


def e4m3_decode(codes) -> np.ndarray:
    """Decoded value of each e4m3 code, fp64 (NaN for the NaN codes)."""
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([L.orc_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def e4m3_encode(y) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_array(_ptr(y), _ptr(out), y.size)
    return out


def e4m3_encode_nearest(y) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_nearest_array(_ptr(y), _ptr(out), y.size)
    return out


def e4m3_encode_bits(bits) -> np.ndarray:
    b = _c(bits, np.uint32)
    out = np.empty(b.shape, dtype=np.uint8)
    lib().orc_e4m3_encode_bits(_ptr(b), _ptr(out), b.size)
    return out


def e4m3_sweep(lo: int, hi: int, threads: int = 0):
    """Disagreements between the two encoders over fp32 bit patterns [lo, hi)."""
    first = ctypes.c_uint64(0)
    n = lib().orc_e4m3_sweep(lo, hi, threads or os.cpu_count() or 1, ctypes.byref(first))
    return int(n), (None if n == 0 else int(first.value))


def quantize(x_bf16_bits, s) -> int:
    return int(lib().orc_quantize(int(x_bf16_bits), float(s)))


def scale_from_amax(amax: float) -> float:
    return float(lib().orc_scale_from_amax(float(amax)))


def calibrate_per_head(rows_bf16) -> np.ndarray:
    """rows_bf16: uint16 bf16 bits [N][H][D] -> fp32 scale[H] = amax/448."""
    x = _c(rows_bf16, np.uint16)
    n, H, D = x.shape
    s = np.empty(H, dtype=np.float32)
    lib().orc_calibrate_per_head(_ptr(x), n, H, D, _ptr(s))
    return s


# ---------------------------------------------------------------- cache


class Cache:
    """Host-memory paged cache in the oracle's own arrays."""

    def __init__(self, num_pages, page_size, num_kv_heads, head_dim, v_head_dim=None, kv_shared=False,
                 dtype=DTYPE_FP8, scale_mode=SCALE_PER_HEAD, page_tags=None, k_scale=None, v_scale=None,
                 sentinel=0xA5):
        self.P, self.S, self.H, self.D = int(num_pages), int(page_size), int(num_kv_heads), int(head_dim)
        self.Dv = int(v_head_dim if v_head_dim is not None else head_dim)
        self.kv_shared, self.dtype, self.scale_mode = bool(kv_shared), int(dtype), int(scale_mode)
        rows = self.P * self.H * self.S
        if self.dtype == DTYPE_FP8:
            self.k_pool = np.full(rows * self.D, sentinel, dtype=np.uint8)
            self.v_pool = None if kv_shared else np.full(rows * self.Dv, sentinel, dtype=np.uint8)
        else:
            sv = (sentinel << 8) | sentinel
            self.k_pool = np.full(rows * self.D, sv, dtype=np.uint16)
            self.v_pool = None if kv_shared else np.full(rows * self.Dv, sv, dtype=np.uint16)
        if self.scale_mode == SCALE_PER_TOKEN:
            self.k_scale = np.zeros(rows, dtype=np.float32)
            self.v_scale = None if kv_shared else np.zeros(rows, dtype=np.float32)
        else:
            self.k_scale = _c(k_scale if k_scale is not None else np.ones(self.H), np.float32)
            self.v_scale = None if kv_shared else _c(v_scale if v_scale is not None else np.ones(self.H), np.float32)
        self.page_tags = _c(page_tags if page_tags is not None else np.zeros(self.P), np.uint32)

    def _struct(self):
        return _Cache(self.P, self.S, self.H, self.D, self.Dv, int(self.kv_shared), self.dtype, self.scale_mode,
                      _ptr(self.k_pool), _ptr(self.v_pool), _ptr(self.k_scale), _ptr(self.v_scale),
                      _ptr(self.page_tags))

    def append(self, k_new, v_new, positions, block_table, block_tags, flags=0, row_req=None, batch=None):
        k = _c(k_new, np.uint16)
        v = None if self.kv_shared else _c(v_new, np.uint16)
        pos = _c(positions, np.int32)
        bt = _c(block_table, np.int32)
        tags = _c(block_tags, np.uint32)
        rr = None if row_req is None else _c(row_req, np.int32)
        B, MP = bt.shape
        n = pos.shape[0]
        batch = B if batch is None else batch
        status = np.zeros(batch, dtype=np.uint32)
        cs = self._struct()
        lib().orc_append(ctypes.byref(cs), _ptr(k), _ptr(v), n, _ptr(rr), _ptr(pos), _ptr(bt), _ptr(tags),
                         batch, MP, flags, _ptr(status))
        return status

    def decode(self, q, seq_lens, block_table, block_tags, softmax_scale, flags=0, threads=1):
        qq = _c(q, np.uint16)
        B, Hq, D = qq.shape
        lens = _c(seq_lens, np.int32)
        bt = _c(block_table, np.int32)
        tags = _c(block_tags, np.uint32)
        out = np.zeros((B, Hq, self.Dv), dtype=np.float64)
        status = np.zeros(B, dtype=np.uint32)
        cs = self._struct()
        lib().orc_decode(ctypes.byref(cs), _ptr(qq), Hq, _ptr(lens), _ptr(bt), _ptr(tags), B, bt.shape[1],
                         float(softmax_scale), flags, _ptr(out), _ptr(status), threads)
        return out, status

    def handoff_from(self, src: "Cache", src_pages, dst_pages):
        """Quantize pages of a BF16 oracle cache into this FP8 cache; returns page status."""
        sp = _c(src_pages, np.int32)
        dp = _c(dst_pages, np.int32)
        st = np.zeros(sp.shape[0], dtype=np.uint32)
        cs, cd = src._struct(), self._struct()
        lib().orc_handoff(ctypes.byref(cs), ctypes.byref(cd), _ptr(sp), _ptr(dp), sp.shape[0], _ptr(st))
        return st

    # views for comparison
    def k_rows(self):
        return self.k_pool.reshape(self.P, self.H, self.S, self.D)

    def v_rows(self):
        return None if self.v_pool is None else self.v_pool.reshape(self.P, self.H, self.S, self.Dv)


# ---------------------------------------------------------------- page allocator


class Allocator:
    """The oracle's sequential page allocator over a tag array it does not own."""

    def __init__(self, num_pages, page_tags, held_pages=()):
        self.P = int(num_pages)
        self.page_tags = page_tags  # uint32 [P], updated in place
        assert self.page_tags.dtype == np.uint32 and self.page_tags.flags.c_contiguous
        self.stack = np.zeros(self.P, dtype=np.int32)
        self.held = np.zeros(self.P, dtype=np.uint8)
        self.count = np.zeros(1, dtype=np.int32)
        hp = _c(np.asarray(held_pages, dtype=np.int64), np.int32)
        lib().orc_alloc_init(_ptr(self.stack), _ptr(self.held), _ptr(self.count), self.P, _ptr(hp), hp.size)

    @property
    def free_count(self):
        return int(self.count[0])

    def free_list(self):
        """Free ids, bottom of the stack first."""
        return self.stack[: self.free_count].copy()

    def alloc(self, n):
        pages = np.zeros(n, dtype=np.int32)
        tags = np.zeros(n, dtype=np.uint32)
        st = np.zeros(1, dtype=np.uint32)
        lib().orc_page_alloc(_ptr(self.stack), _ptr(self.held), _ptr(self.count), _ptr(self.page_tags), int(n),
                             _ptr(pages), _ptr(tags), _ptr(st))
        return pages, tags, int(st[0])

    def free(self, pages):
        pg = _c(pages, np.int32)
        st = np.zeros(pg.size, dtype=np.uint32)
        lib().orc_page_free(_ptr(self.stack), _ptr(self.held), _ptr(self.count), self.P, _ptr(pg), pg.size, _ptr(st))
        return st

    def realloc(self, pages):
        pg = _c(pages, np.int32)
        tags = np.zeros(pg.size, dtype=np.uint32)
        st = np.zeros(pg.size, dtype=np.uint32)
        lib().orc_page_realloc(_ptr(self.held), self.P, _ptr(self.page_tags), _ptr(pg), pg.size, _ptr(tags), _ptr(st))
        return tags, st
