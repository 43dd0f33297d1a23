"""Thin ctypes binding of libpfkv (include/pfkv.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  If the
shared library is missing this module raises on import -- there is no other
implementation behind it.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpfkv.so")

DTYPE_BF16 = 0
DTYPE_FP8_E4M3 = 1
SCALE_PER_HEAD = 0
SCALE_PER_TOKEN = 1
FLAG_TAG_CHECK = 1
FLAG_TEST_WITHHOLD = 0x80000000  # test hook: the grouped-query decode's abort path (see pfkv.h)
ST_STALE_TAG = 1
ST_PAGE_OOB = 2
ST_BAD_LEN = 4
ST_TIMEOUT = 8
ST_NO_PAGES = 16
ST_NOT_HELD = 32
ST_DUPLICATE = 64

EXPORTS = (
    "pfkv_kv_append_quantize",
    "pfkv_decode_workspace_bytes",
    "pfkv_paged_decode_attention_fp8",
    "pfkv_paged_decode_attention_bf16",
    "pfkv_paged_decode_attention_fp8_noalloc",
    "pfkv_paged_decode_step",
    "pfkv_handoff_bf16_to_fp8",
    "pfkv_page_allocator_bytes",
    "pfkv_page_allocator_init",
    "pfkv_page_alloc",
    "pfkv_page_free",
    "pfkv_page_realloc",
    "pfkv_calibrate_scales",
    "pfkv_e4m3_encode",
    "pfkv_strerror",
    "pfkv_last_error_detail",
    "pfkv_abi_version",
)


class PfkvError(RuntimeError):
    def __init__(self, fn, code):
        detail = lib.pfkv_last_error_detail().decode() if code == -7 else ""
        super().__init__(f"{fn} failed: {code} ({strerror(code)}){': ' + detail if detail else ''}")
        self.code = code


class CacheDesc(ctypes.Structure):
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


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpfkv.so is not built ({LIB_PATH}); run paged_fp8_kv_quantize_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    cp = ctypes.POINTER(CacheDesc)
    L.pfkv_kv_append_quantize.restype = ctypes.c_int
    L.pfkv_kv_append_quantize.argtypes = [cp, P, P, i32, P, P, P, P, i32, i32, u32, P, P]
    L.pfkv_decode_workspace_bytes.restype = sz
    L.pfkv_decode_workspace_bytes.argtypes = [cp, i32, i32, i32]
    for n in ("pfkv_paged_decode_attention_fp8", "pfkv_paged_decode_attention_bf16"):
        f = getattr(L, n)
        f.restype = ctypes.c_int
        f.argtypes = [cp, P, i32, P, P, P, i32, i32, ctypes.c_float, u32, i32, P, sz, P, P, P]
    L.pfkv_paged_decode_attention_fp8_noalloc.restype = ctypes.c_int
    L.pfkv_paged_decode_attention_fp8_noalloc.argtypes = [cp, P, i32, P, P, P, i32, i32, ctypes.c_float, u32, i32,
                                                          P, P, P]
    L.pfkv_paged_decode_step.restype = ctypes.c_int
    L.pfkv_paged_decode_step.argtypes = [cp, P, P, P, i32, P, P, P, i32, i32, ctypes.c_float, u32, i32, P, sz, P, P,
                                         P]
    L.pfkv_handoff_bf16_to_fp8.restype = ctypes.c_int
    L.pfkv_handoff_bf16_to_fp8.argtypes = [cp, cp, P, P, i32, P, P]
    L.pfkv_page_allocator_bytes.restype = sz
    L.pfkv_page_allocator_bytes.argtypes = [i32]
    L.pfkv_page_allocator_init.restype = ctypes.c_int
    L.pfkv_page_allocator_init.argtypes = [P, sz, i32, P, i32, P]
    L.pfkv_page_alloc.restype = ctypes.c_int
    L.pfkv_page_alloc.argtypes = [P, P, i32, P, P, P, P]
    L.pfkv_page_free.restype = ctypes.c_int
    L.pfkv_page_free.argtypes = [P, P, i32, P, P]
    L.pfkv_page_realloc.restype = ctypes.c_int
    L.pfkv_page_realloc.argtypes = [P, P, P, i32, P, P, P]
    L.pfkv_calibrate_scales.restype = ctypes.c_int
    L.pfkv_calibrate_scales.argtypes = [P, i64, i32, i32, P, P]
    L.pfkv_e4m3_encode.restype = ctypes.c_int
    L.pfkv_e4m3_encode.argtypes = [P, P, i64, P]
    L.pfkv_strerror.restype = ctypes.c_char_p
    L.pfkv_strerror.argtypes = [ctypes.c_int]
    L.pfkv_last_error_detail.restype = ctypes.c_char_p
    L.pfkv_last_error_detail.argtypes = []
    L.pfkv_abi_version.restype = ctypes.c_int
    L.pfkv_abi_version.argtypes = []
    return L


lib = _load()


def strerror(code: int) -> str:
    return lib.pfkv_strerror(int(code)).decode()


def _check(fn, rc):
    if rc != 0:
        raise PfkvError(fn, rc)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


class PagedCache:
    """Device-resident paged KV cache (pools, scales, page tags) + its descriptor.

    Layout: k_pool [P][Hkv][S][D], v_pool [P][Hkv][S][Dv] (uint8 e4m3 codes or
    bf16); scales per head [Hkv] or per token [P][Hkv][S]; page_tags [P] uint32
    (stored as int32 -- torch has no uint32 arithmetic on every version).
    """

    def __init__(self, num_pages, page_size, num_kv_heads, head_dim, v_head_dim=None, kv_shared=False,
                 dtype=DTYPE_FP8_E4M3, scale_mode=SCALE_PER_HEAD, device="cuda", fill=None, alloc_pools=True):
        self.P, self.S, self.H, self.D = int(num_pages), int(page_size), int(num_kv_heads), int(head_dim)
        self.Dv = int(v_head_dim if v_head_dim is not None else head_dim)
        self.kv_shared, self.dtype, self.scale_mode = bool(kv_shared), int(dtype), int(scale_mode)
        self.device = torch.device(device)
        el = torch.uint8 if self.dtype == DTYPE_FP8_E4M3 else torch.bfloat16
        rows = self.P * self.H * self.S
        self.k_pool = self.v_pool = None
        if alloc_pools:
            self.k_pool = torch.empty(rows * self.D, dtype=el, device=self.device)
            self.v_pool = None if kv_shared else torch.empty(rows * self.Dv, dtype=el, device=self.device)
            if fill is not None:
                self.fill_pools(fill)
        if self.dtype == DTYPE_FP8_E4M3:
            n = rows if self.scale_mode == SCALE_PER_TOKEN else self.H
            self.k_scale = torch.ones(n, dtype=torch.float32, device=self.device)
            self.v_scale = None if kv_shared else torch.ones(n, dtype=torch.float32, device=self.device)
        else:
            self.k_scale = self.v_scale = None
        self.page_tags = torch.zeros(self.P, dtype=torch.int32, device=self.device)

    def fill_pools(self, byte):
        for t in (self.k_pool, self.v_pool):
            if t is not None:
                t.view(torch.uint8).fill_(int(byte))

    def desc(self) -> CacheDesc:
        return CacheDesc(self.P, self.S, self.H, self.D, self.Dv, int(self.kv_shared), self.dtype, self.scale_mode,
                         _ptr(self.k_pool), _ptr(self.v_pool), _ptr(self.k_scale), _ptr(self.v_scale),
                         _ptr(self.page_tags))

    def k_rows(self):
        return self.k_pool.view(self.P, self.H, self.S, self.D)

    def v_rows(self):
        return None if self.v_pool is None else self.v_pool.view(self.P, self.H, self.S, self.Dv)


def kv_append_quantize(cache: PagedCache, k_new, v_new, positions, block_table, block_tags=None, flags=0,
                       row_req=None, batch=None, status=None, stream=None):
    """Quantize-and-append rows (see pfkv_kv_append_quantize).  Returns status [batch] (int32 view of uint32)."""
    i32 = torch.int32
    n_rows = positions.shape[0]
    B, MP = block_table.shape
    batch = B if batch is None else int(batch)
    if status is None:
        status = torch.empty(batch, dtype=i32, device=block_table.device)
    d = cache.desc()
    rc = lib.pfkv_kv_append_quantize(
        ctypes.byref(d), _ptr(_dev(k_new, "k_new", torch.bfloat16)),
        _ptr(_dev(v_new, "v_new", torch.bfloat16)) if v_new is not None else None, n_rows,
        _ptr(_dev(row_req, "row_req", i32)), _ptr(_dev(positions, "positions", i32)),
        _ptr(_dev(block_table, "block_table", i32)), _ptr(_dev(block_tags, "block_tags", i32)), batch, MP,
        int(flags), _ptr(_dev(status, "status", i32)), _stream(stream))
    _check("pfkv_kv_append_quantize", rc)
    return status


def decode_workspace_bytes(cache: PagedCache, batch, num_q_heads, max_splits=64) -> int:
    d = cache.desc()
    return int(lib.pfkv_decode_workspace_bytes(ctypes.byref(d), int(batch), int(num_q_heads), int(max_splits)))


def _decode(fn_name, cache, q, seq_lens, block_table, block_tags, softmax_scale, flags, max_splits, workspace, out,
            status, stream):
    B, Hq, D = q.shape
    MP = block_table.shape[1]
    dev = q.device
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(cache, B, Hq, max_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(B, Hq, cache.Dv, dtype=torch.float32, device=dev)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    d = cache.desc()
    rc = getattr(lib, fn_name)(
        ctypes.byref(d), _ptr(_dev(q, "q", torch.bfloat16)), Hq, _ptr(_dev(seq_lens, "seq_lens", torch.int32)),
        _ptr(_dev(block_table, "block_table", torch.int32)), _ptr(_dev(block_tags, "block_tags", torch.int32)), B,
        MP, float(softmax_scale), int(flags), int(max_splits), _ptr(workspace), workspace.numel(),
        _ptr(_dev(out, "out", torch.float32)), _ptr(_dev(status, "status", torch.int32)), _stream(stream))
    _check(fn_name, rc)
    return out, status


def paged_decode_attention_fp8(cache, q, seq_lens, block_table, block_tags, softmax_scale, flags=0, max_splits=64,
                               workspace=None, out=None, status=None, stream=None):
    return _decode("pfkv_paged_decode_attention_fp8", cache, q, seq_lens, block_table, block_tags, softmax_scale,
                   flags, max_splits, workspace, out, status, stream)


def paged_decode_attention_bf16(cache, q, seq_lens, block_table, block_tags, softmax_scale, flags=0, max_splits=64,
                                workspace=None, out=None, status=None, stream=None):
    return _decode("pfkv_paged_decode_attention_bf16", cache, q, seq_lens, block_table, block_tags, softmax_scale,
                   flags, max_splits, workspace, out, status, stream)


def paged_decode_step(cache, k_new, v_new, q, seq_lens, block_table, block_tags, softmax_scale, flags=0,
                      max_splits=64, workspace=None, out=None, status=None, stream=None):
    """Append each request's new token (k_new/v_new bf16 [B][Hkv][D], position
    seq_lens[b] - 1) and attend, in one call (pfkv_paged_decode_step)."""
    B, Hq, D = q.shape
    MP = block_table.shape[1]
    dev = q.device
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(cache, B, Hq, max_splits), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(B, Hq, cache.Dv, dtype=torch.float32, device=dev)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    d = cache.desc()
    rc = lib.pfkv_paged_decode_step(
        ctypes.byref(d), _ptr(_dev(k_new, "k_new", torch.bfloat16)),
        _ptr(_dev(v_new, "v_new", torch.bfloat16)) if v_new is not None else None, _ptr(_dev(q, "q", torch.bfloat16)),
        Hq, _ptr(_dev(seq_lens, "seq_lens", torch.int32)), _ptr(_dev(block_table, "block_table", torch.int32)),
        _ptr(_dev(block_tags, "block_tags", torch.int32)), B, MP, float(softmax_scale), int(flags), int(max_splits),
        _ptr(workspace), workspace.numel(), _ptr(_dev(out, "out", torch.float32)),
        _ptr(_dev(status, "status", torch.int32)), _stream(stream))
    _check("pfkv_paged_decode_step", rc)
    return out, status


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # PFKV_NOALLOC_SCRATCH_BYTES


def paged_decode_attention_fp8_noalloc(cache, q, seq_lens, block_table, block_tags, softmax_scale, flags=0,
                                       max_splits=64, out=None, status=None, stream=None):
    """FP8 decode without a caller-provided workspace (see pfkv_paged_decode_attention_fp8_noalloc).

    For callers that cannot allocate device scratch: the library uses its own
    fixed buffer of NOALLOC_SCRATCH_BYTES.  Pass `out` and `status` to keep the
    call free of allocations on the Python side as well; calls that overlap on
    the GPU race on the shared buffer."""
    B, Hq, D = q.shape
    MP = block_table.shape[1]
    if out is None:
        out = torch.empty(B, Hq, cache.Dv, dtype=torch.float32, device=q.device)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=q.device)
    d = cache.desc()
    rc = lib.pfkv_paged_decode_attention_fp8_noalloc(
        ctypes.byref(d), _ptr(_dev(q, "q", torch.bfloat16)), Hq, _ptr(_dev(seq_lens, "seq_lens", torch.int32)),
        _ptr(_dev(block_table, "block_table", torch.int32)), _ptr(_dev(block_tags, "block_tags", torch.int32)), B,
        MP, float(softmax_scale), int(flags), int(max_splits), _ptr(_dev(out, "out", torch.float32)),
        _ptr(_dev(status, "status", torch.int32)), _stream(stream))
    _check("pfkv_paged_decode_attention_fp8_noalloc", rc)
    return out, status


def paged_decode_attention(cache, *args, **kw):
    """Dispatch on the cache dtype to the FP8 or BF16 entry point."""
    f = paged_decode_attention_fp8 if cache.dtype == DTYPE_FP8_E4M3 else paged_decode_attention_bf16
    return f(cache, *args, **kw)


def handoff_bf16_to_fp8(src: PagedCache, dst: PagedCache, src_pages, dst_pages, page_status=None, stream=None):
    """Quantize pages src_pages[i] of a BF16 cache into pages dst_pages[i] of an FP8 cache."""
    n = src_pages.shape[0]
    if page_status is None:
        page_status = torch.empty(n, dtype=torch.int32, device=src_pages.device)
    ds, dd = src.desc(), dst.desc()
    rc = lib.pfkv_handoff_bf16_to_fp8(ctypes.byref(ds), ctypes.byref(dd),
                                      _ptr(_dev(src_pages, "src_pages", torch.int32)),
                                      _ptr(_dev(dst_pages, "dst_pages", torch.int32)), n,
                                      _ptr(_dev(page_status, "page_status", torch.int32)), _stream(stream))
    _check("pfkv_handoff_bf16_to_fp8", rc)
    return page_status


class PageAllocator:
    """Device-resident free list over num_pages pages (pfkv_page_allocator_*).

    Every hand-out (alloc, realloc) advances the page's tag in the cache's
    page_tags; the returned tags go into the new owner's block_tags."""

    def __init__(self, num_pages, held_pages=None, device="cuda", stream=None):
        self.num_pages = int(num_pages)
        nbytes = lib.pfkv_page_allocator_bytes(self.num_pages)
        if nbytes == 0:
            raise PfkvError("pfkv_page_allocator_bytes", -2)
        self.state = torch.empty(nbytes, dtype=torch.uint8, device=device)  # torch blocks are 512-byte aligned
        n_held, hp = 0, None
        if held_pages is not None:
            hp = _dev(held_pages, "held_pages", torch.int32)
            n_held = hp.numel()
        rc = lib.pfkv_page_allocator_init(_ptr(self.state), nbytes, self.num_pages, _ptr(hp) if n_held else None,
                                          n_held, _stream(stream))
        _check("pfkv_page_allocator_init", rc)

    def alloc(self, n, page_tags, stream=None):
        """-> (pages int32 [n], tags int32 [n] (uint32 bits), status int32 [1]) on the device."""
        dev = self.state.device
        pages = torch.empty(max(n, 1), dtype=torch.int32, device=dev)[:n]
        tags = torch.empty(max(n, 1), dtype=torch.int32, device=dev)[:n]
        status = torch.empty(1, dtype=torch.int32, device=dev)
        rc = lib.pfkv_page_alloc(_ptr(self.state), _ptr(_dev(page_tags, "page_tags", torch.int32)), int(n),
                                 _ptr(pages) if n else None, _ptr(tags) if n else None, _ptr(status), _stream(stream))
        _check("pfkv_page_alloc", rc)
        return pages, tags, status

    def free(self, pages, stream=None):
        pages = _dev(pages, "pages", torch.int32)
        st = torch.zeros(pages.numel(), dtype=torch.int32, device=self.state.device)
        rc = lib.pfkv_page_free(_ptr(self.state), _ptr(pages), pages.numel(), _ptr(st), _stream(stream))
        _check("pfkv_page_free", rc)
        return st

    def realloc(self, pages, page_tags, stream=None):
        pages = _dev(pages, "pages", torch.int32)
        n = pages.numel()
        tags = torch.zeros(n, dtype=torch.int32, device=self.state.device)
        st = torch.zeros(n, dtype=torch.int32, device=self.state.device)
        rc = lib.pfkv_page_realloc(_ptr(self.state), _ptr(_dev(page_tags, "page_tags", torch.int32)), _ptr(pages), n,
                                   _ptr(tags), _ptr(st), _stream(stream))
        _check("pfkv_page_realloc", rc)
        return tags, st

    def free_count(self):
        """Reads the state's free count (synchronises with the device)."""
        return int(self.state[4:8].view(torch.int32).item())

    def free_list(self):
        """Free ids, bottom of the stack first (synchronises with the device)."""
        fc = self.free_count()
        return self.state[256:256 + 4 * self.num_pages].view(torch.int32)[:fc].clone()


def calibrate_scales(rows, scale=None, stream=None):
    """rows: bf16 [N][H][D] -> fp32 scale[H] = amax/448 (1 for an all-zero head)."""
    N, H, D = rows.shape
    if scale is None:
        scale = torch.empty(H, dtype=torch.float32, device=rows.device)
    rc = lib.pfkv_calibrate_scales(_ptr(_dev(rows, "rows", torch.bfloat16)), N, H, D,
                                   _ptr(_dev(scale, "scale", torch.float32)), _stream(stream))
    _check("pfkv_calibrate_scales", rc)
    return scale


def e4m3_encode(x, out=None, stream=None):
    x = _dev(x, "x", torch.float32)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    rc = lib.pfkv_e4m3_encode(_ptr(x), _ptr(out), x.numel(), _stream(stream))
    _check("pfkv_e4m3_encode", rc)
    return out
