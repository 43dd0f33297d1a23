"""GPU-side test helpers: upload a synthetic workload and build the cache
through the library's own entry points (calibrate + append).  Nothing here
computes the method; the oracle side lives in oracle_helpers.py."""
from __future__ import annotations

import numpy as np
import torch

from paged_fp8_kv_quantize_gb300 import abi, synth

ABS_TOL = 2e-3  # max |out_gpu - out_oracle|
REL_TOL = 1e-2  # max |err| / max |out_oracle| per (request, head) row


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a.astype(np.int32, copy=False)).cuda()


class DeviceCase:
    """Device copies of a workload's tables plus a filled GPU cache."""

    def __init__(self, w: synth.Workload, dtype=abi.DTYPE_FP8_E4M3, sentinel=0xA5, fill_flags=0, num_pages=None,
                 fill=True):
        self.w = w
        P = w.num_pages if num_pages is None else num_pages
        scale_mode = w.scale_mode if dtype == abi.DTYPE_FP8_E4M3 else abi.SCALE_PER_HEAD
        self.cache = abi.PagedCache(P, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, dtype,
                                    scale_mode, fill=sentinel)
        self.cache.page_tags.copy_(dev_i32(w.page_tags))
        self.table = dev_i32(w.block_table)
        self.tags = dev_i32(w.block_tags)
        self.seq_lens = dev_i32(w.seq_lens)
        self.q = dev_bf16(w.q)
        self.fill_status = None
        if fill and w.k_rows is not None:
            k = dev_bf16(w.k_rows)
            v = None if w.kv_shared else dev_bf16(w.v_rows)
            if dtype == abi.DTYPE_FP8_E4M3 and scale_mode == abi.SCALE_PER_HEAD:
                abi.calibrate_scales(k, self.cache.k_scale)
                if v is not None:
                    abi.calibrate_scales(v, self.cache.v_scale)
            self.fill_status = abi.kv_append_quantize(self.cache, k, v, dev_i32(w.row_pos), self.table, self.tags,
                                                      flags=fill_flags, row_req=dev_i32(w.row_req), batch=w.batch)
            del k, v

    def decode(self, flags=0, max_splits=None, q=None, seq_lens=None, table=None, tags=None):
        w = self.w
        out, st = abi.paged_decode_attention(
            self.cache, self.q if q is None else q, self.seq_lens if seq_lens is None else seq_lens,
            self.table if table is None else table, self.tags if tags is None else tags, w.softmax_scale,
            flags=flags, max_splits=w.max_splits if max_splits is None else max_splits)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64), st.cpu().numpy().view(np.uint32)


def assert_close(out_gpu, out_ref, where=""):
    err = np.abs(out_gpu - out_ref)
    mx = float(err.max()) if err.size else 0.0
    assert mx <= ABS_TOL, f"{where}: max abs err {mx:.3e} > {ABS_TOL}"
    ref_row = np.abs(out_ref).max(axis=-1)
    rel = err.max(axis=-1) / np.maximum(ref_row, 1e-6)
    assert float(rel.max()) <= REL_TOL, f"{where}: max row-relative err {float(rel.max()):.3e} > {REL_TOL}"
    return mx
