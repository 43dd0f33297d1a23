"""Test-side helpers: run the CPU oracle on a synthetic workload, and build an
independent dense reference with library routines (torch float8 decode and
torch scaled_dot_product_attention in fp64).  Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_fp8_kv_quantize_gb300 import synth


def oracle_cache(w: synth.Workload, dtype=oracle.DTYPE_FP8, fill_flags=0, sentinel=0xA5):
    """Calibrate (per-head mode) and fill an oracle cache with every context row."""
    ks = vs = None
    if dtype == oracle.DTYPE_FP8 and w.scale_mode == synth.PER_HEAD:
        ks = oracle.calibrate_per_head(w.k_rows)
        vs = None if w.kv_shared else oracle.calibrate_per_head(w.v_rows)
    c = oracle.Cache(w.num_pages, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, dtype,
                     w.scale_mode if dtype == oracle.DTYPE_FP8 else synth.PER_HEAD, w.page_tags, ks, vs,
                     sentinel=sentinel)
    st = c.append(w.k_rows, w.v_rows, w.row_pos, w.block_table, w.block_tags, flags=fill_flags,
                  row_req=w.row_req, batch=w.batch)
    return c, st


def dequant_pool(c: oracle.Cache, which="k"):
    """[P][H][S][D] float64 values of a pool, decoded by torch (library)."""
    pool = c.k_pool if which == "k" else c.v_pool
    D = c.D if which == "k" else c.Dv
    if c.dtype == oracle.DTYPE_FP8:
        vals = torch.from_numpy(pool).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        scale = c.k_scale if which == "k" else c.v_scale
        vals = vals.reshape(c.P, c.H, c.S, D)
        if c.scale_mode == oracle.SCALE_PER_TOKEN:
            return vals * scale.astype(np.float64).reshape(c.P, c.H, c.S, 1)
        return vals * scale.astype(np.float64).reshape(1, c.H, 1, 1)
    vals = torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return vals.reshape(c.P, c.H, c.S, D)


def dense_reference(c: oracle.Cache, q_bits, seq_lens, block_table, tau):
    """Unpage each request into contiguous K/V and call torch SDPA (fp64)."""
    K = dequant_pool(c, "k")
    V = K[..., : c.Dv] if c.kv_shared else dequant_pool(c, "v")
    q = torch.from_numpy(np.ascontiguousarray(q_bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, c.Dv))
    for b in range(B):
        L = int(seq_lens[b])
        n = (L + c.S - 1) // c.S
        pages = block_table[b, :n]
        kb = K[pages].transpose(1, 0, 2, 3).reshape(c.H, n * c.S, D)[:, :L]
        vb = V[pages].transpose(1, 0, 2, 3).reshape(c.H, n * c.S, c.Dv)[:, :L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].reshape(1, Hq, 1, D), torch.from_numpy(kb).unsqueeze(0), torch.from_numpy(vb).unsqueeze(0),
            scale=tau, enable_gqa=True)
        out[b] = o.reshape(Hq, c.Dv).numpy()
    return out


def oracle_cache_subset(w: synth.Workload, idx, dtype=oracle.DTYPE_FP8, scales=None):
    """Oracle cache holding only requests `idx`, page ids renumbered densely.

    Per-head scales are calibrated over ALL of the workload's rows (as the GPU
    path does) unless given.  Returns (cache, table, tags, used_pages) where
    used_pages[k] is the workload's page id stored at compact page k."""
    idx = np.asarray(idx)
    tab = w.block_table[idx]
    used = np.unique(tab[tab >= 0])
    remap = np.full(w.num_pages, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    ctab = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
    ks = vs = None
    if dtype == oracle.DTYPE_FP8 and w.scale_mode == synth.PER_HEAD:
        ks, vs = scales if scales is not None else (oracle.calibrate_per_head(w.k_rows),
                                                    None if w.kv_shared else oracle.calibrate_per_head(w.v_rows))
    c = oracle.Cache(used.size, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, dtype,
                     w.scale_mode if dtype == oracle.DTYPE_FP8 else synth.PER_HEAD, w.page_tags[used], ks, vs)
    sel = np.isin(w.row_req, idx)
    rr = np.searchsorted(idx, w.row_req[sel]).astype(np.int32)
    c.append(w.k_rows[sel], None if w.kv_shared else w.v_rows[sel], w.row_pos[sel], ctab, w.block_tags[idx],
             row_req=rr, batch=idx.size)
    return c, ctab, w.block_tags[idx].copy(), used
