"""Seeded synthetic inputs for the paged KV cache.

This module only *draws* inputs: BF16 keys/values/queries, context lengths,
page tables, page tags and stale-tag injections.  It holds none of the
method's arithmetic (no scale, no quantization, no attention); both the CUDA
path and the CPU oracle consume exactly the arrays produced here.

Every array is host numpy.  BF16 values are carried as their uint16 bit
patterns (round-to-nearest-even from an fp32 draw).  Randomness is numpy's
PCG64 with the seed recorded on the workload.

Workload recipes (the shapes of the long-context decode workloads that the
post "Smaller, faster, safer: running Kimi and GLM at scale" serves; its
section "Quantizing the KV cache" names no sizes, so these are the stated
benchmark shapes):

  tiny     batch 2, lengths 37 and 100, 4 q heads / 1 KV head, D 64, page 16,
           pool of 32 shuffled pages, one stale block tag in request 1.
  gqa      batch 32, 32/8 heads, D 128, page 16, lengths U[1024, 8192],
           1% of K/V elements x20, pool 1.25x the pages needed.
  latent   batch 64, 64 q heads over one shared 576-wide stream (V = first
           512), page 64, lengths U[4096, 32768], per-token scales.
  long     batch 8, 131072 tokens each, 8/1 heads, D 128, page 64, pages
           scattered over a caller-sized pool, up to 64 splits.
  ragged   batch 64, lengths log-uniform in [1, 65536], 32/8 heads, D 128,
           page 16, room for 100 appended tokens per request, 100 decode
           steps of new K/V/q, 0.1% of used table entries stale after a
           simulated reallocation (the page's tag is bumped).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

PER_HEAD = 0
PER_TOKEN = 1


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng, shape, outlier_p=0.0, outlier_mult=20.0, chunk=1 << 24):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if outlier_p > 0.0:
            m = rng.random(e - s, dtype=np.float32) < outlier_p
            x[m] *= np.float32(outlier_mult)
        out[s:e] = bf16_bits(x)
    return out.reshape(shape)


@dataclass
class Workload:
    name: str
    seed: int
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    v_head_dim: int
    kv_shared: bool
    page_size: int
    num_pages: int
    max_pages: int
    scale_mode: int
    softmax_scale: float
    max_splits: int
    seq_lens: np.ndarray          # int32 [B]   (context before any decode step)
    block_table: np.ndarray       # int32 [B][MP], -1 where unassigned
    block_tags: np.ndarray        # uint32 [B][MP], expected tag per entry
    page_tags: np.ndarray         # uint32 [P], current tag per page
    q: np.ndarray                 # bf16 bits [B][Hq][D]
    k_rows: np.ndarray | None     # bf16 bits [N][Hkv][D]   all context tokens
    v_rows: np.ndarray | None     # bf16 bits [N][Hkv][Dv]  (None when shared)
    row_req: np.ndarray | None    # int32 [N]
    row_pos: np.ndarray | None    # int32 [N]
    steps: int = 0
    q_steps: np.ndarray | None = None   # [T][B][Hq][D]
    k_steps: np.ndarray | None = None   # [T][B][Hkv][D]
    v_steps: np.ndarray | None = None   # [T][B][Hkv][Dv]
    stale: list = field(default_factory=list)  # (b, i) entries made stale

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def rows_of(self, b: int):
        """Index range of request b's rows inside k_rows / v_rows."""
        off = int(self.seq_lens[:b].astype(np.int64).sum())
        return off, off + int(self.seq_lens[b])


def make(name, seed, *, batch, q_heads, kv_heads, head_dim, page_size, seq_lens, v_head_dim=None,
         kv_shared=False, scale_mode=PER_HEAD, softmax_scale=None, num_pages=None, pool_factor=1.25,
         room_tokens=0, outlier_p=0.0, steps=0, stale_block_entries=None, stale_page_fraction=0.0,
         max_splits=64, with_rows=True) -> Workload:
    """Draw one workload.  See the module docstring for the named recipes."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, S = int(batch), int(page_size)
    Dv = int(v_head_dim if v_head_dim is not None else head_dim)
    lens = np.asarray(seq_lens, dtype=np.int64)
    assert lens.shape == (B,)
    need = (lens + room_tokens + S - 1) // S
    MP = int(max(1, need.max()))
    total_pages = int(need.sum())
    P = int(num_pages if num_pages is not None else max(total_pages, math.ceil(pool_factor * total_pages)))
    assert P >= total_pages, "pool too small for the requests"
    # pages of each request: a sample without replacement from the whole pool
    perm = rng.permutation(P).astype(np.int64)
    table = np.full((B, MP), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(need[b])
        table[b, :n] = perm[off:off + n]
        off += n
    page_tags = rng.integers(0, 1 << 32, size=P, dtype=np.uint64).astype(np.uint32)
    block_tags = np.zeros((B, MP), dtype=np.uint32)
    valid = table >= 0
    block_tags[valid] = page_tags[table[valid]]

    stale = []
    used = [(b, i) for b in range(B) for i in range(int((lens[b] + S - 1) // S))]
    if stale_block_entries:
        # the mapping holds a wrong expected tag (e.g. a request holding an old mapping)
        for (b, i) in stale_block_entries:
            block_tags[b, i] ^= np.uint32(1)
            stale.append((b, i))
    if stale_page_fraction > 0.0 and used:
        k = max(1, int(round(stale_page_fraction * len(used))))
        pick = rng.choice(len(used), size=k, replace=False)
        for j in sorted(pick.tolist()):
            b, i = used[j]
            p = int(table[b, i])
            page_tags[p] = np.uint32((int(page_tags[p]) + 1) & 0xFFFFFFFF)  # simulated reallocation
            stale.append((b, i))

    q = _normal_bf16(rng, (B, q_heads, head_dim))
    k_rows = v_rows = row_req = row_pos = None
    if with_rows:
        N = int(lens.sum())
        k_rows = _normal_bf16(rng, (N, kv_heads, head_dim), outlier_p)
        v_rows = None if kv_shared else _normal_bf16(rng, (N, kv_heads, Dv), outlier_p)
        row_req = np.repeat(np.arange(B, dtype=np.int32), lens.astype(np.int64))
        row_pos = np.concatenate([np.arange(int(l), dtype=np.int32) for l in lens]) if N else np.zeros(0, np.int32)
    q_steps = k_steps = v_steps = None
    if steps:
        q_steps = _normal_bf16(rng, (steps, B, q_heads, head_dim))
        k_steps = _normal_bf16(rng, (steps, B, kv_heads, head_dim), outlier_p)
        v_steps = None if kv_shared else _normal_bf16(rng, (steps, B, kv_heads, Dv), outlier_p)
    tau = float(softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(head_dim))
    return Workload(name=name, seed=seed, batch=B, q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                    v_head_dim=Dv, kv_shared=kv_shared, page_size=S, num_pages=P, max_pages=MP,
                    scale_mode=scale_mode, softmax_scale=tau, max_splits=max_splits,
                    seq_lens=lens.astype(np.int32), block_table=table, block_tags=block_tags,
                    page_tags=page_tags, q=q, k_rows=k_rows, v_rows=v_rows, row_req=row_req, row_pos=row_pos,
                    steps=steps, q_steps=q_steps, k_steps=k_steps, v_steps=v_steps, stale=stale)


# ---------------------------------------------------------------- named recipes


def tiny(seed=1001) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    lens = [37, 100]
    # one used entry of request 1 gets a wrong expected tag
    stale_i = int(rng.integers(0, (100 + 15) // 16))
    return make("tiny", seed, batch=2, q_heads=4, kv_heads=1, head_dim=64, page_size=16, seq_lens=lens,
                num_pages=32, stale_block_entries=[(1, stale_i)], softmax_scale=1.0 / 8.0)


def gqa(seed=1002, batch=32, lo=1024, hi=8192, outlier_p=0.01) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    lens = rng.integers(lo, hi + 1, size=batch)
    return make("gqa", seed, batch=batch, q_heads=32, kv_heads=8, head_dim=128, page_size=16, seq_lens=lens,
                outlier_p=outlier_p)


def latent(seed=1003, batch=64, lo=4096, hi=32768) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    lens = rng.integers(lo, hi + 1, size=batch)
    return make("latent", seed, batch=batch, q_heads=64, kv_heads=1, head_dim=576, v_head_dim=512,
                kv_shared=True, page_size=64, seq_lens=lens, scale_mode=PER_TOKEN,
                softmax_scale=1.0 / math.sqrt(576.0))


def long_ctx(seed=1004, batch=8, length=131072, num_pages=None, with_rows=True) -> Workload:
    return make("long", seed, batch=batch, q_heads=8, kv_heads=1, head_dim=128, page_size=64,
                seq_lens=[length] * batch, num_pages=num_pages, max_splits=64, with_rows=with_rows)


def ragged(seed=1005, batch=64, max_len=65536, steps=100, stale_fraction=0.001, room=100) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    lens = np.floor(np.exp(rng.uniform(0.0, math.log(max_len), size=batch))).astype(np.int64)
    lens = np.clip(lens, 1, max_len)
    return make("ragged", seed, batch=batch, q_heads=32, kv_heads=8, head_dim=128, page_size=16, seq_lens=lens,
                room_tokens=room, steps=steps, stale_page_fraction=stale_fraction)
