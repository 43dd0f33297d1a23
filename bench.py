#!/usr/bin/env python3
"""Benchmark: FP8 paged decode attention with the tag check, batch 64.

Workload (one "step" = the whole hot path once): the mixed ragged batch --
64 requests with context lengths log-uniform in [1, 65536], 32 query / 8 KV
heads, head_dim 128, 16-token pages, FP8 e4m3 cache with per-head scales,
0.1% of the used page-table entries stale after a simulated reallocation.
Each step appends one new token per request (quantize-on-append) and then
runs tag-checked paged decode attention over every request's context.

Prints ONE JSON line (rank 0).  value = algorithmic KV GB/s of the step with
inputs resident in HBM; e2e = the same with per-step inputs copied from
pinned host memory and results copied back inside the timed region (on a
second stream, double-buffered, overlapping the neighbouring steps).
Inputs are larger than L2 (the cache alone is ~0.8 GB), so no flush.
Also reported: per-call p50/p95 (one-call graphs, events between replays),
the tag check's on/off ratio with a bootstrap interval and its p95, the BF16
cache, the other benchmark shapes (grouped-query batch, long contexts over
a pool of 80% of the free memory and over a dense pool, the latent stream),
and the CPU oracle on the host cores (all cores and one thread on the ragged
batch, all cores on the other shapes).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_fp8_kv_quantize_gb300 import synth  # noqa: E402

METRIC = "FP8 paged decode-attention KV GB/s and tokens/s at batch 64 (% of HBM peak)"
WORKLOAD = ("mixed ragged decode: batch 64, lengths log-uniform [1, 65536], 32 q / 8 KV heads, head_dim 128, "
            "page 16, FP8 e4m3 per-head scales, tag check on, 0.1% stale entries; step = append 1 token/request "
            "+ paged decode attention")


# ---------------------------------------------------------------- accounting


def decode_alg_bytes(lens, Hkv, D, S, Hq, Dv, fp8=True, tag_check=True):
    """Algorithmic bytes of one decode call: KV rows + table/tag words + q + out."""
    lens = np.asarray(lens, dtype=np.int64)
    per_tok = 2 * Hkv * D * (1 if fp8 else 2)
    pages = (lens + S - 1) // S
    b = int(lens.sum()) * per_tok + int(pages.sum()) * (8 + (4 if tag_check else 0))
    b += len(lens) * Hq * D * 2 + len(lens) * Hq * Dv * 4
    return b


def append_alg_bytes(B, Hkv, D, fp8=True):
    # bf16 rows in, cache rows out (K and V), positions + table entries
    return B * (2 * Hkv * D * 2 + 2 * Hkv * D * (1 if fp8 else 2) + 12)


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ---------------------------------------------------------------- peaks


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def fp8_dense_peak_tflops():
    """Dense e4m3 tensor peak: the measured bf16 GEMM burst figure times the
    nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s), or the fallback bf16 figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 x 2"
    return 2.0 * 1900.0, "fallback bf16 x 2"


def global_max(value, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (the job's time is its slowest rank)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def percentile(xs, q):
    xs = sorted(xs)
    if not xs:
        return None
    k = (len(xs) - 1) * q / 100.0
    lo, hi = int(math.floor(k)), int(math.ceil(k))
    return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)


def bootstrap_ci(xs, stat=statistics.median, n=2000, seed=7):
    """95% percentile-bootstrap interval of stat over the samples xs."""
    rng = np.random.default_rng(seed)
    arr = np.asarray(xs, dtype=np.float64)
    vals = [stat(arr[rng.integers(0, arr.size, arr.size)]) for _ in range(n)]
    return [percentile(vals, 2.5), percentile(vals, 97.5)]


def job_throughput(units_per_rank, world, max_ms):
    """Whole-job rate: every rank runs the same replica, timed by the slowest."""
    return world * units_per_rank / (max_ms * 1e-3)


def recorded_traffic():
    """DRAM bytes per launch of the split kernel from the committed ncu record,
    or None when the kernel sources changed since the counters were taken."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "gqa_split_fp8_ragged_b64.traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    for rel, digest in rec["sources"].items():
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return rec["dram_bytes_read"] + rec["dram_bytes_write"]


# ---------------------------------------------------------------- CPU oracle leg


def oracle_step_sample(w, frac, threads=None):
    """Build the oracle's cache for a bounded sample of requests; return a callable step.

    The oracle runs with the tag check off: it skips the attention of an
    aborted request entirely, so with the check on it would do less work
    than the GPU, which reads every page before it knows a request aborts."""
    import oracle

    total = w.total_tokens
    idx, acc = [], 0
    for b in range(w.batch):
        idx.append(b)
        acc += int(w.seq_lens[b])
        if acc >= frac * total:
            break
    idx = np.array(idx)
    # compact page ids for the sample (bookkeeping only)
    tab = w.block_table[idx]
    used = np.unique(tab[tab >= 0])
    remap = np.full(w.num_pages, -1, dtype=np.int64)
    remap[used] = np.arange(used.size)
    ctab = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
    ks = oracle.calibrate_per_head(w.k_rows)
    vs = oracle.calibrate_per_head(w.v_rows)
    c = oracle.Cache(used.size, w.page_size, w.kv_heads, w.head_dim, page_tags=w.page_tags[used], k_scale=ks,
                     v_scale=vs)
    sel = np.isin(w.row_req, idx)
    rr = np.searchsorted(idx, w.row_req[sel]).astype(np.int32)
    c.append(w.k_rows[sel], w.v_rows[sel], w.row_pos[sel], ctab, w.block_tags[idx], row_req=rr, batch=idx.size)
    threads = threads or len(os.sched_getaffinity(0))
    lens0 = w.seq_lens[idx].astype(np.int32)
    state = {"j": 0}

    def step():
        j = state["j"] % max(1, w.steps)
        state["j"] += 1
        pos = lens0 + j
        c.append(w.k_steps[j][idx], w.v_steps[j][idx], pos, ctab, w.block_tags[idx], flags=0)
        c.decode(w.q_steps[j][idx], pos + 1, ctab, w.block_tags[idx], w.softmax_scale, flags=0, threads=threads)
        return decode_alg_bytes(pos + 1, w.kv_heads, w.head_dim, w.page_size, w.q_heads, w.v_head_dim) + \
            append_alg_bytes(idx.size, w.kv_heads, w.head_dim)

    desc = (f"{idx.size} of {w.batch} requests ({int(lens0.sum())} of {total} context tokens), full step each, "
            f"tag check off")
    return step, threads, desc, idx.size


def oracle_config_timings(latent_w=None):
    """The oracle as it stands, timed on the host cores on the other
    benchmark shapes: the tiny, grouped-query and long-context batches in
    full, and one call of the latent-stream batch (decode only; the cache is
    built first).  Returns {name: {...}}."""
    import oracle

    threads = len(os.sched_getaffinity(0))
    res = {}

    def one(name, w, fp8_per_head=True):
        idx = np.arange(w.batch)
        tab = w.block_table
        used = np.unique(tab[tab >= 0])
        remap = np.full(w.num_pages, -1, dtype=np.int64)
        remap[used] = np.arange(used.size)
        ctab = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
        ks = vs = None
        if fp8_per_head:
            ks = oracle.calibrate_per_head(w.k_rows)
            vs = None if w.kv_shared else oracle.calibrate_per_head(w.v_rows)
        c = oracle.Cache(used.size, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, oracle.DTYPE_FP8,
                         w.scale_mode, w.page_tags[used], ks, vs)
        c.append(w.k_rows, w.v_rows, w.row_pos, ctab, w.block_tags, row_req=w.row_req, batch=w.batch)
        t0 = time.perf_counter()
        c.decode(w.q, w.seq_lens, ctab, w.block_tags, w.softmax_scale, flags=0, threads=threads)
        dt = time.perf_counter() - t0
        if w.kv_shared:
            tokens = int(w.seq_lens.astype(np.int64).sum())
            pages = int(((w.seq_lens.astype(np.int64) + w.page_size - 1) // w.page_size).sum())
            nbytes = tokens * (w.head_dim + 4) + pages * 8 + w.q.size * 2 + w.batch * w.q_heads * w.v_head_dim * 4
        else:
            nbytes = decode_alg_bytes(w.seq_lens, w.kv_heads, w.head_dim, w.page_size, w.q_heads, w.head_dim,
                                      tag_check=False)
        res[name] = {"seconds": dt, "value": nbytes / dt / 1e9, "unit": "GB/s", "cores": threads,
                     "context_tokens": int(w.seq_lens.astype(np.int64).sum()), "tag_check": "off"}
        del c

    one("tiny", synth.tiny())
    one("gqa", synth.gqa())
    one("long", synth.long_ctx())
    if latent_w is not None:
        one("latent_one_call", latent_w, fp8_per_head=False)
    return res


def run_reference(args, w):
    """The oracle as it stands, timed on the host cores (the reference arm).

    Each step is a bounded sample of the workload, sized so that the whole
    K + W steps stay around a minute and a half of wall time."""
    frac = min(args.cpu_frac, 2.0e7 / max(1, args.steps + args.warmup) / max(1, w.total_tokens))
    step, threads, desc, nb = oracle_step_sample(w, frac)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    tot = 0
    for _ in range(args.steps):
        tot += step()
    dt = time.perf_counter() - t0
    gbs = tot / dt / 1e9
    return {"metric": METRIC, "value": gbs, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "seed": w.seed, "sample": desc},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- GPU leg


def bench_latent(abi, wl, dev, i32, bf16, capture, time_graph, peak, n_calls):
    """Tag-checked decode over the latent-shared workload (64 requests,
    lengths U[4096, 32768], 576-wide stream, per-token scales, page 64)."""
    import torch

    B, S = wl.batch, wl.page_size
    cache = abi.PagedCache(wl.num_pages, S, 1, wl.head_dim, wl.v_head_dim, True, abi.DTYPE_FP8_E4M3,
                           abi.SCALE_PER_TOKEN, device=dev, fill=0)
    cache.page_tags.copy_(i32(wl.page_tags))
    table, tags, lens = i32(wl.block_table), i32(wl.block_tags), i32(wl.seq_lens)
    k = bf16(wl.k_rows)
    abi.kv_append_quantize(cache, k, None, i32(wl.row_pos), table, tags, row_req=i32(wl.row_req), batch=B)
    del k
    q = bf16(wl.q)
    ws = torch.empty(abi.decode_workspace_bytes(cache, B, wl.q_heads, wl.max_splits), dtype=torch.uint8, device=dev)
    out = torch.empty(B, wl.q_heads, wl.v_head_dim, dtype=torch.float32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)

    def call(_, flags=abi.FLAG_TAG_CHECK):
        abi.paged_decode_attention_fp8(cache, q, lens, table, tags, wl.softmax_scale, flags=flags,
                                       max_splits=wl.max_splits, workspace=ws, out=out, status=st)

    for _ in range(3):
        call(0)
    g = capture(call, n_calls)
    g.replay()
    ms = time_graph(g) / n_calls
    g1 = capture(call, 1)
    g1.replay()
    each = time_graph.each(g1, 30)
    # tag check on / off, alternated (all tags valid)
    g_off = capture(lambda j: call(j, flags=0), n_calls)
    g_off.replay()
    ratios = []
    for _ in range(5):
        a, b = time_graph(g), time_graph(g_off)
        ratios.append(a / b)
    tokens = int(wl.seq_lens.astype(np.int64).sum())
    pages = int(((wl.seq_lens.astype(np.int64) + S - 1) // S).sum())
    nbytes = tokens * (wl.head_dim + 4) + pages * 12 + q.numel() * 2 + out.numel() * 4
    flops = tokens * wl.q_heads * (wl.head_dim + wl.v_head_dim) * 2
    # The tensor cores run e4m3 MMAs over whole pages: S = [T1; T2] K^T (two
    # query terms, 128 rows x 576) and O^T += V^T (P1 + P2 + P3)^T (three
    # probability terms, 512 values x 64 heads).
    mma_flops = pages * S * (2 * 2 * wl.q_heads * wl.head_dim + 2 * 3 * wl.q_heads * wl.v_head_dim)
    tpeak, tpeak_kind = fp8_dense_peak_tflops()
    tach = flops / (ms * 1e-3) / 1e12
    return {"workload": "latent-shared stream: batch 64, lengths U[4096, 32768], 64 q heads over one 576-wide "
                        "FP8 stream (V = first 512), per-token scales, page 64, tag check on",
            "us_per_call": ms * 1e3, "p50_us": statistics.median(each) * 1e3, "p95_us": percentile(each, 95) * 1e3,
            "kv_gbs": nbytes / (ms * 1e-3) / 1e9, "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak,
            "tflops": flops / (ms * 1e-3) / 1e12, "context_tokens": tokens, "alg_bytes_per_call": nbytes,
            "decode_tokens_per_s": B / (ms * 1e-3), "aborted_requests": int((st.cpu().numpy() != 0).sum()),
            "tag_check_ratio_on_over_off": statistics.median(ratios),
            "roofline": {"bound": "tensor", "kernel": "latent_tc_kernel + merge_kernel", "achieved": tach,
                         "peak": tpeak, "peak_kind": tpeak_kind, "unit": "TFLOP/s", "frac": tach / tpeak,
                         "flops_per_call": flops, "what": "algorithmic flops: 2 x 64 heads x (576 + 512) per token",
                         "executed_mma_flops_per_call": mma_flops,
                         "executed_frac": mma_flops / (ms * 1e-3) / 1e12 / tpeak,
                         "executed_what": "e4m3 MMA work as issued: query terms x2, probability terms x3 (x4 on pages "
                                          "with values above 8), whole pages"}}



def bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls, dtype, num_pages=None):
    """Decode-only timing of one workload (all rows appended first)."""
    import torch

    fp8 = dtype == abi.DTYPE_FP8_E4M3
    P = w.num_pages if num_pages is None else num_pages
    cache = abi.PagedCache(P, w.page_size, w.kv_heads, w.head_dim, dtype=dtype, device=dev, fill=0)
    cache.page_tags.copy_(i32(w.page_tags))
    table, tags, lens = i32(w.block_table), i32(w.block_tags), i32(w.seq_lens)
    k, v = bf16(w.k_rows), bf16(w.v_rows)
    if fp8:
        abi.calibrate_scales(k, cache.k_scale)
        abi.calibrate_scales(v, cache.v_scale)
    abi.kv_append_quantize(cache, k, v, i32(w.row_pos), table, tags, row_req=i32(w.row_req), batch=w.batch)
    del k, v
    q = bf16(w.q)
    ws = torch.empty(abi.decode_workspace_bytes(cache, w.batch, w.q_heads, w.max_splits), dtype=torch.uint8,
                     device=dev)
    out = torch.empty(w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device=dev)
    st = torch.empty(w.batch, dtype=torch.int32, device=dev)

    def call(_):
        abi.paged_decode_attention(cache, q, lens, table, tags, w.softmax_scale, flags=abi.FLAG_TAG_CHECK,
                                   max_splits=w.max_splits, workspace=ws, out=out, status=st)

    for _ in range(3):
        call(0)
    g = capture(call, n_calls)
    g.replay()
    ms = time_graph(g) / n_calls
    g1 = capture(call, 1)
    g1.replay()
    each = time_graph.each(g1, 30)
    nbytes = decode_alg_bytes(w.seq_lens, w.kv_heads, w.head_dim, w.page_size, w.q_heads, w.head_dim, fp8=fp8)
    res = {"us_per_call": ms * 1e3, "p50_us": statistics.median(each) * 1e3, "p95_us": percentile(each, 95) * 1e3,
           "kv_gbs": nbytes / (ms * 1e-3) / 1e9,
           "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak, "alg_bytes_per_call": nbytes,
           "aborted_requests": int((st.cpu().numpy() != 0).sum()), "pool_pages": P}
    del cache, ws
    torch.cuda.empty_cache()
    return res


def bench_configs(abi, dev, i32, bf16, capture, time_graph, peak, n_calls):
    """The other shapes of the benchmark table: the tiny batch, the grouped-query batch and the long-context batch."""
    import torch

    res = {}
    w = synth.tiny()
    res["tiny"] = {"workload": "batch 2, lengths 37 and 100, 4 q / 1 KV head, head_dim 64, page 16, pool of 32, "
                               "one stale entry, tag check on (launch-bound)",
                   "fp8": bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls,
                                              abi.DTYPE_FP8_E4M3)}
    w = synth.gqa()
    res["gqa"] = {"workload": "batch 32, lengths U[1024, 8192], 32 q / 8 KV heads, head_dim 128, page 16, "
                              "1% outliers x20, tag check on",
                  "fp8": bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls,
                                             abi.DTYPE_FP8_E4M3),
                  "bf16": bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls,
                                              abi.DTYPE_BF16)}
    del w
    # long contexts: pages scattered over a pool that fills ~80% of the free
    # device memory (each cache type in turn, the same byte budget), and the
    # same batch over a dense pool (1.25x the pages needed, permuted), which
    # separates the cost of scattering the pages over the whole device
    res["long"] = {"workload": "batch 8 x 131072 tokens, 8 q / 1 KV head, head_dim 128, page 64, tag check on"}
    for name, dtype, esz in (("fp8", abi.DTYPE_FP8_E4M3, 1), ("bf16", abi.DTYPE_BF16, 2)):
        free, _ = torch.cuda.mem_get_info(dev)
        big = int(0.8 * free) // (2 * 64 * 128 * esz)
        w = synth.long_ctx(num_pages=big)
        r = bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls, dtype, num_pages=big)
        r["pool"] = f"{big} pages scattered over {big * 2 * 64 * 128 * esz / 2**30:.1f} GiB (80% of the free memory)"
        res["long"][name] = r
        del w
        w = synth.long_ctx()
        r = bench_decode_config(abi, w, dev, i32, bf16, capture, time_graph, peak, n_calls, dtype)
        r["pool"] = "1.25x the pages needed, permuted (dense)"
        res["long"][name + "_dense_pool"] = r
        del w
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-frac", type=float, default=0.5, help="share of context tokens in the CPU sample")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="minimum wall time of the CPU oracle leg (whole steps are repeated until it is reached)")
    ap.add_argument("--no-variants", action="store_true", help="skip the BF16 / tag-off comparisons")
    ap.add_argument("--no-latent", action="store_true", help="skip the latent-stream measurement")
    ap.add_argument("--batch", type=int, default=64,
                    help="requests of the mixed ragged workload (the first N of the seeded batch of 64); "
                         "smaller batches are for profiler captures, the reported figure is batch 64")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if not 1 <= args.batch <= 64:
        ap.error("--batch must be in [1, 64]")
    w = synth.ragged(batch=args.batch)  # seeded; every rank draws the same replica
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return

    import torch

    from paged_fp8_kv_quantize_gb300 import abi

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    def i32(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a.astype(np.int32)).to(dev)

    B, Hq, Hkv, D, S, T = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.page_size, w.steps
    table, tags = i32(w.block_table), i32(w.block_tags)
    lens0 = w.seq_lens.astype(np.int64)
    pos_steps = i32(np.stack([lens0 + j for j in range(T)]))            # [T][B]
    len_steps = i32(np.stack([lens0 + j + 1 for j in range(T)]))        # [T][B]
    q_steps, k_steps, v_steps = bf16(w.q_steps), bf16(w.k_steps), bf16(w.v_steps)

    def make_cache(dtype):
        c = abi.PagedCache(w.num_pages, S, Hkv, D, dtype=dtype, device=dev, fill=0)
        c.page_tags.copy_(i32(w.page_tags))
        return c

    caches = {"fp8": make_cache(abi.DTYPE_FP8_E4M3)}
    if not args.no_variants:
        caches["bf16"] = make_cache(abi.DTYPE_BF16)
    k_rows, v_rows = bf16(w.k_rows), bf16(w.v_rows)
    abi.calibrate_scales(k_rows, caches["fp8"].k_scale)
    abi.calibrate_scales(v_rows, caches["fp8"].v_scale)
    rr, rp = i32(w.row_req), i32(w.row_pos)
    for c in caches.values():
        abi.kv_append_quantize(c, k_rows, v_rows, rp, table, tags, row_req=rr, batch=B)  # prefill hand-off
    del k_rows, v_rows
    torch.cuda.synchronize()

    max_splits = w.max_splits
    ws = torch.empty(abi.decode_workspace_bytes(caches["fp8"], B, Hq, max_splits), dtype=torch.uint8, device=dev)
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
    st_dec = torch.empty(B, dtype=torch.int32, device=dev)
    st_app = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    FLAGS = abi.FLAG_TAG_CHECK

    def step(cache, j, flags=FLAGS, do_append=True):
        """One decode step: the fused call (new tokens written by the split kernel's page loader, then attention)."""
        j %= T
        if do_append:
            abi.paged_decode_step(cache, k_steps[j], v_steps[j], q_steps[j], len_steps[j], table, tags,
                                  w.softmax_scale, flags=flags, max_splits=max_splits, workspace=ws, out=out,
                                  status=st_dec)
        else:
            abi.paged_decode_attention(cache, q_steps[j], len_steps[j], table, tags, w.softmax_scale, flags=flags,
                                       max_splits=max_splits, workspace=ws, out=out, status=st_dec)

    def step_unfused(cache, j, flags=FLAGS):
        """The same step as two calls: kv_append_quantize, then paged decode attention."""
        j %= T
        abi.kv_append_quantize(cache, k_steps[j], v_steps[j], pos_steps[j], table, tags, flags=flags, status=st_app)
        abi.paged_decode_attention(cache, q_steps[j], len_steps[j], table, tags, w.softmax_scale, flags=flags,
                                   max_splits=max_splits, workspace=ws, out=out, status=st_dec)

    def capture(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for j in range(n):
                fn(j)
        return g

    def time_graph(g, reps=1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return global_max(e0.elapsed_time(e1), dist, dev)

    def time_each(g, n):
        """Per-replay times (ms) of n back-to-back replays (events between them)."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(n):
            g.replay()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]

    time_graph.each = time_each

    K = args.steps
    fp8 = caches["fp8"]
    # warm-up: W untimed steps
    for j in range(args.warmup):
        step(fp8, j)
    torch.cuda.synchronize()

    # ---- headline: K full steps (append + decode), inputs resident in HBM
    g_step = capture(lambda j: step(fp8, j), K)
    g_step.replay()  # untimed replay (graph upload)
    with ClockSampler(local) as clk:
        ms_step = time_graph(g_step)
    ms_per_step = ms_step / K
    step_bytes = [decode_alg_bytes(lens0 + j % T + 1, Hkv, D, S, Hq, D) + append_alg_bytes(B, Hkv, D) for j in range(K)]
    value = job_throughput(sum(step_bytes), world, ms_step) / 1e9
    dec_bytes = [decode_alg_bytes(lens0 + j % T + 1, Hkv, D, S, Hq, D) for j in range(K)]

    # ---- dominant kernel group: decode alone (split + merge), same stream
    g_dec = capture(lambda j: step(fp8, j, do_append=False), K)
    g_dec.replay()
    ms_dec = time_graph(g_dec) / K
    dec_gbs = statistics.mean(dec_bytes) / (ms_dec * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    # per-call distribution: one call per graph, 60 back-to-back replays with
    # an event between replays (inputs larger than L2, so no flush)
    g1_step = capture(lambda j: step(fp8, j), 1)
    g1_dec = capture(lambda j: step(fp8, j, do_append=False), 1)
    g1_step.replay()
    g1_dec.replay()
    each_step, each_dec = time_each(g1_step, 60), time_each(g1_dec, 60)
    per_call = {"step": {"p50_us": statistics.median(each_step) * 1e3, "p95_us": percentile(each_step, 95) * 1e3,
                         "replays": 60},
                "decode": {"p50_us": statistics.median(each_dec) * 1e3, "p95_us": percentile(each_dec, 95) * 1e3,
                           "replays": 60},
                "what": "one call per CUDA graph, replayed back to back, CUDA events between replays"}

    extra = {}
    if not args.no_variants:
        # tag-check overhead: interleaved replays, median ratio.  Both arms run
        # with every tag valid so that they do identical work apart from the
        # check (with stale tags the aborted requests skip their merge).
        valid_np = w.page_tags.copy()
        used = w.block_table >= 0
        valid_np[w.block_table[used]] = w.block_tags[used]
        stale_tags = fp8.page_tags
        valid_tags = i32(valid_np)  # kept alive while the graphs below use it
        fp8.page_tags = valid_tags
        g_on = capture(lambda j: step(fp8, j, do_append=False), K)
        g_off = capture(lambda j: step(fp8, j, flags=0, do_append=False), K)
        g1_on = capture(lambda j: step(fp8, j, do_append=False), 1)
        g1_off = capture(lambda j: step(fp8, j, flags=0, do_append=False), 1)
        fp8.page_tags = stale_tags
        for gg in (g_on, g_off, g1_on, g1_off):
            gg.replay()
        ratios, on_ms, off_ms = [], [], []
        n_alt = 21
        for _ in range(n_alt):
            a = time_graph(g_on)
            b = time_graph(g_off)
            on_ms.append(a)
            off_ms.append(b)
            ratios.append(a / b)
        each_on, each_off = [], []
        for _ in range(3):  # per-call distributions, interleaved in blocks of 20 replays
            each_on += time_each(g1_on, 20)
            each_off += time_each(g1_off, 20)
        extra["tag_check_overhead"] = {
            "median_ratio_on_over_off": statistics.median(ratios), "ratio_ci95": bootstrap_ci(ratios),
            "on_us_per_call": statistics.median(on_ms) / K * 1e3, "off_us_per_call": statistics.median(off_ms) / K * 1e3,
            "alternations": n_alt,
            "p95_ratio_on_over_off": percentile(each_on, 95) / percentile(each_off, 95),
            "on_p50_us": statistics.median(each_on) * 1e3, "on_p95_us": percentile(each_on, 95) * 1e3,
            "off_p50_us": statistics.median(each_off) * 1e3, "off_p95_us": percentile(each_off, 95) * 1e3,
            "tags": "all valid in both arms",
            "what": "ratio: median over alternated K-call graph replays, 95% bootstrap interval of the median; "
                    "p50/p95: one-call graphs, 60 replays each arm"}
        del g_on, g_off, g1_on, g1_off
        g_unf = capture(lambda j: step_unfused(fp8, j), K)
        g_unf.replay()
        ms_unf = time_graph(g_unf) / K
        extra["unfused_step"] = {"us_per_step": ms_unf * 1e3, "fused_us_per_step": ms_per_step * 1e3,
                                 "what": "kv_append_quantize + paged_decode_attention as two calls"}
        bf = caches["bf16"]
        g_bf = capture(lambda j: step(bf, j, do_append=False), K)
        g_bf.replay()
        ms_bf = time_graph(g_bf) / K
        bf_bytes = statistics.mean(decode_alg_bytes(lens0 + j % T + 1, Hkv, D, S, Hq, D, fp8=False) for j in range(K))
        extra["bf16_cache"] = {"us_per_decode": ms_bf * 1e3, "kv_gbs": bf_bytes / (ms_bf * 1e-3) / 1e9,
                               "hbm_frac": bf_bytes / (ms_bf * 1e-3) / 1e9 / peak,
                               "fp8_speedup_per_call": ms_bf / ms_dec}

    # ---- the other benchmark shapes (grouped-query batch, long contexts)
    if not args.no_variants:
        extra["configs"] = bench_configs(abi, dev, i32, bf16, capture, time_graph, peak, max(3, K // 5))

    # ---- latent-shared stream (64 heads over one 576-wide FP8 stream, batch 64)
    latent_w = None
    if not args.no_latent:
        del caches
        torch.cuda.empty_cache()
        latent_w = synth.latent()
        extra["latent"] = bench_latent(abi, latent_w, dev, i32, bf16, capture, time_graph, peak, max(3, K // 5))

    # ---- end to end: per-step inputs from pinned host memory, results back to host.
    # A step's inputs sit in one pinned row (q | k | v | lengths) and go over in
    # one copy; its results (out | status) come back in one copy.  The copies
    # run on a second stream, double-buffered, so that step j + 1's inputs go
    # over while step j runs and step j's results come back while step j + 1
    # runs (a serving loop's pipeline); every step's copies stay inside the
    # timed graph.
    def as_bytes(a):
        return np.ascontiguousarray(a).reshape(T, -1).view(np.uint8)

    parts = [as_bytes(w.q_steps), as_bytes(w.k_steps), as_bytes(w.v_steps),
             as_bytes(np.stack([lens0 + j + 1 for j in range(T)]).astype(np.int32))]
    offs = np.cumsum([0] + [p.shape[1] for p in parts])
    h_in = torch.from_numpy(np.concatenate(parts, axis=1)).pin_memory()
    n_out = B * Hq * D * 4
    d_in = [torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev) for _ in range(2)]
    d_res = [torch.empty(n_out + B * 4, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_res = [torch.empty(n_out + B * 4, dtype=torch.uint8).pin_memory() for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_call(j):
        di, dr = d_in[j % 2], d_res[j % 2]
        d_q = di[offs[0]:offs[1]].view(torch.bfloat16).view(B, Hq, D)
        d_k = di[offs[1]:offs[2]].view(torch.bfloat16).view(B, Hkv, D)
        d_v = di[offs[2]:offs[3]].view(torch.bfloat16).view(B, Hkv, D)
        d_len = di[offs[3]:offs[4]].view(torch.int32)
        out_e, st_e = dr[:n_out].view(torch.float32).view(B, Hq, D), dr[n_out:].view(torch.int32)
        abi.paged_decode_step(fp8, d_k, d_v, d_q, d_len, table, tags, w.softmax_scale, flags=FLAGS,
                              max_splits=max_splits, workspace=ws, out=out_e, status=st_e)

    def capture_e2e(n):
        g = torch.cuda.CUDAGraph()
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_cmp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            cap = torch.cuda.current_stream()
            copy_stream.wait_stream(cap)
            with torch.cuda.stream(copy_stream):
                d_in[0].copy_(h_in[0], non_blocking=True)
                ev_in[0].record(copy_stream)
            for j in range(n):
                cap.wait_event(ev_in[j])
                if j >= 2:
                    cap.wait_event(ev_out[j - 2])  # d_res[j % 2] has been read back
                e2e_call(j)
                ev_cmp[j].record(cap)
                with torch.cuda.stream(copy_stream):
                    if j + 1 < n:
                        if j >= 1:
                            copy_stream.wait_event(ev_cmp[j - 1])  # d_in[(j + 1) % 2] is free
                        d_in[(j + 1) % 2].copy_(h_in[(j + 1) % T], non_blocking=True)
                        ev_in[j + 1].record(copy_stream)
                    copy_stream.wait_event(ev_cmp[j])
                    h_res[j % 2].copy_(d_res[j % 2], non_blocking=True)
                    ev_out[j].record(copy_stream)
            cap.wait_stream(copy_stream)
        return g

    g_e2e = capture_e2e(K)
    # the replayed graph must move the bytes: poison the device inputs and the
    # host results, replay, and check that the last step's copies happened
    for t_ in d_in:
        t_.fill_(0xFF)
    for t_ in h_res:
        t_.zero_()
    torch.cuda.synchronize()
    g_e2e.replay()
    torch.cuda.synchronize()
    last = (K - 1) % 2
    assert torch.equal(d_in[last].cpu(), h_in[(K - 1) % T]), "end-to-end graph did not copy the step inputs"
    assert torch.equal(h_res[last], d_res[last].cpu()), "end-to-end graph did not copy the step results back"
    assert h_res[last].any(), "end-to-end graph left the host result empty"
    ms_e2e = time_graph(g_e2e)
    e2e_val = job_throughput(sum(step_bytes), world, ms_e2e) / 1e9
    h2d = int(offs[-1])
    d2h = n_out + B * 4

    # ---- the CPU oracle on the host cores (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        stepc, threads, desc, nb = oracle_step_sample(w, args.cpu_frac)
        t0 = time.perf_counter()
        tot, n_cpu = 0, 0
        while n_cpu == 0 or time.perf_counter() - t0 < args.cpu_seconds:
            tot += stepc()
            n_cpu += 1
        dt = time.perf_counter() - t0
        cpu = {"value": tot / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{n_cpu} consecutive steps over {desc}", "seconds": dt}
        # the same sample on one thread (at least a few seconds, whole steps)
        stepc1, _, _, _ = oracle_step_sample(w, args.cpu_frac, threads=1)
        t0 = time.perf_counter()
        tot1, n1 = 0, 0
        while n1 == 0 or time.perf_counter() - t0 < args.cpu_seconds / 2:
            tot1 += stepc1()
            n1 += 1
        dt1 = time.perf_counter() - t0
        cpu["single_thread"] = {"value": tot1 / dt1 / 1e9, "unit": "GB/s", "cores": 1, "steps": n1, "seconds": dt1}
        if not args.no_variants:
            cpu["configs"] = oracle_config_timings(latent_w)

    st_final = st_dec.cpu().numpy()
    launches_per_step = 2  # split (page loader also appends the new tokens), merge kernels
    mean_lens = lens0 + (K - 1) % T + 1
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 cache, f16/bf16 MMA, fp32 accumulate", "data": "synthetic",
        "config": {"workload": WORKLOAD if B == 64 else WORKLOAD.replace("batch 64", "first %d requests of batch 64" % B),
                   "seed": w.seed, "batch": B, "context_tokens": int(lens0.sum()),
                   "steps_in_cycle": T, "l2": "inputs larger than L2 (FP8 cache ~0.8 GB per step)",
                   "timing": "CUDA graph of K steps, CUDA events on the launching stream"},
        "decode_tokens_per_s": world * B / (ms_per_step * 1e-3),
        "kv_tokens_per_s": world * float(mean_lens.sum()) / (ms_per_step * 1e-3),
        "hbm_frac_step": value / world / peak,
        "aborted_requests": int((st_final != 0).sum()),
        "roofline": {"bound": "hbm", "kernel": "paged_decode_attention_fp8 (split + merge kernels)",
                     "achieved": dec_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": dec_gbs / peak, "us_per_launch": ms_dec * 1e3,
                     "alg_bytes_per_launch": statistics.mean(dec_bytes), "traffic": recorded_traffic(),
                     "traffic_kernel": "gqa_split_kernel alone (ncu dram read + write per launch)"},
        "per_call": per_call,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e / K},
        "gpu_launches": K * launches_per_step,
        "device_mem_peak_bytes": int(torch.cuda.max_memory_allocated(dev)),
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    res.update(extra)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
