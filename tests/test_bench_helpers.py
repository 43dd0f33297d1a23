"""The benchmark's host-side arithmetic (no GPU): the algorithmic byte count
the roofline divides by, the per-call percentiles, the bootstrap interval of
the tag-check ratio, the whole-job throughput and the recorded DRAM traffic."""
import json
import math
import os
import statistics
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_fp8_kv_quantize_gb300 import synth  # noqa: E402


def test_decode_alg_bytes_by_hand():
    # two requests of 1 and 17 tokens, 2 KV heads of 8 values, pages of 16,
    # 4 query heads, value width 8: KV rows (FP8: one byte per value, K and
    # V), 12 bytes per page (table entry, expected tag, page tag), the bf16
    # query rows and the fp32 output rows
    kv = (1 + 17) * 2 * 2 * 8
    table = (1 + 2) * 12
    q = 2 * 4 * 8 * 2
    out = 2 * 4 * 8 * 4
    assert bench.decode_alg_bytes([1, 17], 2, 8, 16, 4, 8) == kv + table + q + out
    # BF16 doubles the rows; no tag check drops the page tag word
    assert bench.decode_alg_bytes([1, 17], 2, 8, 16, 4, 8, fp8=False, tag_check=False) == \
        2 * kv + (1 + 2) * 8 + q + out


def test_decode_alg_bytes_of_the_bench_workload():
    # the figure the docs quote for the ragged batch of 64: the mean over the
    # bench's 100-step cycle (every request one token longer per step)
    w = synth.ragged()
    lens = w.seq_lens.astype(np.int64)
    b = [bench.decode_alg_bytes(lens + j + 1, w.kv_heads, w.head_dim, w.page_size, w.q_heads, w.head_dim)
         for j in range(w.steps)]
    assert 648.9e6 < b[0] < 649.0e6
    assert abs(statistics.mean(b) - 655.452e6) < 0.01e6


def test_percentile_matches_linear_interpolation():
    rng = np.random.default_rng(3)
    for n in (1, 2, 7, 60):
        xs = list(rng.normal(size=n))
        for q in (0, 50, 95, 100):
            assert math.isclose(bench.percentile(xs, q), float(np.percentile(xs, q)), rel_tol=1e-12, abs_tol=1e-12)
    assert bench.percentile([], 50) is None


def test_bootstrap_interval_brackets_the_median():
    rng = np.random.default_rng(4)
    xs = list(1.003 + 0.001 * rng.standard_normal(21))
    lo, hi = bench.bootstrap_ci(xs)
    assert lo <= statistics.median(xs) <= hi
    assert bench.bootstrap_ci(xs) == [lo, hi]  # seeded: the same interval every time
    assert bench.bootstrap_ci([2.0] * 5) == [2.0, 2.0]


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(100.0, 1, 2.0) == 100.0 / 2e-3
    assert bench.job_throughput(100.0, 4, 2.0) == 4 * 100.0 / 2e-3


def test_recorded_traffic_follows_the_hashed_sources():
    path = os.path.join(ROOT, "profiles", "gqa_split_fp8_ragged_b64.traffic.json")
    with open(path) as f:
        rec = json.load(f)
    got = bench.recorded_traffic()
    # the counters are reported while the hashed kernel sources are unchanged,
    # and withheld (None) once any of them differs
    assert got is None or got == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert rec["sources"] and all(os.path.exists(os.path.join(ROOT, p)) for p in rec["sources"])
