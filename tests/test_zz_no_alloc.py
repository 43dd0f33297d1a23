"""The no-allocation FP8 decode entry point against the regular one.

pfkv_paged_decode_attention_fp8_noalloc exists for callers that cannot hand
the library device scratch (a host framework that owns every allocation,
a plugin that must not bypass its host's allocator, a serving path where a
cudaMalloc would synchronise the device).  It must give what the regular
entry point gives, and what the oracle gives, call after call, while the
library's fixed scratch buffer keeps the previous call's contents.  This
file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ABS_TOL, DeviceCase, assert_close
from oracle_helpers import oracle_cache
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu


def _noalloc_call(run, out, status, flags, max_splits):
    """Call the entry point straight through the C ABI."""
    w = run.w
    d = run.cache.desc()
    return abi.lib.pfkv_paged_decode_attention_fp8_noalloc(
        ctypes.byref(d), ctypes.c_void_p(run.q.data_ptr()), w.q_heads, ctypes.c_void_p(run.seq_lens.data_ptr()),
        ctypes.c_void_p(run.table.data_ptr()), ctypes.c_void_p(run.tags.data_ptr()), w.batch, w.max_pages,
        float(w.softmax_scale), flags, max_splits, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _case(seed, n, lo, hi, stale):
    rng = np.random.default_rng(seed)
    lens = list(rng.integers(lo, hi, size=n)) + [1, 16, 17]
    return synth.make(f"noalloc{seed}", seed, batch=len(lens), q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                      seq_lens=lens, outlier_p=0.01, stale_block_entries=[stale])


def _noalloc_checked(run, max_splits, ref, st_ref, o_oracle, what):
    w = run.w
    out = torch.empty(w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device="cuda")
    status = torch.empty(w.batch, dtype=torch.int32, device="cuda")
    out.fill_(float("nan"))
    status.fill_(-1)
    rc = _noalloc_call(run, out, status, abi.FLAG_TAG_CHECK, max_splits)
    assert rc == 0, abi.strerror(rc)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    st = status.cpu().numpy().view(np.uint32)
    assert np.array_equal(st, st_ref), f"{what}: status {st} != {st_ref}"
    assert_close(got, ref, f"{what} against the regular entry point")
    assert np.abs(got - ref).max() <= ABS_TOL
    assert_close(got, o_oracle, f"{what} against the oracle")


def test_noalloc_matches_regular_entry_point_and_oracle():
    # The shared buffer keeps the previous call's contents, so each checked
    # call follows a call on a different workload (other batch, lengths,
    # split cap and stale entry), in both orders; every call must match the
    # regular entry point (bit-equal status, output within the tolerance) and
    # the oracle.
    small = DeviceCase(_case(900, 12, 1, 6000, (3, 0)))
    large = DeviceCase(_case(903, 40, 500, 20000, (17, 2)))
    cases = []
    for run, splits in ((small, 16), (large, 32)):
        w = run.w
        assert abi.decode_workspace_bytes(run.cache, w.batch, w.q_heads, splits) <= abi.NOALLOC_SCRATCH_BYTES
        ref, st_ref = run.decode(flags=abi.FLAG_TAG_CHECK, max_splits=splits)
        oc, _ = oracle_cache(w)
        o_oracle, st_oracle = oc.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale,
                                        flags=oracle.FLAG_TAG_CHECK, threads=16)
        assert np.array_equal(st_ref, st_oracle)
        cases.append((run, splits, ref, st_ref, o_oracle))
    assert cases[0][3][3] == abi.ST_STALE_TAG and cases[1][3][17] == abi.ST_STALE_TAG
    for order in ((0, 1, 0), (1, 0, 1)):
        for k, i in enumerate(order):
            run, splits, ref, st_ref, o_oracle = cases[i]
            _noalloc_checked(run, splits, ref, st_ref, o_oracle, f"order {order} call {k}")


def test_noalloc_rejects_requests_beyond_its_buffer():
    w = synth.make("noalloc_big", 901, batch=2, q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                   seq_lens=[100, 200])
    run = DeviceCase(w)
    # 256 splits x 32 heads x 128 dims needs far more than the fixed buffer for a large batch
    big_batch = 4096
    assert abi.decode_workspace_bytes(run.cache, big_batch, 32, 256) > abi.NOALLOC_SCRATCH_BYTES
    d = run.cache.desc()
    rc = abi.lib.pfkv_paged_decode_attention_fp8_noalloc(
        ctypes.byref(d), None, 32, None, None, None, big_batch, 64, 1.0, 0, 256, None, None, None)
    assert rc == -5  # PFKV_ERR_WORKSPACE, returned before any device work
