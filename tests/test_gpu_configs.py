"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (default split cap, tag check on, one workspace per call).

Outputs are compared with the fp64 oracle on sampled requests (the oracle
builds a compact cache for those requests from the same BF16 rows); pool
bytes of the sampled pages and the status of every request are compared
bit-exactly."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, assert_close, dev_bf16, dev_i32
from oracle_helpers import oracle_cache_subset
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu
FLAGS = abi.FLAG_TAG_CHECK


def _pool_pages(run, used, which="k"):
    rows = run.cache.k_rows() if which == "k" else run.cache.v_rows()
    return rows[torch.as_tensor(used, device="cuda", dtype=torch.long)].view(torch.uint8).cpu().numpy()


def _sample(w, n_short=2, n_long=2):
    order = np.argsort(w.seq_lens, kind="stable")
    return np.unique(np.concatenate([order[:n_short], order[-n_long:]]))


@pytest.mark.parametrize("dtype", [abi.DTYPE_FP8_E4M3, abi.DTYPE_BF16])
def test_gqa_batch32_full_size(dtype):
    w = synth.gqa()
    run = DeviceCase(w, dtype)
    out, st = run.decode(flags=FLAGS)
    assert not st.any()
    idx = _sample(w)
    c, ctab, ctags, used = oracle_cache_subset(w, idx, dtype)
    assert np.array_equal(_pool_pages(run, used, "k").reshape(-1), c.k_pool.view(np.uint8))
    assert np.array_equal(_pool_pages(run, used, "v").reshape(-1), c.v_pool.view(np.uint8))
    o_ref, st_ref = c.decode(w.q[idx], w.seq_lens[idx], ctab, ctags, w.softmax_scale, flags=FLAGS, threads=16)
    assert not st_ref.any()
    assert_close(out[idx], o_ref, f"gqa dtype={dtype}")


def test_long_context_full_size_scattered_pool():
    # 8 x 131072 tokens, pages scattered over a pool 8x larger than needed
    w = synth.long_ctx(num_pages=8 * 8 * 2048)
    run = DeviceCase(w)
    out, st = run.decode(flags=FLAGS)
    assert not st.any()
    idx = np.array([3])
    c, ctab, ctags, used = oracle_cache_subset(w, idx)
    assert np.array_equal(_pool_pages(run, used, "k").reshape(-1), c.k_pool.view(np.uint8))
    o_ref, _ = c.decode(w.q[idx], w.seq_lens[idx], ctab, ctags, w.softmax_scale, flags=FLAGS, threads=16)
    assert_close(out[idx], o_ref, "long context")


def test_ragged_batch64_100_steps():
    """The benchmark's workload: every step appends one token per request and
    decodes; parity at steps 0, 1, 50 and 99; status of all 64 requests and
    of every append bit-exact."""
    w = synth.ragged()
    run = DeviceCase(w)
    assert not run.fill_status.cpu().numpy().any()
    c, ctab, ctags, used = oracle_cache_subset(w, np.arange(w.batch))
    B = w.batch
    ws = torch.empty(abi.decode_workspace_bytes(run.cache, B, w.q_heads, w.max_splits), dtype=torch.uint8,
                     device="cuda")
    aborted = set()
    for j in range(w.steps):
        pos = w.seq_lens.astype(np.int64) + j
        st_app = abi.kv_append_quantize(run.cache, dev_bf16(w.k_steps[j]), dev_bf16(w.v_steps[j]), dev_i32(pos),
                                        run.table, run.tags, flags=FLAGS)
        st_app_ref = c.append(w.k_steps[j], w.v_steps[j], pos, ctab, ctags, flags=oracle.FLAG_TAG_CHECK)
        assert np.array_equal(st_app.cpu().numpy().view(np.uint32), st_app_ref), f"append status, step {j}"
        if j in (0, 1, 50, 99):
            out, st = abi.paged_decode_attention_fp8(run.cache, dev_bf16(w.q_steps[j]), dev_i32(pos + 1), run.table,
                                                     run.tags, w.softmax_scale, flags=FLAGS,
                                                     max_splits=w.max_splits, workspace=ws)
            torch.cuda.synchronize()
            out = out.cpu().numpy().astype(np.float64)
            st = st.cpu().numpy().view(np.uint32)
            o_ref, st_ref = c.decode(w.q_steps[j], pos + 1, ctab, ctags, w.softmax_scale,
                                     flags=oracle.FLAG_TAG_CHECK, threads=16)
            assert np.array_equal(st, st_ref), f"decode status, step {j}"
            assert not out[st != 0].any()
            assert_close(out, o_ref, f"ragged step {j}")
            aborted |= set(np.nonzero(st)[0].tolist())
    # the 0.1% stale entries abort some requests, and only those
    stale_reqs = {b for b, _ in w.stale}
    assert aborted == stale_reqs
    assert np.array_equal(_pool_pages(run, used, "k").reshape(-1), c.k_pool.view(np.uint8))
    assert np.array_equal(_pool_pages(run, used, "v").reshape(-1), c.v_pool.view(np.uint8))


def test_ragged_batch64_100_fused_steps():
    """The benchmark's timed call: pfkv_paged_decode_step (the new token of
    every request written by the attention kernel, then attention) for 100
    steps; parity at steps 0, 1, 50 and 99, status of every checked step and
    the final pool bytes bit-exact."""
    w = synth.ragged()
    run = DeviceCase(w)
    c, ctab, ctags, used = oracle_cache_subset(w, np.arange(w.batch))
    B = w.batch
    ws = torch.empty(abi.decode_workspace_bytes(run.cache, B, w.q_heads, w.max_splits), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(B, w.q_heads, w.head_dim, dtype=torch.float32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    for j in range(w.steps):
        pos = w.seq_lens.astype(np.int64) + j
        abi.paged_decode_step(run.cache, dev_bf16(w.k_steps[j]), dev_bf16(w.v_steps[j]), dev_bf16(w.q_steps[j]),
                              dev_i32(pos + 1), run.table, run.tags, w.softmax_scale, flags=FLAGS,
                              max_splits=w.max_splits, workspace=ws, out=out, status=st)
        c.append(w.k_steps[j], w.v_steps[j], pos, ctab, ctags, flags=oracle.FLAG_TAG_CHECK)
        if j in (0, 1, 50, 99):
            torch.cuda.synchronize()
            o = out.cpu().numpy().astype(np.float64)
            s = st.cpu().numpy().view(np.uint32)
            o_ref, st_ref = c.decode(w.q_steps[j], pos + 1, ctab, ctags, w.softmax_scale,
                                     flags=oracle.FLAG_TAG_CHECK, threads=16)
            assert np.array_equal(s, st_ref), f"step status, step {j}"
            assert not o[s != 0].any()
            assert_close(o, o_ref, f"fused ragged step {j}")
    torch.cuda.synchronize()
    assert np.array_equal(_pool_pages(run, used, "k").reshape(-1), c.k_pool.view(np.uint8))
    assert np.array_equal(_pool_pages(run, used, "v").reshape(-1), c.v_pool.view(np.uint8))

