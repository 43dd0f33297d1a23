"""GPU append/quantize parity: pool bytes, scales and status bit-exact
against the oracle; untouched bytes keep the 0xA5 sentinel."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, dev_bf16, dev_i32
from oracle_helpers import oracle_cache
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu


def _small(seed, **kw):
    rng = np.random.default_rng(seed)
    B = kw.pop("B", 4)
    lens = rng.integers(1, kw.pop("max_len", 90) + 1, size=B)
    G, Hkv = kw.pop("G", 4), kw.pop("Hkv", 2)
    return synth.make(f"app{seed}", seed, batch=B, q_heads=G * Hkv, kv_heads=Hkv, seq_lens=lens, outlier_p=0.01, **kw)


def _compare_pools(run, ref):
    c = run.cache
    assert np.array_equal(c.k_pool.view(torch.uint8).cpu().numpy(), ref.k_pool.view(np.uint8))
    if ref.v_pool is not None:
        assert np.array_equal(c.v_pool.view(torch.uint8).cpu().numpy(), ref.v_pool.view(np.uint8))
    if c.k_scale is not None:
        ks = c.k_scale.cpu().numpy()
        if ref.scale_mode == oracle.SCALE_PER_TOKEN:
            written = ref.k_scale != 0  # rows the append wrote
            assert np.array_equal(ks[written].view(np.uint32), ref.k_scale[written].view(np.uint32))
        else:
            assert np.array_equal(ks.view(np.uint32), ref.k_scale.view(np.uint32))
        if ref.v_scale is not None:
            vs = c.v_scale.cpu().numpy()
            if ref.scale_mode == oracle.SCALE_PER_TOKEN:
                written = ref.v_scale != 0
                assert np.array_equal(vs[written].view(np.uint32), ref.v_scale[written].view(np.uint32))
            else:
                assert np.array_equal(vs.view(np.uint32), ref.v_scale.view(np.uint32))


CASES = [
    dict(head_dim=128, page_size=16),
    dict(head_dim=64, page_size=16, G=4, Hkv=1),
    dict(head_dim=128, page_size=64, G=8, Hkv=1, scale_mode=synth.PER_TOKEN),
    dict(head_dim=576, v_head_dim=512, kv_shared=True, page_size=64, G=64, Hkv=1, scale_mode=synth.PER_TOKEN),
]


@pytest.mark.parametrize("dtype", [abi.DTYPE_FP8_E4M3, abi.DTYPE_BF16])
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_bulk_fill_matches_oracle(dtype, ci):
    kw = dict(CASES[ci])
    if dtype == abi.DTYPE_BF16 and kw.get("scale_mode") == synth.PER_TOKEN:
        kw["scale_mode"] = synth.PER_HEAD
    w = _small(200 + ci, **kw)
    run = DeviceCase(w, dtype)
    ref, st = oracle_cache(w, dtype)
    assert not run.fill_status.cpu().numpy().any() and not st.any()
    _compare_pools(run, ref)


def test_tiny_fill_and_decode_step_append():
    w = synth.tiny()
    run = DeviceCase(w)
    ref, _ = oracle_cache(w)
    _compare_pools(run, ref)
    # one decode-step append per request at position L (row_req NULL path), tag check on
    rng = np.random.default_rng(1)
    k_new = synth.bf16_bits(rng.standard_normal((2, 1, 64)).astype(np.float32) * 3)
    v_new = synth.bf16_bits(rng.standard_normal((2, 1, 64)).astype(np.float32) * 3)
    st_gpu = abi.kv_append_quantize(run.cache, dev_bf16(k_new), dev_bf16(v_new), dev_i32(w.seq_lens), run.table,
                                    run.tags, flags=abi.FLAG_TAG_CHECK)
    st_ref = ref.append(k_new, v_new, w.seq_lens, w.block_table, w.block_tags, flags=oracle.FLAG_TAG_CHECK)
    assert np.array_equal(st_gpu.cpu().numpy().view(np.uint32), st_ref)
    _compare_pools(run, ref)


def test_refused_rows_write_nothing():
    w = synth.make("ref", 21, batch=5, q_heads=8, kv_heads=2, head_dim=128, page_size=16, seq_lens=[3, 3, 3, 3, 3],
                   room_tokens=16)
    run = DeviceCase(w, fill=False)
    run.cache.k_scale.fill_(0.01)
    run.cache.v_scale.fill_(0.02)
    ref = oracle.Cache(w.num_pages, 16, 2, 128, 128, False, oracle.DTYPE_FP8, oracle.SCALE_PER_HEAD, w.page_tags,
                       k_scale=np.full(2, 0.01, np.float32), v_scale=np.full(2, 0.02, np.float32))
    rng = np.random.default_rng(2)
    k_new = synth.bf16_bits(rng.standard_normal((5, 2, 128)).astype(np.float32))
    v_new = synth.bf16_bits(rng.standard_normal((5, 2, 128)).astype(np.float32))
    bt, tags, pos = w.block_table.copy(), w.block_tags.copy(), w.seq_lens.copy()
    tags[0, 0] ^= 5           # stale destination
    bt[1, 0] = w.num_pages    # outside the pool
    pos[2] = -3               # before the context
    pos[3] = w.max_pages * 16  # past the table
    st = abi.kv_append_quantize(run.cache, dev_bf16(k_new), dev_bf16(v_new), dev_i32(pos), dev_i32(bt), dev_i32(tags),
                                flags=abi.FLAG_TAG_CHECK)
    st_ref = ref.append(k_new, v_new, pos, bt, tags, flags=oracle.FLAG_TAG_CHECK)
    assert list(st_ref) == [1, 2, 4, 4, 0]
    assert np.array_equal(st.cpu().numpy().view(np.uint32), st_ref)
    _compare_pools(run, ref)


def test_calibration_matches_oracle():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5000, 8, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    x[:, 5, :] = 0.0
    bits = synth.bf16_bits(x)
    s = abi.calibrate_scales(dev_bf16(bits)).cpu().numpy()
    assert np.array_equal(s.view(np.uint32), oracle.calibrate_per_head(bits).view(np.uint32))
