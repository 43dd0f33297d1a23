"""Pin of the oracle's BF16 -> FP8 page hand-off: every code equals torch's
e4m3 cast of numpy's IEEE fp32 quotient x / s (library routines), with s the
per-head scale or each row's amax / 448."""
import numpy as np
import pytest
import torch

import oracle
from paged_fp8_kv_quantize_gb300 import synth


def _bf16_cache(P, S, H, D, rng):
    c = oracle.Cache(P, S, H, D, D, False, oracle.DTYPE_BF16)
    c.k_pool[:] = synth.bf16_bits(rng.standard_normal(c.k_pool.size).astype(np.float32) * 2)
    c.v_pool[:] = synth.bf16_bits(rng.standard_normal(c.v_pool.size).astype(np.float32))
    return c


def _e4m3(y):
    return torch.from_numpy(np.ascontiguousarray(y, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("mode", [oracle.SCALE_PER_HEAD, oracle.SCALE_PER_TOKEN])
def test_handoff_codes_are_fp32_division_then_e4m3(mode):
    rng = np.random.default_rng(31)
    P, S, H, D = 6, 16, 2, 64
    src = _bf16_cache(P, S, H, D, rng)
    fk = synth.bf16_to_f32(src.k_pool).reshape(P, H, S, D)
    fv = synth.bf16_to_f32(src.v_pool).reshape(P, H, S, D)
    ks = (np.abs(fk).max(axis=(0, 2, 3)) / np.float32(448)).astype(np.float32)
    vs = (np.abs(fv).max(axis=(0, 2, 3)) / np.float32(448)).astype(np.float32)
    dst = oracle.Cache(5, S, H, D, D, False, oracle.DTYPE_FP8, mode, k_scale=ks, v_scale=vs)
    src_pages, dst_pages = np.array([4, 0, 2, 9]), np.array([1, 3, 0, 2])  # the last source id is out of range
    st = dst.handoff_from(src, src_pages, dst_pages)
    assert list(st) == [0, 0, 0, oracle.ST_PAGE_OOB]
    K, V = dst.k_rows(), dst.v_rows()
    for s_id, d_id in zip(src_pages[:3], dst_pages[:3]):
        for f, out, hs, sc in ((fk, K, ks, dst.k_scale), (fv, V, vs, dst.v_scale)):
            x = f[s_id]  # [H][S][D]
            if mode == oracle.SCALE_PER_HEAD:
                s = hs.reshape(H, 1, 1)
            else:
                s = (np.abs(x).max(axis=2, keepdims=True) / np.float32(448)).astype(np.float32)
                assert np.array_equal(sc.reshape(5, H, S)[d_id].view(np.uint32), s[..., 0].view(np.uint32))
            assert np.array_equal(out[d_id], _e4m3(x / s))
    assert np.all(K[4] == 0xA5)  # page 4 of dst was not a target
