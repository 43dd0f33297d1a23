"""GPU BF16 -> FP8 page hand-off against the oracle: codes, per-token scales
and page status bit-exact; pages that are not targets keep the sentinel."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, dev_i32
from oracle_helpers import oracle_cache
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["gqa", "latent", "narrow"])
def test_handoff_matches_oracle(case):
    if case == "narrow":  # head_dim 40: five 16-byte chunks per row, per-token scales
        w = synth.make("ho_narrow", 602, batch=2, q_heads=4, kv_heads=2, head_dim=40, page_size=16,
                       seq_lens=[33, 70], scale_mode=synth.PER_TOKEN)
    elif case == "latent":
        w = synth.make("ho_lat", 601, batch=3, q_heads=64, kv_heads=1, head_dim=576, v_head_dim=512, kv_shared=True,
                       page_size=64, seq_lens=[100, 64, 300], scale_mode=synth.PER_TOKEN)
    else:
        w = synth.make("ho", 600, batch=4, q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                       seq_lens=[40, 300, 17, 1000])
    src = DeviceCase(w, abi.DTYPE_BF16)
    ref_src, _ = oracle_cache(w, oracle.DTYPE_BF16)
    used = np.unique(w.block_table[w.block_table >= 0])
    rng = np.random.default_rng(5)
    P2 = used.size + 7
    dst_ids = rng.permutation(P2)[: used.size]
    src_ids = np.concatenate([used, [w.num_pages + 2]])  # one out-of-range pair
    dst_ids = np.concatenate([dst_ids, [0]])
    mode = w.scale_mode
    dst = abi.PagedCache(P2, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, abi.DTYPE_FP8_E4M3, mode,
                         fill=0xA5)
    ks = vs = None
    if mode == synth.PER_HEAD:
        ks, vs = oracle.calibrate_per_head(w.k_rows), oracle.calibrate_per_head(w.v_rows)
        dst.k_scale.copy_(torch.from_numpy(ks))
        dst.v_scale.copy_(torch.from_numpy(vs))
    st = abi.handoff_bf16_to_fp8(src.cache, dst, dev_i32(src_ids), dev_i32(dst_ids))
    torch.cuda.synchronize()
    ref = oracle.Cache(P2, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared, oracle.DTYPE_FP8, mode,
                       k_scale=ks, v_scale=vs)
    st_ref = ref.handoff_from(ref_src, src_ids, dst_ids)
    assert np.array_equal(st.cpu().numpy().view(np.uint32), st_ref)
    assert st_ref[-1] == oracle.ST_PAGE_OOB
    assert np.array_equal(dst.k_pool.cpu().numpy(), ref.k_pool)
    if not w.kv_shared:
        assert np.array_equal(dst.v_pool.cpu().numpy(), ref.v_pool)
    if mode == synth.PER_TOKEN:
        written = ref.k_scale != 0
        assert np.array_equal(dst.k_scale.cpu().numpy()[written].view(np.uint32), ref.k_scale[written].view(np.uint32))
