"""GPU decode step (append every request's new token, then attend, in one
call) against the oracle doing the same two things in order: oracle append
of the new rows, then oracle decode.  Output within tolerance, status and
every pool byte (and per-token scale) bit-exact, including requests whose
new row is refused (stale or out-of-range destination page)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, assert_close, dev_bf16, dev_i32
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu
FP8, BF16 = abi.DTYPE_FP8_E4M3, abi.DTYPE_BF16


def _split(w):
    """History rows (every position but the last) and the new rows, one per request in request order."""
    last = w.row_pos == (w.seq_lens[w.row_req] - 1)
    order = np.argsort(w.row_req[last], kind="stable")
    assert np.array_equal(w.row_req[last][order], np.arange(w.batch))
    k_new = w.k_rows[last][order]
    v_new = None if w.kv_shared else w.v_rows[last][order]
    return ~last, k_new, v_new


def _run(w, dtype, flags, max_splits=None):
    hist, k_new, v_new = _split(w)
    mode = w.scale_mode if dtype == FP8 else synth.PER_HEAD
    # GPU: calibrate on all rows, append history, then the one-call step
    run = DeviceCase(w, dtype, fill=False)
    if dtype == FP8 and mode == synth.PER_HEAD:
        abi.calibrate_scales(dev_bf16(w.k_rows), run.cache.k_scale)
        abi.calibrate_scales(dev_bf16(w.v_rows), run.cache.v_scale)
    if hist.any():
        abi.kv_append_quantize(run.cache, dev_bf16(w.k_rows[hist]),
                               None if w.kv_shared else dev_bf16(w.v_rows[hist]), dev_i32(w.row_pos[hist]),
                               run.table, run.tags, row_req=dev_i32(w.row_req[hist]), batch=w.batch)
    out, st = abi.paged_decode_step(run.cache, dev_bf16(k_new), None if v_new is None else dev_bf16(v_new), run.q,
                                    run.seq_lens, run.table, run.tags, w.softmax_scale, flags=flags,
                                    max_splits=w.max_splits if max_splits is None else max_splits)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    st = st.cpu().numpy().view(np.uint32)
    # oracle: the same two steps in order
    ks = vs = None
    if dtype == FP8 and mode == synth.PER_HEAD:
        ks, vs = oracle.calibrate_per_head(w.k_rows), oracle.calibrate_per_head(w.v_rows)
    ref = oracle.Cache(w.num_pages, w.page_size, w.kv_heads, w.head_dim, w.v_head_dim, w.kv_shared,
                       oracle.DTYPE_FP8 if dtype == FP8 else oracle.DTYPE_BF16, mode, w.page_tags, ks, vs)
    ref.append(w.k_rows[hist], None if w.kv_shared else w.v_rows[hist], w.row_pos[hist], w.block_table, w.block_tags,
               row_req=w.row_req[hist], batch=w.batch)
    st_app = ref.append(k_new, v_new, w.seq_lens - 1, w.block_table, w.block_tags, flags=flags,
                        row_req=np.arange(w.batch, dtype=np.int32), batch=w.batch)
    o_ref, st_ref = ref.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, flags=flags, threads=8)
    assert np.all((st_app & ~st_ref) == 0), "an append refusal the attention does not report"
    assert np.array_equal(st, st_ref), (st, st_ref)
    assert_close(out, o_ref, f"{w.name} step")
    assert not out[st != 0].any()
    # every byte of the pools, sentinel included
    c = run.cache
    if dtype == FP8:
        assert np.array_equal(c.k_pool.cpu().numpy().reshape(-1), ref.k_pool)
        if not w.kv_shared:
            assert np.array_equal(c.v_pool.cpu().numpy().reshape(-1), ref.v_pool)
    else:
        assert np.array_equal(c.k_pool.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16), ref.k_pool)
        assert np.array_equal(c.v_pool.view(torch.int16).cpu().numpy().reshape(-1).view(np.uint16), ref.v_pool)
    if dtype == FP8 and mode == synth.PER_TOKEN:
        written = ref.k_scale != 0
        assert np.array_equal(c.k_scale.cpu().numpy().reshape(-1)[written].view(np.uint32),
                              ref.k_scale[written].view(np.uint32))
    return st


LENS = [1, 16, 17, 300, 2049, 40, 5000, 33]


@pytest.mark.parametrize("flags", [0, abi.FLAG_TAG_CHECK])
@pytest.mark.parametrize("dtype", [FP8, BF16])
def test_step_gqa(dtype, flags):
    # request 2's last page (the new row's destination) and an earlier page of request 4 are stale
    w = synth.make("step_gqa", 900, batch=len(LENS), q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                   seq_lens=LENS, stale_block_entries=[(2, 1), (4, 0)], outlier_p=0.01)
    st = _run(w, dtype, flags)
    if flags:
        assert st[2] == abi.ST_STALE_TAG and st[4] == abi.ST_STALE_TAG


@pytest.mark.parametrize("max_splits", [1, 2])
@pytest.mark.parametrize("dtype", [FP8, BF16])
def test_step_gqa_chunk_rule(dtype, max_splits):
    # max_splits < 3: requests cut into chunks, a range taking the chunks that
    # start in it; the new rows are still written by the piece that holds
    # each last page
    w = synth.make("step_lpt", 903, batch=len(LENS), q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                   seq_lens=LENS, stale_block_entries=[(2, 1)], outlier_p=0.01)
    st = _run(w, dtype, abi.FLAG_TAG_CHECK, max_splits=max_splits)
    assert st[2] == abi.ST_STALE_TAG


@pytest.mark.parametrize("dtype", [FP8, BF16])
@pytest.mark.parametrize("shape", [(8, 1, 128, 64), (4, 2, 64, 16), (2, 4, 64, 32), (3, 2, 128, 16),
                                   (16, 2, 64, 16)])
def test_step_other_shapes(dtype, shape):
    # group sizes 8 and 2, head width 64, pages of 64 and 32 tokens: the new
    # rows are written by the item holding each request's last page
    G, Hkv, D, S = shape
    lens = [1, S, S + 1, 3 * S - 1, 2000, 5000]
    w = synth.make("step_shapes", 904 + G, batch=len(lens), q_heads=G * Hkv, kv_heads=Hkv, head_dim=D,
                   page_size=S, seq_lens=lens, stale_block_entries=[(4, 1)], outlier_p=0.01)
    st = _run(w, dtype, abi.FLAG_TAG_CHECK)
    assert st[4] == abi.ST_STALE_TAG


def test_step_per_token_scales_and_oob_destination():
    w = synth.make("step_tok", 901, batch=6, q_heads=16, kv_heads=2, head_dim=64, page_size=16,
                   seq_lens=[1, 65, 200, 1000, 16, 3000], scale_mode=synth.PER_TOKEN)
    w.block_table = w.block_table.copy()
    w.block_table[1, 4] = w.num_pages + 3  # request 1's new row (position 64) has no page
    st = _run(w, FP8, abi.FLAG_TAG_CHECK)
    assert st[1] == abi.ST_PAGE_OOB


def test_step_latent_stream():
    w = synth.make("step_lat", 902, batch=5, q_heads=64, kv_heads=1, head_dim=576, v_head_dim=512, kv_shared=True,
                   page_size=64, seq_lens=[1, 64, 65, 900, 4000], scale_mode=synth.PER_TOKEN,
                   stale_block_entries=[(3, 14)], softmax_scale=1.0 / 24.0)
    st = _run(w, FP8, abi.FLAG_TAG_CHECK)
    assert st[3] == abi.ST_STALE_TAG
