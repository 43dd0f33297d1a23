"""Latent-shared stream (64 heads over one 576-wide FP8 stream, V = first
512 values, per-token scales, 64-token pages) against the fp64 oracle."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import DeviceCase, assert_close, dev_i32
from oracle_helpers import oracle_cache, oracle_cache_subset
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu
TAU = 1.0 / math.sqrt(576.0)


def _lat(seed, lens, **kw):
    return synth.make(f"lat{seed}", seed, batch=len(lens), q_heads=64, kv_heads=1, head_dim=576, v_head_dim=512,
                      kv_shared=True, page_size=64, seq_lens=lens, scale_mode=synth.PER_TOKEN, softmax_scale=TAU,
                      **kw)


def _check(w, flags=0, max_splits=None, tables=None):
    run = DeviceCase(w)
    ref, _ = oracle_cache(w)
    bt, tags, lens = tables if tables else (w.block_table, w.block_tags, w.seq_lens)
    out, st = run.decode(flags=flags, max_splits=max_splits, table=dev_i32(bt), tags=dev_i32(tags),
                         seq_lens=dev_i32(lens))
    o_ref, st_ref = ref.decode(w.q, lens, bt, tags, w.softmax_scale, flags=flags, threads=16)
    assert np.array_equal(st, st_ref), (st, st_ref)
    assert not out[st != 0].any()
    assert_close(out, o_ref, w.name)
    return out, st


def test_latent_small_ragged():
    _check(_lat(500, [1, 63, 64, 65, 127, 129, 300, 1000]))


@pytest.mark.parametrize("max_splits", [1, 2, 3, 5, 64])
def test_latent_splits(max_splits):
    _check(_lat(501, [5000, 2100, 77]), max_splits=max_splits)


def test_latent_tags_oob_and_bad_length():
    w = _lat(502, [200, 200, 200, 200], room_tokens=64)
    bt, tags, lens = w.block_table.copy(), w.block_tags.copy(), w.seq_lens.copy()
    tags[1, 2] ^= 1                 # stale, inspected
    tags[0, 4] ^= 1                 # stale, past ceil(200/64) = 4: not inspected
    bt[2, 0] = w.num_pages          # outside the pool
    lens[3] = w.max_pages * 64 + 1  # past the table
    out, st = _check(w, flags=abi.FLAG_TAG_CHECK, tables=(bt, tags, lens))
    assert list(st) == [0, abi.ST_STALE_TAG, abi.ST_PAGE_OOB, abi.ST_BAD_LEN]


def test_latent_full_size_sampled():
    w = synth.latent()
    run = DeviceCase(w)
    out, st = run.decode(flags=abi.FLAG_TAG_CHECK)
    assert not st.any()
    order = np.argsort(w.seq_lens, kind="stable")
    idx = np.unique(np.array([order[0], order[-1]]))
    c, ctab, ctags, used = oracle_cache_subset(w, idx)
    k_gpu = run.cache.k_rows()[np.asarray(used)].cpu().numpy().reshape(-1)
    assert np.array_equal(k_gpu, c.k_pool)
    ks_gpu = run.cache.k_scale.view(w.num_pages, 1, 64)[np.asarray(used)].cpu().numpy().reshape(-1)
    written = c.k_scale != 0  # slots past a request's last token were never written on either side
    assert written.sum() == w.seq_lens[idx].sum()
    assert np.array_equal(ks_gpu[written].view(np.uint32), c.k_scale[written].view(np.uint32))
    o_ref, _ = c.decode(w.q[idx], w.seq_lens[idx], ctab, ctags, w.softmax_scale, flags=oracle.FLAG_TAG_CHECK,
                        threads=16)
    assert_close(out[idx], o_ref, "latent full size")
