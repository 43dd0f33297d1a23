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


def test_latent_peaked_softmax_and_moving_maximum():
    # request 0: large softmax scale (scores spread over hundreds of log2
    # units: a few tokens hold all the mass); request 1: 1% of key values x20;
    # request 2: keys drift towards head 0's query, so that head's running
    # maximum climbs many times (every rescale threshold crossing); request 3:
    # one key far above the rest in the middle of a long context
    lens = [3000, 2500, 4100, 6000]
    w = _lat(503, lens, outlier_p=0.01)
    f = synth.bf16_to_f32(w.k_rows).copy()
    qf = synth.bf16_to_f32(w.q).copy()
    off, end = w.rows_of(2)
    lam = np.linspace(0.0, 1.0, end - off, dtype=np.float32)[:, None, None]
    f[off:end] = 0.5 * f[off:end] + lam * qf[2, 0][None, None, :] / 2.0
    off3 = w.rows_of(3)[0]
    f[off3 + 4321, 0, :] = qf[3, 5] * 1.5
    w.k_rows[:] = synth.bf16_bits(f)
    _check(w)
    w.softmax_scale = 1.0  # every request peaked
    _check(w)


def test_latent_query_spanning_wide_range():
    # query values spread over 2^-16 .. 1 of each row's largest: the two e4m3
    # terms represent the row exactly only within 2^10 of its largest element
    w = _lat(504, [700, 64, 2000])
    rng = np.random.default_rng(504)
    qf = synth.bf16_to_f32(w.q).copy()
    qf *= np.exp2(-rng.integers(0, 17, size=qf.shape)).astype(np.float32)
    qf[:, :, 7] = 3.0  # each row keeps one large element
    w.q[:] = synth.bf16_bits(qf)
    _check(w)


def test_latent_closed_forms():
    # length 1 gives the value row; a constant V (same codes and scale for
    # every token: the rope part stays below the latent part's largest value)
    # gives the constant, whatever the scores; both within the tolerance of
    # the parity tests (the kernel carries the probabilities as three or four
    # 8-bit terms, 11 to 15 significant bits)
    w = _lat(505, [1, 1, 300, 900])
    f = synth.bf16_to_f32(w.k_rows).copy()
    off = w.rows_of(2)[0]
    rng = np.random.default_rng(505)
    const = rng.standard_normal(512).astype(np.float32)
    const[0] = 4.0
    f[off:, 0, :512] = const
    f[off:, 0, 512:] = np.clip(f[off:, 0, 512:], -3.5, 3.5)
    w.k_rows[:] = synth.bf16_bits(f)
    out, st = _check(w)
    ref, _ = oracle_cache(w)
    for b in (0, 1):  # one token: every head returns that token's dequantized value row
        page = w.block_table[b, 0]
        codes = ref.k_pool.reshape(w.num_pages, 64, 576)[page, 0, :512]
        row = oracle.e4m3_decode(codes).astype(np.float64) * float(ref.k_scale.reshape(w.num_pages, 64)[page, 0])
        assert_close(out[b], np.broadcast_to(row, (64, 512)), f"length 1, request {b}")
    page = w.block_table[2, 0]
    codes = ref.k_pool.reshape(w.num_pages, 64, 576)[page, 0, :512]
    row = oracle.e4m3_decode(codes).astype(np.float64) * float(ref.k_scale.reshape(w.num_pages, 64)[page, 0])
    for b in (2, 3):
        assert_close(out[b], np.broadcast_to(row, (64, 512)), f"constant V, request {b}")


def test_latent_full_size_sampled():
    w = synth.latent()
    run = DeviceCase(w)
    out, st = run.decode(flags=abi.FLAG_TAG_CHECK)
    assert not st.any()
    # the shortest, the longest and six more (most requests of this batch are
    # cut into several pieces, so these straddle piece boundaries)
    order = np.argsort(w.seq_lens, kind="stable")
    rng = np.random.default_rng(1003)
    idx = np.unique(np.concatenate([[order[0], order[-1]], rng.choice(order[1:-1], size=6, replace=False)]))
    assert idx.size == 8
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
