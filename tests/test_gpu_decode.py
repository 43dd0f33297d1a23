"""GPU paged decode attention parity against the fp64 oracle, element by
element, on sizes that span several tiles, several splits and ragged tails;
status bit-exact; invariants (page permutation, tag on/off) checked on the
GPU itself."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, assert_close, dev_i32
from oracle_helpers import oracle_cache
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu
FP8, BF16 = abi.DTYPE_FP8_E4M3, abi.DTYPE_BF16


def _work(seed, *, G, Hkv, D, S, lens, scale_mode=synth.PER_HEAD, outlier_p=0.01, **kw):
    return synth.make(f"dec{seed}", seed, batch=len(lens), q_heads=G * Hkv, kv_heads=Hkv, head_dim=D, page_size=S,
                      seq_lens=lens, scale_mode=scale_mode, outlier_p=outlier_p, **kw)


def _check(w, dtype, flags=0, max_splits=None, threads=8):
    run = DeviceCase(w, dtype)
    ref, _ = oracle_cache(w, dtype)
    out, st = run.decode(flags=flags, max_splits=max_splits)
    o_ref, st_ref = ref.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, flags=flags,
                               threads=threads)
    assert np.array_equal(st, st_ref), (st, st_ref)
    assert_close(out, o_ref, f"{w.name} dtype={dtype}")
    assert not out[st != 0].any()
    return run, out, st


SHAPES = [
    # (G, Hkv, D, S)
    (4, 8, 128, 16),
    (4, 2, 128, 16),
    (8, 1, 128, 64),
    (4, 1, 64, 16),
    (1, 4, 128, 16),
    (2, 4, 64, 32),
    (8, 2, 64, 16),
    (4, 2, 128, 64),
]


@pytest.mark.parametrize("dtype", [FP8, BF16])
@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_decode_shapes(dtype, si):
    G, Hkv, D, S = SHAPES[si]
    rng = np.random.default_rng(300 + si)
    lens = list(rng.integers(1, 3000, size=6)) + [1, S, S + 1, 5000]
    _check(_work(300 + si, G=G, Hkv=Hkv, D=D, S=S, lens=lens), dtype)


# Group sizes outside 1, 2, 4, 8: up to 8 query heads per head group, with
# padding slots (3, 5, 6, 7), and larger groups cut into several head groups
# that read the same KV head (12, 16, 24, 64).  The attention is the plain
# definition for any grouping of query heads over KV heads.
GENERAL_G = [
    # (G, Hkv, D, S)
    (3, 4, 128, 16),
    (5, 2, 64, 16),
    (6, 2, 128, 32),
    (7, 1, 64, 64),
    (12, 2, 128, 16),
    (16, 2, 128, 16),
    (16, 4, 64, 64),
    (24, 1, 128, 16),
    (64, 1, 64, 16),
]


@pytest.mark.parametrize("dtype", [FP8, BF16])
@pytest.mark.parametrize("gi", range(len(GENERAL_G)))
def test_decode_general_group_sizes(dtype, gi):
    G, Hkv, D, S = GENERAL_G[gi]
    rng = np.random.default_rng(700 + gi)
    lens = list(rng.integers(1, 2500, size=5)) + [1, S + 1, 4000]
    _check(_work(700 + gi, G=G, Hkv=Hkv, D=D, S=S, lens=lens), dtype, flags=abi.FLAG_TAG_CHECK)


def test_decode_general_group_per_token_and_faults():
    # G = 16 (two head groups per KV head) with per-token scales, a stale tag,
    # an out-of-pool page and a bad length, over several splits
    w = _work(710, G=16, Hkv=2, D=128, S=16, lens=[3000, 700, 1500, 20, 2200], scale_mode=synth.PER_TOKEN,
              stale_block_entries=[(1, 3)])
    w.block_table[2, 5] = w.num_pages + 7
    w.seq_lens[3] = w.max_pages * 16 + 1
    run, out, st = _check(w, FP8, flags=abi.FLAG_TAG_CHECK, max_splits=8)
    assert list(st) == [0, abi.ST_STALE_TAG, abi.ST_PAGE_OOB, abi.ST_BAD_LEN, 0]


@pytest.mark.parametrize("max_splits", [1, 2, 3, 64, 256])
def test_split_counts(max_splits):
    # 1, 2: chunk rule; 3: the cut rule's cap leaves too few ranges, so the
    # CTAs fall back to the chunk rule; 64, 256: cut rule (equal page ranges)
    w = _work(400, G=4, Hkv=8, D=128, S=16, lens=[7, 1000, 4097, 20000])
    _check(w, FP8, max_splits=max_splits)


@pytest.mark.parametrize("lens", [[16384] * 8, [16384] * 7 + [100]])
def test_balanced_ranges_cross_requests(lens):
    # one KV head: every CTA owns a range, and a request is cut into more
    # pieces than a warp has lanes (pieces numbered across many CTAs, merged
    # from more than 32 partials)
    w = _work(403, G=8, Hkv=1, D=128, S=64, lens=lens)
    _check(w, FP8, max_splits=64)


@pytest.mark.parametrize("max_splits", [2, 5, 10, 64])
def test_self_split_many_requests(max_splits):
    # 70 requests: each CTA's search for its first piece takes three warp
    # passes; bad lengths (0, -1, beyond the table) count no pages and sit
    # between valid ones.  max_splits 2 and 5: chunk rule; 10: cut rule with
    # fewer ranges than CTA groups (the longest request caps them); 64: cut
    # rule
    rng = np.random.default_rng(404)
    lens = [int(x) for x in np.exp(rng.uniform(0, np.log(20000), size=70)).round()]
    w = _work(404, G=4, Hkv=8, D=128, S=16, lens=lens)
    bad = w.seq_lens.copy()
    bad[3], bad[33], bad[64] = 0, -1, w.max_pages * 16 + 1
    run = DeviceCase(w)
    out, st = run.decode(max_splits=max_splits, seq_lens=dev_i32(bad))
    ref, _ = oracle_cache(w)
    o_ref, st_ref = ref.decode(w.q, bad, w.block_table, w.block_tags, w.softmax_scale, threads=8)
    assert list(np.nonzero(st_ref)[0]) == [3, 33, 64]
    assert np.array_equal(st, st_ref), (st, st_ref)
    assert not out[st != 0].any()
    assert_close(out, o_ref, f"70 requests, max_splits={max_splits}")


def test_per_token_scales_gqa():
    w = _work(401, G=4, Hkv=8, D=128, S=16, lens=[33, 900, 4000], scale_mode=synth.PER_TOKEN)
    _check(w, FP8)


def test_tiny_config_tag_check():
    w = synth.tiny()
    run, out, st = _check(w, FP8, flags=abi.FLAG_TAG_CHECK)
    assert list(st) == [0, abi.ST_STALE_TAG]
    assert not out[1].any()
    off, st_off = run.decode(flags=0)
    assert list(st_off) == [0, 0]
    assert np.array_equal(off[0], out[0])  # tag check changes nothing for a valid request


def test_tag_on_off_identical_when_valid():
    w = _work(402, G=4, Hkv=8, D=128, S=16, lens=[100, 2000, 3333])
    run = DeviceCase(w)
    a, sa = run.decode(flags=0)
    b, sb = run.decode(flags=abi.FLAG_TAG_CHECK)
    assert not sa.any() and not sb.any() and np.array_equal(a, b)


def test_stale_entry_past_context_not_inspected_and_oob():
    w = synth.make("st", 403, batch=4, q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                   seq_lens=[40, 40, 40, 40], room_tokens=64)
    run = DeviceCase(w)
    tags = w.block_tags.copy()
    tags[0, 3] ^= 1  # entry 3 >= ceil(40/16) = 3: never read
    tags[1, 2] ^= 1  # read: stale
    bt = w.block_table.copy()
    bt[2, 1] = w.num_pages + 7  # outside the pool
    lens = w.seq_lens.copy()
    lens[3] = w.max_pages * 16 + 1
    out, st = run.decode(flags=abi.FLAG_TAG_CHECK, table=dev_i32(bt), tags=dev_i32(tags), seq_lens=dev_i32(lens))
    ref, _ = oracle_cache(w)
    o_ref, st_ref = ref.decode(w.q, lens, bt, tags, w.softmax_scale, flags=oracle.FLAG_TAG_CHECK)
    assert list(st_ref) == [0, oracle.ST_STALE_TAG, oracle.ST_PAGE_OOB, oracle.ST_BAD_LEN]
    assert np.array_equal(st, st_ref)
    assert not out[1:].any()
    assert_close(out, o_ref, "stale/oob")


@pytest.mark.parametrize("dtype", [FP8, BF16])
def test_page_permutation_bit_identical_on_gpu(dtype):
    w = _work(404, G=4, Hkv=8, D=128, S=16, lens=[17, 700, 2500])
    run1 = DeviceCase(w, dtype)
    a, _ = run1.decode(flags=abi.FLAG_TAG_CHECK)
    perm = np.random.default_rng(5).permutation(w.num_pages)
    w2 = _work(404, G=4, Hkv=8, D=128, S=16, lens=[17, 700, 2500])
    valid = w.block_table >= 0
    w2.block_table = np.where(valid, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    w2.page_tags = np.zeros_like(w.page_tags)
    w2.page_tags[perm] = w.page_tags
    run2 = DeviceCase(w2, dtype)
    b, _ = run2.decode(flags=abi.FLAG_TAG_CHECK)
    assert np.array_equal(a, b)


def test_special_cases_on_gpu():
    # length 1 -> the value row; constant V -> the constant (BF16 cache keeps it exact)
    w = _work(405, G=4, Hkv=2, D=128, S=16, lens=[1, 1, 50, 300], outlier_p=0.0)
    f = synth.bf16_to_f32(w.v_rows).copy()
    off = w.rows_of(2)[0]
    f[off:] = 0.625  # requests 2 and 3: constant V
    w.v_rows[:] = synth.bf16_bits(f)
    run = DeviceCase(w, BF16)
    out, st = run.decode()
    assert not st.any()
    for b in (0, 1):
        row = w.rows_of(b)[0]
        for h in range(8):
            np.testing.assert_allclose(out[b, h], synth.bf16_to_f32(w.v_rows[row, h // 4]), atol=1e-6, rtol=0)
    np.testing.assert_allclose(out[2:], 0.625, atol=1e-6, rtol=0)


def test_empty_batch_and_deterministic():
    w = _work(406, G=4, Hkv=8, D=128, S=16, lens=[3000, 10, 5000])
    run = DeviceCase(w)
    a, _ = run.decode()
    b, _ = run.decode()
    assert np.array_equal(a, b)
    e = torch.empty(0, 8 * 4, 128, dtype=torch.bfloat16, device="cuda")
    out, st = abi.paged_decode_attention(run.cache, e, run.seq_lens[:0], run.table[:0], run.tags[:0],
                                         w.softmax_scale)
    assert out.shape[0] == 0 and st.shape[0] == 0


def test_host_errors():
    w = _work(407, G=4, Hkv=8, D=128, S=16, lens=[10])
    run = DeviceCase(w)
    with pytest.raises(abi.PfkvError) as e:  # wrong entry point for the cache dtype
        abi.paged_decode_attention_bf16(run.cache, run.q, run.seq_lens, run.table, run.tags, 1.0)
    assert e.value.code == -4
    with pytest.raises(abi.PfkvError) as e:  # too small a workspace
        abi.paged_decode_attention_fp8(run.cache, run.q, run.seq_lens, run.table, run.tags, 1.0,
                                       workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -5
    q20 = torch.zeros(1, 20, 128, dtype=torch.bfloat16, device="cuda")  # 20 query heads over 8 KV heads
    with pytest.raises(abi.PfkvError) as e:
        abi.paged_decode_attention_fp8(run.cache, q20, run.seq_lens, run.table, run.tags, 1.0)
    assert e.value.code == -2
