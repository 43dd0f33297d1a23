"""Pins for the oracle's paged decode attention, page walk, tags and append.

Checked against: torch SDPA in fp64 on an unpaged contiguous copy (library
routine), closed-form special cases, invariants (page permutation, tag flag
on/off) and deliberately stale / out-of-range / bad-length inputs.
"""
import numpy as np
import pytest

import oracle
from oracle_helpers import dense_reference, oracle_cache
from paged_fp8_kv_quantize_gb300 import synth

FP8, BF16 = oracle.DTYPE_FP8, oracle.DTYPE_BF16


def _small(seed, *, G=4, Hkv=2, D=64, Dv=None, S=16, B=3, max_len=70, scale_mode=synth.PER_HEAD,
           kv_shared=False, outlier_p=0.01):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len + 1, size=B)
    return synth.make(f"small{seed}", seed, batch=B, q_heads=G * Hkv, kv_heads=Hkv, head_dim=D, v_head_dim=Dv,
                      kv_shared=kv_shared, page_size=S, seq_lens=lens, scale_mode=scale_mode,
                      outlier_p=outlier_p)


CASES = [
    dict(G=4, Hkv=2, D=64, S=16),
    dict(G=1, Hkv=3, D=16, S=4),
    dict(G=8, Hkv=1, D=128, S=16),
    dict(G=2, Hkv=2, D=32, S=8, scale_mode=synth.PER_TOKEN),
    dict(G=4, Hkv=1, D=40, Dv=32, S=4, kv_shared=True, scale_mode=synth.PER_TOKEN, Hkv_=1),
    dict(G=3, Hkv=2, D=32, S=8),
    dict(G=16, Hkv=1, D=64, S=16, B=2),
]


@pytest.mark.parametrize("dtype", [FP8, BF16])
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_decode_matches_torch_sdpa(dtype, ci):
    kw = {k: v for k, v in CASES[ci].items() if not k.endswith("_")}
    if dtype == BF16 and kw.get("kv_shared"):
        kw["scale_mode"] = synth.PER_HEAD
    w = _small(100 + ci, **kw)
    c, st = oracle_cache(w, dtype)
    assert not st.any()
    out, status = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale)
    assert not status.any()
    ref = dense_reference(c, w.q, w.seq_lens, w.block_table, w.softmax_scale)
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_threads_do_not_change_results():
    w = _small(7, G=4, Hkv=2, D=64, S=16, B=5)
    c, _ = oracle_cache(w)
    a, sa = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, threads=1)
    b, sb = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, threads=4)
    assert np.array_equal(a, b) and np.array_equal(sa, sb)


def _decoded_rows(c, w, b):
    """Dequantized K and V rows of request b, fp64, in token order (via the dense helper's decoder)."""
    from oracle_helpers import dequant_pool

    K = dequant_pool(c, "k")
    V = K[..., : c.Dv] if c.kv_shared else dequant_pool(c, "v")
    L = int(w.seq_lens[b])
    n = (L + c.S - 1) // c.S
    pages = w.block_table[b, :n]
    kb = K[pages].transpose(1, 0, 2, 3).reshape(c.H, n * c.S, -1)[:, :L]
    vb = V[pages].transpose(1, 0, 2, 3).reshape(c.H, n * c.S, -1)[:, :L]
    return kb, vb


def test_length_one_returns_the_value_row():
    w = _small(11, G=4, Hkv=2, D=64, S=16, B=2)
    w.seq_lens[:] = 1
    c, _ = oracle_cache(w)
    out, st = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale)
    for b in range(w.batch):
        _, vb = _decoded_rows(c, w, b)
        for h in range(w.q_heads):
            assert np.array_equal(out[b, h], vb[h // w.group, 0])


def test_zero_query_is_mean_of_values():
    w = _small(12, G=2, Hkv=2, D=32, S=8, B=3)
    w.q[:] = 0
    c, _ = oracle_cache(w)
    out, _ = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale)
    for b in range(w.batch):
        _, vb = _decoded_rows(c, w, b)
        for h in range(w.q_heads):
            np.testing.assert_allclose(out[b, h], vb[h // w.group].mean(axis=0), rtol=0, atol=1e-12)


def test_constant_values_give_the_constant():
    w = _small(13, G=4, Hkv=1, D=64, S=16, B=2, outlier_p=0.0)
    w.v_rows[:] = synth.bf16_bits(np.full(w.v_rows.shape, 0.75, np.float32))
    c, _ = oracle_cache(w, BF16)
    out, _ = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale)
    np.testing.assert_allclose(out, 0.75, rtol=0, atol=1e-14)  # softmax weights sum to one


def test_dominant_key_selects_its_value():
    w = synth.make("dom", 14, batch=1, q_heads=1, kv_heads=1, head_dim=16, page_size=4, seq_lens=[30])
    t_star = 17
    w.q[:] = synth.bf16_bits(np.ones((1, 1, 16), np.float32))
    k = synth.bf16_to_f32(w.k_rows).copy()
    k[:] = 0.0
    k[t_star] = 8.0  # score 16*8*tau*... dominates all others (which are 0)
    w.k_rows[:] = synth.bf16_bits(k)
    c, _ = oracle_cache(w, BF16)
    out, _ = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, softmax_scale=1.0)
    _, vb = _decoded_rows(c, w, 0)
    # weight of the other 29 tokens: 29*e^-128 relative -- far below fp64 resolution
    np.testing.assert_allclose(out[0, 0], vb[0, t_star], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [FP8, BF16])
def test_page_permutation_is_bit_identical(dtype):
    w = _small(15, G=4, Hkv=2, D=64, S=4, B=4, max_len=60)
    c1, _ = oracle_cache(w, dtype)
    o1, s1 = c1.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, flags=1)
    rng = np.random.default_rng(99)
    perm = rng.permutation(w.num_pages)
    w2 = synth.make(w.name, w.seed, batch=w.batch, q_heads=w.q_heads, kv_heads=w.kv_heads, head_dim=w.head_dim,
                    page_size=w.page_size, seq_lens=w.seq_lens, outlier_p=0.01)
    assert np.array_equal(w2.k_rows, w.k_rows)
    valid = w.block_table >= 0
    w2.block_table = np.where(valid, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    w2.page_tags = np.zeros_like(w.page_tags)
    w2.page_tags[perm] = w.page_tags
    c2, _ = oracle_cache(w2, dtype)
    o2, s2 = c2.decode(w2.q, w2.seq_lens, w2.block_table, w2.block_tags, w2.softmax_scale, flags=1)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_tiny_stale_tag_aborts_exactly_that_request():
    w = synth.tiny()
    assert w.stale and all(b == 1 for b, _ in w.stale)
    c, st = oracle_cache(w)
    assert not st.any()
    on, s_on = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, flags=oracle.FLAG_TAG_CHECK)
    off, s_off = c.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale, flags=0)
    assert list(s_on) == [0, oracle.ST_STALE_TAG]
    assert list(s_off) == [0, 0]  # the check is off by default
    assert not on[1].any()  # aborted: no data returned
    assert np.array_equal(on[0], off[0])  # tag check changes nothing for a valid request
    assert off[1].any()


def test_stale_entry_past_the_context_is_not_inspected():
    # request 0 gets table entries past ceil(5/4) = 2 (room for appends)
    w2 = synth.make("room", 16, batch=2, q_heads=4, kv_heads=1, head_dim=16, page_size=4, seq_lens=[5, 9],
                    room_tokens=8)
    w2.block_tags[0, 2] ^= 1  # entry 2 >= ceil(5/4): never read
    c, _ = oracle_cache(w2)
    _, s = c.decode(w2.q, w2.seq_lens, w2.block_table, w2.block_tags, w2.softmax_scale, flags=1)
    assert list(s) == [0, 0]
    w2.block_tags[0, 1] ^= 1  # entry 1 < 2: read
    _, s = c.decode(w2.q, w2.seq_lens, w2.block_table, w2.block_tags, w2.softmax_scale, flags=1)
    assert list(s) == [oracle.ST_STALE_TAG, 0]


def test_out_of_range_page_and_bad_length():
    w = synth.make("oob", 17, batch=4, q_heads=4, kv_heads=1, head_dim=16, page_size=4, seq_lens=[6, 6, 6, 6])
    c, _ = oracle_cache(w)
    bt = w.block_table.copy()
    lens = w.seq_lens.copy()
    bt[0, 1] = w.num_pages  # past the pool
    bt[1, 0] = -1
    lens[2] = 0  # empty context
    lens[3] = w.max_pages * w.page_size + 1  # past the request's table
    out, s = c.decode(w.q, lens, bt, w.block_tags, w.softmax_scale, flags=0)
    assert list(s) == [oracle.ST_PAGE_OOB, oracle.ST_PAGE_OOB, oracle.ST_BAD_LEN, oracle.ST_BAD_LEN]
    assert not out.any()


@pytest.mark.parametrize("mode", [synth.PER_HEAD, synth.PER_TOKEN])
def test_append_writes_exactly_its_slot(mode):
    w = synth.make("app", 18, batch=3, q_heads=8, kv_heads=2, head_dim=32, page_size=8, seq_lens=[3, 17, 9],
                   room_tokens=4, scale_mode=mode)
    c = oracle.Cache(w.num_pages, 8, 2, 32, 32, False, FP8, mode, w.page_tags,
                     k_scale=np.array([0.01, 0.02], np.float32), v_scale=np.array([0.03, 0.04], np.float32))
    rng = np.random.default_rng(3)
    k_new = synth.bf16_bits(rng.standard_normal((3, 2, 32)).astype(np.float32))
    v_new = synth.bf16_bits(rng.standard_normal((3, 2, 32)).astype(np.float32))
    pos = w.seq_lens.copy()
    st = c.append(k_new, v_new, pos, w.block_table, w.block_tags, flags=1)
    assert not st.any()
    K, V = c.k_rows(), c.v_rows()
    touched = np.zeros(K.shape[:3], bool)
    for b in range(3):
        p, slot = w.block_table[b, pos[b] // 8], pos[b] % 8
        for h in range(2):
            if mode == synth.PER_HEAD:
                sk, sv = c.k_scale[h], c.v_scale[h]
            else:
                fk = np.abs(synth.bf16_to_f32(k_new[b, h])).max()
                fv = np.abs(synth.bf16_to_f32(v_new[b, h])).max()
                sk, sv = np.float32(fk) / np.float32(448), np.float32(fv) / np.float32(448)
                r = (p * 2 + h) * 8 + slot
                assert c.k_scale[r] == sk and c.v_scale[r] == sv
            want_k = [oracle.quantize(int(x), float(sk)) for x in k_new[b, h]]
            want_v = [oracle.quantize(int(x), float(sv)) for x in v_new[b, h]]
            assert list(K[p, h, slot]) == want_k and list(V[p, h, slot]) == want_v
            touched[p, h, slot] = True
    assert np.all(K[~touched] == 0xA5) and np.all(V[~touched] == 0xA5)


def test_append_refuses_bad_destinations():
    w = synth.make("app2", 19, batch=4, q_heads=4, kv_heads=1, head_dim=16, page_size=4, seq_lens=[2, 2, 2, 2],
                   room_tokens=4)
    c = oracle.Cache(w.num_pages, 4, 1, 16, 16, False, FP8, synth.PER_HEAD, w.page_tags,
                     k_scale=np.ones(1, np.float32), v_scale=np.ones(1, np.float32))
    k_new = synth.bf16_bits(np.ones((4, 1, 16), np.float32))
    tags = w.block_tags.copy()
    bt = w.block_table.copy()
    pos = w.seq_lens.copy()
    tags[0, 0] ^= 7  # stale destination
    bt[1, 0] = w.num_pages + 3  # out of the pool
    pos[2] = -1  # before the context
    pos[3] = w.max_pages * 4  # past the table
    st = c.append(k_new, k_new, pos, bt, tags, flags=oracle.FLAG_TAG_CHECK)
    assert list(st) == [oracle.ST_STALE_TAG, oracle.ST_PAGE_OOB, oracle.ST_BAD_LEN, oracle.ST_BAD_LEN]
    assert np.all(c.k_pool == 0xA5) and np.all(c.v_pool == 0xA5)
    # with the check off, the stale destination is written
    st = c.append(k_new, k_new, w.seq_lens, w.block_table, tags, flags=0)
    assert not st.any() and not np.all(c.k_pool == 0xA5)
