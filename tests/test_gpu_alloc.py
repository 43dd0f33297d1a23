"""GPU page allocator against the oracle's sequential allocator: every
returned page id, tag and status, the page-tag array and the free list are
bit-exact after each call; plus the end-to-end effect on the tag check
(a page moved to a new owner makes the old owner's decode abort)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DeviceCase, dev_i32
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu


def u32(t):
    return t.cpu().numpy().view(np.uint32)


def i32(t):
    return t.cpu().numpy().astype(np.int32)


def _same_state(ga, gtags, oa, otags):
    torch.cuda.synchronize()
    assert ga.free_count() == oa.free_count
    assert np.array_equal(i32(ga.free_list()), oa.free_list())
    assert np.array_equal(u32(gtags), otags)


@pytest.mark.parametrize("seed,P,max_n", [(11, 97, 40), (12, 5000, 3000)])
def test_random_sequences_match_oracle(seed, P, max_n):
    """Lists up to 3000 ids cross the kernels' 1024-entry chunks; free and
    realloc lists carry repeats, out-of-range ids and pages not held."""
    rng = np.random.default_rng(seed)
    tags0 = rng.integers(0, 1 << 32, size=P, dtype=np.uint64).astype(np.uint32)
    tags0[:3] = 0xFFFFFFFF  # wrap-around on the first hand-out
    otags = tags0.copy()
    oa = oracle.Allocator(P, otags)
    gtags = dev_i32(tags0)
    ga = abi.PageAllocator(P)
    _same_state(ga, gtags, oa, otags)
    for step in range(60):
        op = int(rng.integers(3))
        if op == 0:
            n = int(rng.integers(0, max_n))
            gp, gt, gs = ga.alloc(n, gtags)
            op_, ot, os_ = oa.alloc(n)
            assert int(u32(gs)[0]) == os_, step
            assert np.array_equal(i32(gp), op_) and np.array_equal(u32(gt), ot), step
        else:
            n = int(rng.integers(1, max_n))
            ids = rng.integers(-2, P + 2, size=n).astype(np.int32)
            held = np.flatnonzero(oa.held)
            if held.size:  # mostly held pages, some repeated
                k = int(rng.integers(0, n + 1))
                ids[:k] = rng.choice(held, size=k)
                rng.shuffle(ids)
            if op == 1:
                gs = ga.free(dev_i32(ids))
                os_ = oa.free(ids)
                assert np.array_equal(u32(gs), os_), step
            else:
                gt, gs = ga.realloc(dev_i32(ids), gtags)
                ot, os_ = oa.realloc(ids)
                assert np.array_equal(u32(gs), os_) and np.array_equal(u32(gt), ot), step
        _same_state(ga, gtags, oa, otags)


def test_init_with_held_pages_on_a_large_pool():
    """Init is grid-wide: 3M pages, a million of them held (with repeats and
    ids outside the pool in the list)."""
    rng = np.random.default_rng(13)
    P = 3_000_000
    held = rng.integers(-5, P + 5, size=1_000_000).astype(np.int32)
    otags = np.zeros(P, dtype=np.uint32)
    oa = oracle.Allocator(P, otags, held_pages=held)
    ga = abi.PageAllocator(P, held_pages=dev_i32(held))
    gtags = torch.zeros(P, dtype=torch.int32, device="cuda")
    _same_state(ga, gtags, oa, otags)
    gp, gt, gs = ga.alloc(2000, gtags)
    op_, ot, os_ = oa.alloc(2000)
    assert int(u32(gs)[0]) == os_ == 0
    assert np.array_equal(i32(gp), op_) and np.array_equal(u32(gt), ot)


def test_exhausted_pool_takes_nothing():
    ga = abi.PageAllocator(10)
    tags = torch.zeros(10, dtype=torch.int32, device="cuda")
    ga.alloc(8, tags)
    gp, gt, gs = ga.alloc(3, tags)
    torch.cuda.synchronize()
    assert int(u32(gs)[0]) == abi.ST_NO_PAGES
    assert i32(gp).tolist() == [-1, -1, -1] and u32(gt).tolist() == [0, 0, 0]
    assert ga.free_count() == 2
    assert u32(tags).tolist() == [1] * 8 + [0, 0]


def test_moved_page_aborts_the_old_owner():
    """Pages of a small GQA workload come from the allocator; one page of
    request 0 is freed and handed to request 1.  With the tag check on,
    request 0 (old mapping, old tag) aborts with zero output and request 1
    does not; with the check off nothing is flagged."""
    w = synth.make("alloc_e2e", 700, batch=2, q_heads=8, kv_heads=2, head_dim=128, page_size=16, seq_lens=[50, 30],
                   room_tokens=20, num_pages=12)
    P = w.num_pages
    ga = abi.PageAllocator(P)
    run = DeviceCase(w, fill=False)
    table = np.full_like(w.block_table, -1)
    btags = np.zeros_like(w.block_tags)
    for b in range(w.batch):
        n = int((w.seq_lens[b] + w.page_size - 1) // w.page_size)
        gp, gt, gs = ga.alloc(n, run.cache.page_tags)
        assert int(u32(gs)[0]) == 0
        table[b, :n], btags[b, :n] = i32(gp), u32(gt)
    run.table, run.tags = dev_i32(table), dev_i32(btags)
    rows = np.concatenate([np.arange(w.seq_lens[b]) for b in range(w.batch)]).astype(np.int32)
    req = np.concatenate([np.full(w.seq_lens[b], b) for b in range(w.batch)]).astype(np.int32)
    kk = torch.randn(rows.size, w.kv_heads, 128, device="cuda").bfloat16()
    vv = torch.randn(rows.size, w.kv_heads, 128, device="cuda").bfloat16()
    abi.calibrate_scales(kk, run.cache.k_scale)
    abi.calibrate_scales(vv, run.cache.v_scale)
    st = abi.kv_append_quantize(run.cache, kk, vv, dev_i32(rows), run.table, run.tags, flags=abi.FLAG_TAG_CHECK,
                                row_req=dev_i32(req), batch=w.batch)
    torch.cuda.synchronize()
    assert not st.any()
    out, st = run.decode(flags=abi.FLAG_TAG_CHECK)
    assert not st.any() and np.abs(out).max() > 0

    victim = int(table[0, 1])
    assert not ga.free(dev_i32(np.array([victim]))).any()
    gp, gt, _ = ga.alloc(1, run.cache.page_tags)
    assert int(i32(gp)[0]) == victim
    table2, btags2 = table.copy(), btags.copy()
    table2[1, 2], btags2[1, 2] = victim, u32(gt)[0]
    lens2 = dev_i32(np.array([50, 33]))
    out, st = run.decode(flags=abi.FLAG_TAG_CHECK, seq_lens=lens2, table=dev_i32(table2), tags=dev_i32(btags2))
    assert st.tolist() == [abi.ST_STALE_TAG, 0]
    assert not out[0].any() and np.abs(out[1]).max() > 0
    _, st = run.decode(flags=0, seq_lens=lens2, table=dev_i32(table2), tags=dev_i32(btags2))
    assert not st.any()
