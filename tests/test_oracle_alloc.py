"""Pins of the oracle's page allocator (the producer side of the page tags).

Cache-protection passage of "Smaller, faster, safer: running Kimi and GLM at
scale": each page carries a tag that changes whenever the page is
reallocated, and a read through a mapping whose tag no longer matches aborts
the request.  The pins are invariants that any correct allocator keeps
(pages are conserved, never handed to two owners, every hand-out moves the
tag) plus the end-to-end property the passage is about: after a page moves
to a new owner, the old owner's decode is flagged stale by the oracle's
attention, and the new owner's is not.
"""
import numpy as np
import pytest

import oracle
from paged_fp8_kv_quantize_gb300 import synth


def _check_partition(a, held_set):
    free = a.free_list()
    assert len(set(free.tolist())) == free.size, "a page is on the free list twice"
    assert set(free.tolist()).isdisjoint(held_set), "a held page is on the free list"
    assert set(free.tolist()) | held_set == set(range(a.P)), "a page was lost"
    assert np.array_equal(np.flatnonzero(a.held), np.array(sorted(held_set), dtype=np.int64))


def test_fresh_pool_hands_out_increasing_ids_and_bumps_each_tag():
    tags = np.arange(10, dtype=np.uint32) * 7
    before = tags.copy()
    a = oracle.Allocator(10, tags)
    pages, new, st = a.alloc(4)
    assert st == 0 and pages.tolist() == [0, 1, 2, 3]
    assert np.array_equal(new, before[:4] + 1) and np.array_equal(tags[:4], new)
    assert np.array_equal(tags[4:], before[4:])
    assert a.free_count == 6


def test_init_with_held_pages_skips_them():
    tags = np.zeros(6, dtype=np.uint32)
    a = oracle.Allocator(6, tags, held_pages=[1, 4, 4, 99])  # duplicates and out-of-range ids are ignored
    _check_partition(a, {1, 4})
    pages, _, st = a.alloc(4)
    assert st == 0 and pages.tolist() == [0, 2, 3, 5]
    assert a.alloc(1)[2] == oracle.ST_NO_PAGES


def test_exhaustion_is_all_or_nothing():
    tags = np.zeros(5, dtype=np.uint32)
    a = oracle.Allocator(5, tags)
    a.alloc(3)
    snap = (a.free_list(), a.held.copy(), tags.copy())
    pages, new, st = a.alloc(3)
    assert st == oracle.ST_NO_PAGES
    assert pages.tolist() == [-1, -1, -1] and new.tolist() == [0, 0, 0]
    assert np.array_equal(a.free_list(), snap[0]) and np.array_equal(a.held, snap[1])
    assert np.array_equal(tags, snap[2])
    assert a.alloc(0)[2] == 0


def test_free_is_last_in_first_out_and_rejects_bad_entries():
    tags = np.zeros(8, dtype=np.uint32)
    a = oracle.Allocator(8, tags)
    a.alloc(5)
    st = a.free([3, 1, 3, -1, 8, 6])  # 3 twice, two out of range, 6 never taken
    assert st.tolist() == [0, 0, oracle.ST_NOT_HELD, oracle.ST_PAGE_OOB, oracle.ST_PAGE_OOB, oracle.ST_NOT_HELD]
    _check_partition(a, {0, 2, 4})
    pages, _, _ = a.alloc(2)
    assert pages.tolist() == [1, 3]  # the most recently freed first
    assert tags[3] == 2 and tags[1] == 2  # second hand-out of each: tag moved twice
    assert tags[6] == 0  # freeing a page never taken does not touch its tag


def test_realloc_moves_tags_once_and_flags_the_rest():
    tags = np.array([5, 5, 5, 5, 0xFFFFFFFF, 5], dtype=np.uint32)
    a = oracle.Allocator(6, tags, held_pages=[0, 2, 4])
    new, st = a.realloc([2, 4, 2, 1, 7])
    assert st.tolist() == [0, 0, oracle.ST_DUPLICATE, oracle.ST_NOT_HELD, oracle.ST_PAGE_OOB]
    assert new.tolist() == [6, 0, 0, 0, 0]  # 0xFFFFFFFF + 1 wraps to 0
    assert tags.tolist() == [5, 5, 6, 5, 0, 5]
    _check_partition(a, {0, 2, 4})


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_sequences_conserve_pages_and_move_tags(seed):
    rng = np.random.default_rng(seed)
    P = 64
    tags = rng.integers(0, 1 << 32, size=P, dtype=np.uint64).astype(np.uint32)
    a = oracle.Allocator(P, tags)
    held, handouts = set(), np.zeros(P, dtype=np.int64)
    start = tags.copy()
    for _ in range(300):
        op = rng.integers(3)
        if op == 0:
            n = int(rng.integers(0, 12))
            fc = a.free_count
            pages, new, st = a.alloc(n)
            if n > fc:
                assert st == oracle.ST_NO_PAGES
                continue
            assert st == 0 and held.isdisjoint(pages.tolist()) and len(set(pages.tolist())) == n
            held |= set(pages.tolist())
            np.add.at(handouts, pages, 1)
            assert np.array_equal(new, tags[pages])
        elif op == 1 and held:
            pick = rng.choice(sorted(held), size=min(len(held), int(rng.integers(1, 6))), replace=False)
            st = a.free(pick)
            assert not st.any()
            held -= set(pick.tolist())
        elif held:
            pick = rng.choice(sorted(held), size=min(len(held), int(rng.integers(1, 6))), replace=False)
            new, st = a.realloc(pick)
            assert not st.any()
            np.add.at(handouts, pick, 1)
        _check_partition(a, held)
        # every hand-out moved the tag by exactly one, and nothing else did
        assert np.array_equal(tags, (start.astype(np.uint64) + handouts.astype(np.uint64)).astype(np.uint32))


def test_reallocated_page_makes_the_old_owner_stale_in_decode():
    """Two requests map pages through the allocator; one page of request 0
    is freed and handed to request 1.  Request 0's decode (still holding the
    old mapping and tag) aborts; request 1's does not."""
    rng = np.random.default_rng(9)
    P, S, H, D = 12, 16, 1, 64
    tags = rng.integers(0, 1 << 32, size=P, dtype=np.uint64).astype(np.uint32)
    a = oracle.Allocator(P, tags)
    c = oracle.Cache(P, S, H, D, page_tags=tags)  # the cache reads the same tag array
    lens = np.array([40, 20], dtype=np.int32)
    MP = 4
    table = np.full((2, MP), -1, dtype=np.int32)
    btags = np.zeros((2, MP), dtype=np.uint32)
    for b in range(2):
        n = (int(lens[b]) + S - 1) // S
        pages, new, st = a.alloc(n)
        assert st == 0
        table[b, :n], btags[b, :n] = pages, new
    rows = []
    for b in range(2):
        pos = np.arange(lens[b], dtype=np.int32)
        k = synth.bf16_bits(rng.standard_normal((lens[b], H, D)).astype(np.float32))
        v = synth.bf16_bits(rng.standard_normal((lens[b], H, D)).astype(np.float32))
        rows.append((k, v, pos, np.full(lens[b], b, dtype=np.int32)))
    k = np.concatenate([r[0] for r in rows]); v = np.concatenate([r[1] for r in rows])
    pos = np.concatenate([r[2] for r in rows]); rr = np.concatenate([r[3] for r in rows])
    assert not c.append(k, v, pos, table, btags, flags=oracle.FLAG_TAG_CHECK, row_req=rr).any()
    q = synth.bf16_bits(rng.standard_normal((2, 4, D)).astype(np.float32))
    _, st = c.decode(q, lens, table, btags, 0.125, flags=oracle.FLAG_TAG_CHECK)
    assert not st.any()

    victim = int(table[0, 1])
    assert not a.free([victim]).any()
    got, new, st = a.alloc(1)
    assert st == 0 and got[0] == victim  # the freed page is the next one handed out
    table2, btags2 = table.copy(), btags.copy()
    table2[1, 2], btags2[1, 2] = victim, new[0]
    lens2 = np.array([40, 33], dtype=np.int32)
    _, st = c.decode(q, lens2, table2, btags2, 0.125, flags=oracle.FLAG_TAG_CHECK)
    assert st.tolist() == [oracle.ST_STALE_TAG, 0]
    _, st = c.decode(q, lens2, table2, btags2, 0.125, flags=0)  # the check is off by default
    assert not st.any()
