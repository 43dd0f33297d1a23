"""The grouped-query split kernel's work split, restated in Python and checked
for the properties the merge relies on (host logic, no GPU).

Every split CTA works out its own pieces from the lengths: the requests, in
request order, lie on a line of T units cut into R ranges
[floor(kT/R), floor((k+1)T/R)); CTA group k takes range k.  Cut rule: each
request's segment of the line is `cost` units of per-piece overhead followed
by its pages, and a piece is the part of one request's pages inside one
range.  Chunk rule (small or lopsided batches): the line is the bare pages,
requests are cut into chunks of about cp pages, at most max_splits of them,
and a range takes the chunks that start in it.  The restatement
follows the kernel step by step (the first piece found by a 32-request pass,
then a walk), so that its index arithmetic can be checked here on many
batches: every valid request is tiled exactly once, in order, by pieces
numbered b * max_splits .. b * max_splits + n_b - 1 with n_b <= max_splits
(so a CTA needs no piece counts of other requests); piece numbers are
distinct and fit the workspace (batch * max_splits); each request has a
first piece (whose CTA records the numbering); under the cut rule each
range's pages plus the overhead units inside it fill the range exactly, and
every busy range holds the same share to within one.  The kernel itself
is checked end to end against the oracle by the GPU parity tests."""
import random

import pytest


def _pages(L, S, max_len):
    return 0 if (L < 1 or L > max_len) else (L + S - 1) // S


def _count(w, off, p, ms):
    """Pieces of a request of p > 0 pages whose cost segment starts at off, and the chunk length."""
    if not w["chunks"]:
        R, T, c = w["R"], w["T"], w["c0"]
        return ((off + c + p) * R - 1) // T - ((off + c + 1) * R - 1) // T + 1, 1
    cp = w["cp"]
    nn = 1 if cp >= p else (p + cp - 1) // cp
    nn = min(nn, ms)
    q = (p + nn - 1) // nn
    return (p + q - 1) // q, q


def _init(lens, S, MP, Hkv, ms, ranges, target, min_chunk, blk, cost=0):
    B = len(lens)
    w = {"max_len": MP * S}
    P = [_pages(L, S, w["max_len"]) for L in lens]
    T = sum(P)
    mx = max(P) if P else 0
    Tc = T + cost * sum(1 for p in P if p)  # the cut rule's line: pages plus `cost` per request
    R = min(ranges, Tc)
    if mx > 0 and ms >= 3:
        R = min(R, (ms - 2) * Tc // (mx + cost))
    w["chunks"] = not (ms >= 3 and T > 0 and R >= 1 and 4 * R >= 3 * ranges)
    if w["chunks"]:
        R = min(ranges, T)
        w["cp"] = max((T * Hkv + target - 1) // target, min_chunk)
        w["c0"] = 0
    else:
        w["cp"] = 0
        w["c0"] = cost
        T = Tc
    w.update(T=T, R=max(R, 1), k=blk // Hkv, b=B, off=0, c=0)
    if T == 0 or w["k"] >= w["R"]:
        return w
    w["r0"] = w["k"] * T // w["R"]
    w["r1"] = (w["k"] + 1) * T // w["R"]
    off_c = 0
    c0 = w["c0"]
    for base in range(0, B, 32):  # one warp pass: 32 requests, a scan of the line
        acc_p = off_c
        for b in range(base, base + 32):
            p = P[b] if b < B else 0
            off = acc_p
            acc_p += p + c0 if p else 0
            has, c_lo = False, 0
            if p > 0 and off + c0 < w["r1"] and off + c0 + p > w["r0"]:
                if not w["chunks"]:
                    has = True
                else:
                    n, ppc = _count(w, off, p, ms)
                    assert w["r0"] - off < p  # the kernel keeps this in 32 bits
                    c_lo = 0 if off >= w["r0"] else (w["r0"] - off + ppc - 1) // ppc
                    has = c_lo < n and off + c_lo * ppc < w["r1"]
            if has:  # the lowest lane with a piece in the range
                w.update(b=b, off=off, c=c_lo)
                return w
        off_c = acc_p
    return w


def _next(w, lens, S, ms):
    B = len(lens)
    while w["b"] < B:
        p = _pages(lens[w["b"]], S, w["max_len"])
        if p == 0:
            w["b"] += 1
            continue
        c0 = w["c0"]
        if w["off"] + c0 >= w["r1"]:
            return None
        n, ppc = _count(w, w["off"], p, ms)
        if not w["chunks"]:
            s0 = w["off"] + c0  # first real page on the cost line
            j = w["k"] - ((s0 + 1) * w["R"] - 1) // w["T"]
            p0 = max(w["r0"], s0) - s0
            p1 = min(w["r1"], s0 + p) - s0
        else:
            if w["c"] >= n:
                w["off"] += p
                w["b"] += 1
                w["c"] = 0
                continue
            if w["off"] + w["c"] * ppc >= w["r1"]:
                return None
            j = w["c"]
            w["c"] += 1
            p0 = j * ppc
            p1 = min(p0 + ppc, p)
        cg = w["b"] * ms + j
        # the kernel ends the walk here instead; it must never be needed
        assert 0 <= j < n <= ms and 0 <= p0 < p1 <= p and cg < B * ms, (j, n, p0, p1, p, cg)
        piece = dict(b=w["b"], cg=cg, p0=p0, p1=p1, nb=n, j=j)
        if not w["chunks"]:
            w["off"] += p + c0
            w["b"] += 1
        return piece
    return None


def _check(lens, S, MP, Hkv, ms, grid, cost=0):
    """Run every CTA group's walk; check the tiling.  Returns (chunk rule?, pieces)."""
    B = len(lens)
    ranges = max(1, grid // Hkv)
    target, min_chunk = ranges * Hkv * 8, (1024 + S - 1) // S
    pieces, loads, chunks = [], [], None
    for k in range(ranges):
        w = _init(lens, S, MP, Hkv, ms, ranges, target, min_chunk, k * Hkv, cost)
        chunks = w["chunks"]
        tot = 0
        while (pc := _next(w, lens, S, ms)) is not None:
            pieces.append(pc)
            tot += pc["p1"] - pc["p0"]
        if not chunks and w["k"] < w["R"]:
            # the range's share of the cost line: its pages plus the overhead
            # segments of the requests that start inside it
            c0, off, virt = w["c0"], 0, 0
            for L in lens:
                p = _pages(L, S, MP * S)
                if p:
                    virt += max(0, min(w["r1"], off + c0) - max(w["r0"], off))
                    off += p + c0
            assert tot + virt == w["r1"] - w["r0"], (k, tot, virt)
            tot += virt
        loads.append(tot)
    cgs = [pc["cg"] for pc in pieces]
    assert len(cgs) == len(set(cgs)), "a piece number used twice"
    by_b = {}
    for pc in pieces:
        by_b.setdefault(pc["b"], []).append(pc)
    for b in range(B):
        p = _pages(lens[b], S, MP * S)
        if p == 0:
            assert b not in by_b
            continue
        ps = sorted(by_b[b], key=lambda x: x["j"])
        n = ps[0]["nb"]
        assert len(ps) == n <= ms and all(x["nb"] == n for x in ps), (b, n, len(ps))
        assert [x["j"] for x in ps] == list(range(n))
        assert [x["cg"] for x in ps] == list(range(b * ms, b * ms + n))
        assert ps[0]["p0"] == 0 and ps[-1]["p1"] == p
        assert all(x["p1"] == y["p0"] for x, y in zip(ps, ps[1:]))
    assert all(0 <= x < B * ms for x in cgs)
    if not chunks and sum(loads):
        busy = [x for x in loads if x]
        assert max(busy) - min(busy) <= 1, loads
    return chunks, len(pieces)


@pytest.mark.parametrize("cost", [0, 16])  # 16: the kernel's piece cost
def test_bench_shapes(cost):
    rng = random.Random(1)
    lens = [int(round(2 ** rng.uniform(0, 16))) for _ in range(64)]
    assert _check(lens, 16, 4096, 8, 64, 456, cost)[0] is False      # ragged batch: cut rule
    assert _check([131072] * 8, 16, 8192, 8, 64, 456, cost) == (False, 64)
    assert _check([37, 100], 16, 8, 8, 64, 456, cost) == (True, 2)   # tiny: chunk rule


@pytest.mark.parametrize("cost", [0, 3, 16])
@pytest.mark.parametrize("seed", range(2))
def test_random_batches(seed, cost):
    rng = random.Random(100 + seed)
    rules = set()
    for _ in range(400):
        B = rng.choice([1, 2, 3, 5, 31, 32, 33, 64, 65, 100, 300])
        S = rng.choice([16, 32, 64])
        MP = rng.choice([1, 2, 8, 64, 600])
        Hkv = rng.choice([1, 2, 4, 8, 16])
        ms = rng.choice([1, 2, 3, 4, 8, 64, 256])
        grid = rng.choice([1, 7, 64, 152, 304, 456])
        kind = rng.random()
        lens = []
        for _ in range(B):
            if kind < 0.3:
                L = rng.randint(1, MP * S)
            elif kind < 0.6:
                L = int(round(2 ** rng.uniform(0, max(1.0, (MP * S).bit_length()))))
            else:  # bad lengths between valid ones
                L = rng.choice([0, -3, 1, S, S + 1, MP * S, MP * S + 1, rng.randint(1, MP * S)])
            lens.append(L)
        rules.add(_check(lens, S, MP, Hkv, ms, grid, cost)[0])
    assert rules == {True, False}
