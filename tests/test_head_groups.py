"""Grouped-query head groups and merge shapes, restated on the host (no GPU).

A KV head's G query heads are run as kv_sub = ceil(G / 8) head groups of
Gs = ceil(G / kv_sub) heads (the last one shorter), each as a virtual KV
head with its own CTAs, because the register-operand MMA takes at most 8
heads on its N dimension.  The merge then takes blocks of float4 columns of
one head group's rows: 64 columns (splits over 4 thread groups), 256 for
very wide groups, or 16 (splits over 16 thread groups) for grids too small
to fill the SMs.  Kernels are instantiated for 1, 2, 4 or 8 head slots (the
latent stream's merge: 16 heads of 512 values); a group of Gs heads takes
the next slot count up and leaves the rest as padding whose columns the
merge skips.  These tests restate that arithmetic, as the launcher and
the merge kernel state it, and check that every query head belongs to
exactly one group of 1 to 8 heads and that the merge blocks tile a group's
columns with each block inside one head or covering whole heads.  The GPU
parity tests (group sizes 1, 2, 3, 4, 8, 16) check the kernels."""


def head_groups(G):
    kv_sub = (G + 7) // 8
    Gs = (G + kv_sub - 1) // kv_sub
    return [(sub * Gs, min(Gs, G - sub * Gs)) for sub in range(kv_sub)]


def merge_shape(D, Gs, wide):
    cols = Gs * D // 4
    if wide:
        kW = cols if cols < 64 else (256 if cols >= 1024 else 64)
    else:
        kW = cols if cols < 16 else 16
    groups, blocks = 256 // kW, cols // kW
    nh = kW * 4 // D if kW * 4 // D > 0 else 1
    return kW, groups, blocks, nh


def test_head_groups_partition_every_group_size():
    for G in range(1, 4097):
        groups = head_groups(G)
        heads = []
        for first, count in groups:
            assert 1 <= count <= 8, (G, first, count)
            heads.extend(range(first, first + count))
        assert heads == list(range(G)), G
        # only the last group may be shorter
        assert all(c == groups[0][1] for _, c in groups[:-1])


def test_virtual_heads_map_back_to_their_kv_head():
    # virtual head v reads KV head v // kv_sub for query heads
    # (v // kv_sub) G + (v % kv_sub) Gs .. + count - 1
    for Hkv, G in ((1, 8), (2, 3), (4, 16), (8, 4), (3, 24), (2, 57)):
        groups = head_groups(G)
        kv_sub = len(groups)
        seen = []
        for v in range(Hkv * kv_sub):
            kv, sub = divmod(v, kv_sub)
            first, count = groups[sub]
            q = list(range(kv * G + first, kv * G + first + count))
            assert all(h // G == kv for h in q)  # the query heads of that KV head
            seen.extend(q)
        assert sorted(seen) == list(range(Hkv * G))


def slots(Gs):
    return 1 if Gs <= 1 else 2 if Gs <= 2 else 4 if Gs <= 4 else 8


def test_every_group_fits_its_slot_count():
    for G in range(1, 4097):
        groups = head_groups(G)
        n = slots(groups[0][1])  # the launcher's slot count for Gs
        assert all(count <= n for _, count in groups)


def test_merge_blocks_tile_a_groups_columns():
    shapes = [(D, kG) for D in (64, 128) for kG in (1, 2, 4, 8)] + [(512, 16)]
    for D, kG in shapes:
        for wide in (True, False):
            kW, groups, blocks, nh = merge_shape(D, kG, wide)
            cols = kG * D // 4
            assert 256 % kW == 0 and groups * kW == 256
            assert blocks * kW == cols  # blocks tile the columns
            for blk in range(blocks):
                lo, hi = blk * kW, (blk + 1) * kW
                h_lo = lo * 4 // D
                heads = {c * 4 // D for c in range(lo, hi)}
                # a block covers nh whole heads or lies inside one head
                assert heads == set(range(h_lo, h_lo + len(heads)))
                assert len(heads) == nh or (len(heads) == 1 and nh == 1)
