"""The latent stream's query image, restated on the host (no GPU).

The query-term kernel writes each request's 128 operand rows (two e4m3 terms
of 64 heads) as one 73,728-byte image; the decode kernel copies the image
into two 36,864-byte entries of its page ring and reads it back: the page
loader copies bytes 0-36863 into one entry and 36864-73727 into the next,
each softmax thread moves 32-byte blocks of one row into tensor memory, and
the 8 KB tail image (columns 512-575, 64-byte swizzle) into the query-tail
buffer.  These tests restate the writer's and the readers' index arithmetic
(as the two kernels' comments state it) and check that they agree: every
(row, 16-byte chunk) has its own place, the places tile the image exactly,
the readers find each chunk where the writer put it, the blocks a reader
takes from each ring entry lie inside that entry, and the 16-byte reads of
one phase of eight lanes fall in distinct shared-memory banks.  The GPU
parity tests check the kernels themselves against the oracle."""

IMAGE = 128 * 576          # bytes per request
ENTRY = 36864              # bytes per ring entry (one 64-token page of 576 bytes)
TAIL = 65536               # the tail image's start
T1_T2_ROW = lambda h, t: 32 * (h // 16) + 16 * t + h % 16  # operand row of term t of head h


def writer_offset(R, r):
    """Byte offset of 16-byte chunk r (columns 16 r .. 16 r + 15) of row R."""
    if r < 32:  # columns 0-511: blocks of 128 rows x 32 bytes, 8-row x 16-byte units
        return (r >> 1) * 4096 + (r & 1) * 128 + (R >> 3) * 256 + (R & 7) * 16
    j = r - 32  # columns 512-575: the 64-byte-swizzled tail image
    return TAIL + R * 64 + 16 * (j ^ ((R >> 1) & 3))


def reader_offset(R, k, c):
    """Where a softmax thread reads bytes 16 c .. 16 c + 15 of block k of row R:
    (ring entry, offset inside the entry)."""
    if k < 9:
        return 0, 4096 * k + (R >> 3) * 256 + (R & 7) * 16 + 128 * c
    return 1, 4096 * (k - 9) + (R >> 3) * 256 + (R & 7) * 16 + 128 * c


def test_rows_cover_every_head_and_term_once():
    rows = sorted(T1_T2_ROW(h, t) for h in range(64) for t in range(2))
    assert rows == list(range(128))


def test_writer_tiles_the_image_exactly():
    offs = [writer_offset(R, r) for R in range(128) for r in range(36)]
    assert len(set(offs)) == len(offs)
    assert all(o % 16 == 0 and 0 <= o <= IMAGE - 16 for o in offs)
    assert sorted(offs) == list(range(0, IMAGE, 16))  # 128 x 36 chunks of 16 bytes, no gap
    assert IMAGE == 2 * ENTRY


def test_readers_find_what_the_writer_wrote():
    for R in range(128):
        for k in range(16):
            for c in range(2):
                entry, off = reader_offset(R, k, c)
                assert 0 <= off <= ENTRY - 16  # inside its ring entry
                assert entry * ENTRY + off == writer_offset(R, 2 * k + c)
        # the tail: softmax thread wt copies bytes 32 wt .. 32 wt + 31 of the
        # 8 KB tail image, which starts at byte 28672 of the second entry
        for r in range(32, 36):
            o = writer_offset(R, r)
            assert ENTRY + (ENTRY - (IMAGE - TAIL)) <= o < IMAGE
    assert ENTRY - (IMAGE - TAIL) == 28672
    assert 256 * 32 == IMAGE - TAIL  # 256 softmax threads x 32 bytes


def test_a_phase_of_eight_lanes_reads_distinct_banks():
    # a 16-byte shared-memory read by 32 lanes runs in phases of 8 lanes;
    # lanes are rows R = 32 q + lane of one block, so each phase must touch
    # 8 x 4 distinct 4-byte banks
    for q in range(4):
        for k in range(16):
            for c in range(2):
                for phase in range(4):
                    lanes = range(8 * phase, 8 * phase + 8)
                    banks = set()
                    for lane in lanes:
                        _, off = reader_offset(32 * q + lane, k, c)
                        banks.update(((off // 4) + i) % 32 for i in range(4))
                    assert len(banks) == 32
