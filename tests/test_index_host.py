"""Index arithmetic of the kernels, checked on the CPU (no GPU needed).

compute-sanitizer is not available here, so the address formulas of the
kernels whose indexing is least obvious are restated in Python and checked
exhaustively over shape classes:

* the row-class kernel: every raw TMA box lands inside its raw stage,
  128-byte aligned and disjoint from the others; every read of the realign
  step stays inside the box it belongs to; every 16-byte chunk of the
  swizzled stage is written exactly once per K block;
* the row-class maps: each class map starts at the 16-byte boundary at or
  below its first row (so inside the matrix's allocation), its rows all sit
  the same delta < 8 elements past that boundary, its pitch is a multiple of
  16 bytes, and it ends at the last row's end;
* the even split of a send list over CTAs used by the exchange kernels.

The constants and formulas mirror fused_tcr.cu and ia2av.cu; a change there
must be made here too.
"""
import itertools

import numpy as np
import pytest

KROW, NROW, BK, BM_CTA, BN_CTA = 144, 272, 64, 128, 128
RAW_A = BM_CTA * KROW
RAW_B = BN_CTA * KROW
SW_A, SW_B, B_BOX = 16384, 16384, 8192


def _classes(rowlen, aligned=True):
    n = 1
    while (rowlen * 2 * n) % 16:
        n *= 2
    if n == 1 and not aligned:
        n = 2
    return n


def _stage_addresses(wt, ncx, ncw):
    """(raw boxes, realign reads and writes) of one CTA and K block."""
    lgx, lgw = ncx.bit_length() - 1, ncw.bit_length() - 1
    boxes = [(b * (RAW_A >> lgx), (BM_CTA // ncx) * KROW) for b in range(ncx)]
    if wt:
        boxes += [(RAW_A + b * (RAW_B >> lgw), (BN_CTA // ncw) * KROW) for b in range(ncw)]
    else:
        boxes += [(RAW_A + b * ((BK * NROW) >> lgw), (BK // ncw) * NROW) for b in range(ncw)]
    sx, sw = 5 - lgx, 5 - lgw
    steps = []
    for bt in range(16):                       # 16 batches of four warp steps
        for s in range(4):
            for lane in range(32):
                rg, c = lane >> 3, lane & 7
                if bt < 8:
                    it0 = bt * 4
                    b, v0 = it0 >> sx, it0 & ((1 << sx) - 1)
                    j = 4 * (v0 + s) + rg
                    i = b + (j << lgx)
                    box = b * (RAW_A >> lgx)
                    src, box_end = box + j * KROW + c * 16, box + (BM_CTA // ncx) * KROW
                    dst = i * 128 + ((c ^ (i & 7)) << 4)
                elif wt:
                    it0 = (bt - 8) * 4
                    b, v0 = it0 >> sw, it0 & ((1 << sw) - 1)
                    j = 4 * (v0 + s) + rg
                    i = b + (j << lgw)
                    box = RAW_A + b * (RAW_B >> lgw)
                    src, box_end = box + j * KROW + c * 16, box + (BN_CTA // ncw) * KROW
                    dst = SW_A + i * 128 + ((c ^ (i & 7)) << 4)
                else:
                    it0 = (bt - 8) * 4
                    b, v0 = it0 >> sw, it0 & ((1 << sw) - 1)
                    j = 2 * (v0 + s) + (rg >> 1)
                    half, kr = rg & 1, b + (j << lgw)
                    box = RAW_A + b * ((BK * NROW) >> lgw)
                    src = box + j * NROW + (half * 8 + c) * 16
                    box_end = box + (BK // ncw) * NROW
                    dst = SW_A + half * B_BOX + kr * 128 + ((c ^ (kr & 7)) << 4)
                steps.append((src, box_end, dst))
    return boxes, steps


@pytest.mark.parametrize("wt", [0, 1])
@pytest.mark.parametrize("ncx,ncw", list(itertools.product((1, 2, 4, 8), repeat=2)))
def test_row_class_stage_addressing(wt, ncx, ncw):
    boxes, steps = _stage_addresses(wt, ncx, ncw)
    for off, size in boxes:
        assert off % 128 == 0 and off + size <= RAW_A + RAW_B
    for (o1, s1), (o2, _) in zip(sorted(boxes), sorted(boxes)[1:]):
        assert o1 + s1 <= o2
    written = {}
    for src, box_end, dst in steps:
        assert src % 16 == 0 and src + 32 <= box_end       # both granules of the shift
        assert dst % 16 == 0 and dst + 16 <= SW_A + SW_B
        written[dst] = written.get(dst, 0) + 1
    assert len(written) == (SW_A + SW_B) // 16 and set(written.values()) == {1}


def _class_map(base, rowlen, nrows, n, q):
    """(map base address, delta, inner extent, outer extent, pitch) of class q."""
    a = base + q * rowlen * 2
    a16 = a & ~15
    d = (a - a16) // 2
    return a16, d, rowlen + d, (nrows - q + n - 1) // n, rowlen * 2 * n


@pytest.mark.parametrize("rowlen", [1, 3, 6, 7, 8, 9, 65, 100, 257, 1025, 2050, 4100, 65535])
@pytest.mark.parametrize("base_off", [0, 2, 6, 14])
def test_row_class_maps_stay_inside_the_matrix(rowlen, base_off):
    base = (1 << 20) + base_off                           # an element-aligned pointer
    alloc_start = base & ~15                              # allocations start 16-byte aligned
    nrows = 37
    end = base + nrows * rowlen * 2
    n = _classes(rowlen, aligned=base_off == 0)
    for q in range(min(n, nrows)):
        a16, d, inner, outer, pitch = _class_map(base, rowlen, nrows, n, q)
        assert a16 >= alloc_start and 0 <= d < 8 and pitch % 16 == 0
        assert pitch >= inner * 2                          # rows do not overlap in the map
        for j in range(outer):
            row = q + j * n
            start = base + row * rowlen * 2
            assert start - (a16 + j * pitch) == 2 * d      # every row sits delta past its boundary
        last = q + (outer - 1) * n
        assert a16 + (outer - 1) * pitch + inner * 2 == base + (last + 1) * rowlen * 2 <= end


@pytest.mark.parametrize("n", [0, 1, 5, 17, 1000, 2 ** 40 + 7])
@pytest.mark.parametrize("parts", [1, 3, 38, 152, 1216])
def test_even_split_covers_the_send_list(n, parts):
    q, rem = divmod(n, parts)
    prev = 0
    for part in range(parts):
        lo = q * part + min(part, rem)
        hi = lo + q + (1 if part < rem else 0)
        assert lo == prev and hi >= lo
        prev = hi
    assert prev == n
