"""The quantiser's shared-memory image and register views, checked on the CPU.

The index arithmetic of quantize_tile_kernel is restated here from its source
comments (the TMA box placement, the row-view lane map and offsets, the
column-view lane map and offsets) and checked:

* the 128-byte-swizzled image puts tile element (r, c) at the byte the kernel
  header states, and every byte of a 32 KB slot holds exactly one element;
* the row view (lane pairs over 16 rows per warp) and the column view (4
  columns x 16 rows per lane) each cover the 128 x 128 tile exactly once, and
  each lane's values are the rows / columns its code stores assume;
* every warp-wide shared-memory load of both views takes the minimum number
  of wavefronts (4 for 16-byte loads, 2 for 8-byte loads): no bank conflicts;
* every TMA box starts on a 16-byte boundary inside the tensor, for plain
  inputs and for the SiLU-gated prologue's [g || u] input.
"""

import numpy as np

WARPS = 8


def swizzled_offset(r, c):
    """Byte offset of tile element (r, c): r = 16 a + l, c = 64 h + 8 k + e
    -> 16384 h + 1024 l + 128 a + 16 (k XOR a) + 2 e."""
    a, l = r // 16, r % 16
    h, k, e = c // 64, (c % 64) // 8, c % 8
    return 16384 * h + 1024 * l + 128 * a + 16 * (k ^ a) + 2 * e


def decode(off):
    h, rest = divmod(off, 16384)
    l, rest = divmod(rest, 1024)
    a, rest = divmod(rest, 128)
    chunk, e2 = divmod(rest, 16)
    k = chunk ^ a
    return 16 * a + l, 64 * h + 8 * k + e2 // 2


def tma_box_image():
    """Element -> byte, by placing each TMA box the way quant_fill issues it:
    lane (l, h) copies view rows y..y+7 (input rows 16 a + l) x 64 columns
    into buf + 16384 h + 1024 l, 128 bytes per row, 128-byte swizzle (chunk k
    of smem row a lands at chunk k XOR (a mod 8))."""
    where = {}
    for lane in range(32):
        l, h = lane >> 1, lane & 1
        base = 16384 * h + 1024 * l
        for a in range(8):
            for k in range(8):
                for e in range(8):
                    r, c = 16 * a + l, 64 * h + 8 * k + e
                    where[(r, c)] = base + 128 * a + 16 * (k ^ (a % 8)) + 2 * e
    return where


def test_tma_boxes_build_the_stated_image():
    where = tma_box_image()
    assert len(where) == 128 * 128
    offs = sorted(where.values())
    assert offs == list(range(0, 32768, 2))  # every bf16 slot used once
    for (r, c), off in where.items():
        assert off == swizzled_offset(r, c)
        assert decode(off) == (r, c)


def row_view(warp, lane):
    """(row, [16-byte offsets of rv[0..7]], [first column of each]) of a lane."""
    jj, hh = lane >> 1, lane & 1
    ra = (jj & 1) | (((jj >> 2) & 1) << 1) | (((jj >> 1) & 1) << 2)
    wrow = 16 * ra + 2 * warp + (jj >> 3)
    roff = 1024 * (2 * warp + (jj >> 3)) + 128 * ra + (((2 * hh) ^ ra) << 4)
    offs = []
    for m in range(4):
        offs.append(16384 * (m >> 1) + (roff ^ (64 * (m & 1))))
        offs.append(16384 * (m >> 1) + (roff ^ (64 * (m & 1) + 16)))
    cols = [32 * m + 16 * hh + 8 * u for m in range(4) for u in range(2)]
    return wrow, offs, cols


def col_view(warp, lane):
    """([8-byte offsets of cv[0..15]], first column, first row) of a lane."""
    cq, g = lane & 3, lane >> 2
    rg = 2 * (g & 3) + (g >> 2)
    coff = 16384 * (warp >> 2) + 128 * rg + (((2 * (warp & 3) + (cq >> 1)) ^ rg) << 4) + 8 * (cq & 1)
    return [coff + 1024 * k for k in range(16)], 16 * warp + 4 * cq, 16 * rg


def test_row_view_covers_the_tile_once_in_store_order():
    seen = np.zeros((128, 128), np.int32)
    for w in range(WARPS):
        for lane in range(32):
            row, offs, cols = row_view(w, lane)
            for off, c0 in zip(offs, cols):
                for e in range(8):  # a 16-byte load: 8 consecutive columns of one row
                    assert decode(off + 2 * e) == (row, c0 + e)
                    seen[row, c0 + e] += 1
    assert np.all(seen == 1)


def test_col_view_covers_the_tile_once():
    seen = np.zeros((128, 128), np.int32)
    for w in range(WARPS):
        for lane in range(32):
            offs, c0, r0 = col_view(w, lane)
            for k, off in enumerate(offs):
                for i in range(4):  # an 8-byte load: 4 consecutive columns of row r0 + k
                    assert decode(off + 2 * i) == (r0 + k, c0 + i)
                    seen[r0 + k, c0 + i] += 1
    assert np.all(seen == 1)


def wavefronts(addrs, size):
    """Shared-memory wavefronts of one warp-wide load of `size` bytes per lane:
    lanes are served in phases of 128 bytes (8 lanes for 16-byte loads, 16 for
    8-byte loads); a phase takes as many wavefronts as the most distinct 4-byte
    words any one of the 32 banks must deliver."""
    per_phase = 128 // size
    total = 0
    for p in range(0, 32, per_phase):
        banks = {}
        for a in addrs[p:p + per_phase]:
            for wd in range(a // 4, (a + size) // 4):
                banks.setdefault(wd % 32, set()).add(wd)
        total += max(len(v) for v in banks.values())
    return total


def test_both_views_load_without_bank_conflicts():
    for w in range(WARPS):
        for i in range(8):
            addrs = [row_view(w, lane)[1][i] for lane in range(32)]
            assert wavefronts(addrs, 16) == 4, (w, i)
        for k in range(16):
            addrs = [col_view(w, lane)[0][k] for lane in range(32)]
            assert wavefronts(addrs, 8) == 2, (w, k)


def test_tma_box_coordinates_are_aligned_and_in_bounds():
    """x = l * xrow + 128 ct + 64 h (+ C for the prologue's u tile) over the
    [R/16, 16 xrow] view, boxes of 64 columns x 8 view rows at y = 8 rt."""
    for R, C, glu in ((128, 128, False), (384, 640, False), (256, 256, True), (1152, 384, True)):
        xrow = 2 * C if glu else C
        dims_x, dims_y = 16 * xrow, R // 16
        for rt in range(R // 128):
            for ct in range(C // 128):
                for lane in range(32):
                    l, h = lane >> 1, lane & 1
                    xs = [l * xrow + 128 * ct + 64 * h]
                    if glu:
                        xs.append(xs[0] + C)
                    for x in xs:
                        assert (x * 2) % 16 == 0          # bf16: x a multiple of 8 elements
                        assert 0 <= x and x + 64 <= dims_x
                    assert 0 <= 8 * rt and 8 * rt + 8 <= dims_y
        # the largest row length the launcher accepts keeps x in int32
        assert 16 * (2 * (1 << 26) if glu else (1 << 27)) <= 2 ** 31
