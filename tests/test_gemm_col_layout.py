"""The WGRAD GEMM's column promotion layout, checked on the CPU.

WGRAD's scale is the outer product sa(i) sb(j) of two vectors per 128-deep
slice.  Its promotion threads read the partial sums from tensor memory with
the 16x256b shape (PTX ISA, tcgen05 matrix fragments: thread t receives, for
each 8-column repeat, lane t/4 and lane t/4 + 8 at columns 2 (t%4) and
2 (t%4) + 1), so each thread needs only BN/8 column scales per slice.  These
tests restate the kernel's index arithmetic (gemm.cuh: promote_col, the
producer's scale copies, GemmSmem) and check that

* the producer's 8-byte copies place every column scale exactly once, where
  the thread that multiplies that column reads it, and the 4 runs a warp reads
  together sit in different banks;
* the accumulator registers of a warp cover its 32 rows x BN/2 columns once;
* each epilogue pass writes every element of its TMA box once, at the
  position of the 64-byte swizzled image, without bank conflicts;
* the shared-memory carve-up is aligned and fits.
"""

import numpy as np
import pytest

from test_quant_smem_layout import wavefronts


def smem(bn, pair):
    """GemmSmem<BN, kPair, kCol = true>, restated."""
    stages = 6 if pair else (4 if bn == 256 else 6)
    a_bytes = 128 * 128
    b_bytes = (bn // 2 if pair else bn) * 128
    b_off = stages * a_bytes
    c_off = b_off + stages * b_bytes
    c_warp = 2048
    slots = stages + 2
    sb_stride = bn // 8 + 4
    slot_floats = 128 + 8 * sb_stride
    scale_off = c_off + 8 * c_warp
    bar_off = scale_off + slots * slot_floats * 4
    bars = 2 * stages + 5 + 2 * slots + 1
    tmem_slot = bar_off + bars * 8
    return dict(stages=stages, a_bytes=a_bytes, b_bytes=b_bytes, b_off=b_off, c_off=c_off, c_warp=c_warp,
                slots=slots, sb_stride=sb_stride, slot_floats=slot_floats, scale_off=scale_off, bar_off=bar_off,
                tmem_slot=tmem_slot, alloc=tmem_slot + 16 + 1024)


def producer_sb_dst(bn, lane, r):
    """(destination float index within the slot's sb region, tile column) of
    the producer's copy r of lane `lane` (two columns per copy)."""
    half_cols = bn // 2
    col = 2 * (32 * r + lane)
    cc = col % half_cols
    dst = ((col // half_cols) * 4 + (cc % 8) // 2) * smem(bn, False)["sb_stride"] + 2 * (cc // 8)
    return dst, col


def thread_columns(bn, warp, lane):
    """Tile columns whose scales thread (warp, lane) reads, in the order of its
    float4 loads (group j = 8 ch + jj, element e)."""
    half = warp >> 2
    tq = lane & 3
    kj = bn // 16
    return [half * (bn // 2) + 8 * j + 2 * tq + e for j in range(kj) for e in range(2)]


@pytest.mark.parametrize("bn", [256, 128])
def test_producer_puts_each_column_scale_where_its_thread_reads_it(bn):
    g = smem(bn, False)
    where = {}
    for lane in range(32):
        for r in range(bn // 64):
            dst, col = producer_sb_dst(bn, lane, r)
            assert dst % 2 == 0 and col % 2 == 0            # 8-byte cp.async: both ends 8-byte aligned
            for e in range(2):
                assert dst + e not in where
                where[dst + e] = col + e
    assert sorted(where.values()) == list(range(bn))
    assert max(where) < 8 * g["sb_stride"]
    for warp in range(8):
        for lane in range(32):
            run = ((warp >> 2) * 4 + (lane & 3)) * g["sb_stride"]
            assert (run * 4) % 16 == 0                          # float4 loads
            got = [where[run + k] for k in range(bn // 8)]
            assert got == thread_columns(bn, warp, lane)


@pytest.mark.parametrize("bn", [256, 128])
def test_column_scale_loads_are_conflict_free(bn):
    g = smem(bn, False)
    for warp in range(8):
        for k in range(bn // 32):  # the thread's float4 loads
            addrs = [4 * (128 + ((warp >> 2) * 4 + (lane & 3)) * g["sb_stride"] + 4 * k) for lane in range(32)]
            # 4 distinct 16-byte pieces, each read by 8 lanes: one wavefront per 8-lane phase
            assert wavefronts(addrs, 16) == 4, (warp, k)
    # without the 4-float padding every run starts in the same bank
    addrs = [4 * (128 + (lane & 3) * (bn // 8)) for lane in range(32)]
    assert wavefronts(addrs, 16) > 4


def acc_cell(bn, lane, idx):
    """(row within the warp's 32, column within its BN/2) of acc[idx]."""
    chunks = bn // 128
    blk, w = divmod(idx, 32)
    h, ch = divmod(blk, chunks)
    jj, rem = divmod(w, 4)
    i, e = divmod(rem, 2)
    return 16 * h + 8 * i + (lane >> 2), 8 * (8 * ch + jj) + 2 * (lane & 3) + e


@pytest.mark.parametrize("bn", [256, 128])
def test_accumulators_cover_the_warp_tile_once(bn):
    seen = np.zeros((32, bn // 2), np.int32)
    for lane in range(32):
        for idx in range(bn // 2):  # 8 kJ = BN/2 accumulators per thread
            r, c = acc_cell(bn, lane, idx)
            seen[r, c] += 1
    assert np.all(seen == 1)
    # a 16x256b.x8 load of lanes 16h.. at column 64 ch lands in acc[32 (h chunks + ch) ..]:
    # register 4 jj + 2 i + e is TMEM lane 16h + 8i + t/4, column 64 ch + 8 jj + 2 (t%4) + e
    for lane in range(32):
        for h in range(2):
            for ch in range(bn // 128):
                for reg in range(32):
                    jj, rem = divmod(reg, 4)
                    i, e = divmod(rem, 2)
                    assert acc_cell(bn, lane, 32 * (h * (bn // 128) + ch) + reg) == (
                        16 * h + 8 * i + (lane >> 2), 64 * ch + 8 * jj + 2 * (lane & 3) + e)


def swizzle64(r, byte):
    """TMA 64-byte swizzle of a box with 64-byte rows (base 512-byte aligned):
    16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)."""
    return r * 64 + (((byte // 16) ^ ((r >> 1) & 3)) * 16) + byte % 16


def epilogue_pass_stores(bn, acc_kind, ps, lane):
    """[(smem offset in the warp's staging, element size, row, column of the warp tile)]
    of one thread in pass ps, restated from promote_col."""
    tq, tr = lane & 3, lane >> 2
    pass_cols = 16 if acc_kind else 32
    out = []
    for h in range(2):
        for i in range(2):
            r = 16 * h + 8 * i + tr
            sw = (r >> 1) & 3
            for g in range(pass_cols // 8):
                col = ps * pass_cols + 8 * g + 2 * tq
                if acc_kind:
                    gg = g ^ ((lane >> 3) & 1)  # lanes with row bit 1 set store the other group first
                    col = ps * pass_cols + 8 * gg + 2 * tq
                    chunk = 2 * gg + (tq >> 1)
                    out.append((r * 64 + ((chunk ^ sw) << 4) + 8 * (tq & 1), 8, r, col))
                else:
                    out.append((r * 64 + ((g ^ sw) << 4) + 4 * tq, 4, r, col))
    return out


@pytest.mark.parametrize("acc_kind", [False, True])
@pytest.mark.parametrize("bn", [256, 128])
def test_epilogue_passes_fill_their_box_once_conflict_free(bn, acc_kind):
    esize = 4 if acc_kind else 2
    pass_cols = 16 if acc_kind else 32
    for ps in range((bn // 2) // pass_cols):
        image = {}
        per_store = {}
        for lane in range(32):
            for k, (off, size, r, col) in enumerate(epilogue_pass_stores(bn, acc_kind, ps, lane)):
                assert 0 <= off and off + size <= 2048 and off % size == 0
                per_store.setdefault(k, []).append(off)
                for e in range(2):  # two consecutive columns per store
                    byte = off + e * esize
                    assert byte not in image
                    image[byte] = (r, col + e)
        # every element of the 32 x pass_cols box, where the 64-byte swizzle puts it
        assert len(image) == 32 * pass_cols
        for byte, (r, col) in image.items():
            c = col - ps * pass_cols
            assert swizzle64(r, c * esize) == byte
        for k, addrs in per_store.items():
            size = 8 if acc_kind else 4
            assert wavefronts(addrs, size) == (2 if acc_kind else 1), (ps, k)


@pytest.mark.parametrize("bn,pair", [(256, False), (128, False), (256, True)])
def test_col_layout_shared_memory_is_aligned_and_fits(bn, pair):
    g = smem(bn, pair)
    for s in range(g["stages"]):
        assert (s * g["a_bytes"]) % 1024 == 0 and (g["b_off"] + s * g["b_bytes"]) % 1024 == 0
    assert g["c_off"] % 1024 == 0 and g["c_warp"] % 512 == 0   # 64-byte swizzle atoms: 512 bytes
    assert g["scale_off"] % 16 == 0 and (g["slot_floats"] * 4) % 16 == 0
    assert g["slots"] >= g["stages"] + 2
    assert g["bar_off"] % 8 == 0
    assert g["alloc"] <= 232448
    # each 32 x 32 bf16 or 32 x 16 fp32 box is one 2 KB staging area
    assert 32 * 32 * 2 == g["c_warp"] == 32 * 16 * 4
