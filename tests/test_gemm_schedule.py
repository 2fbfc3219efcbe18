"""The GEMM's persistent work schedule, checked on the CPU.

The host planner (tile kind, split-K factor) and the kernels' unit -> tile
map are restated here from their sources and checked for every GEMM of the
Puro-2B shapes and the small test shapes, with automatic and forced splits:

* every (output tile, 128-deep slice) pair is computed by exactly one unit;
* every split owns a non-empty, in-range slice range;
* tiles stay inside the output, and consecutive units walk down a band of
  group_m m-tiles before moving to the next column of tiles (the L2 raster);
* the persistent grid's strided walk (CTA b takes units b, b + grid, ...)
  hands every unit to exactly one CTA (or CTA pair);
* the shared-memory carve-up of each kernel instance keeps its TMA tiles and
  staging 1024-byte aligned, its scale ring 16-byte aligned and its barriers
  8-byte aligned, and fits the per-CTA limit and the TMEM columns.
"""

import math

import pytest

SMS, PAIR_CLUSTERS = 148, 74  # B300: SMs, co-resident CTA-pair clusters
FPROP, DGRAD, WGRAD = 0, 1, 2


def plan(layout, M, N, K, forced=0):
    pair = layout != WGRAD and M % 256 == 0 and N % 256 == 0
    bn = 256 if N % 256 == 0 else 128
    m_tiles = M // (256 if pair else 128)
    n_tiles = N // bn
    tiles = m_tiles * n_tiles
    slots = PAIR_CLUSTERS if pair else SMS
    nk = K // 128
    best = 1
    if forced > 0:
        best = min(forced, nk)
    else:
        t_gemm = 2.0 * M * N * K / 4.0e15
        best_t = 1e30
        for s in range(1, min(nk, 16) + 1):
            units = tiles * s
            waves = math.ceil(units / slots)
            eff = units / (waves * slots)
            t = t_gemm / eff + ((s * M * N * 4 * 2 + M * N * 2) / 6.0e12 if s > 1 else 0.0)
            if t < best_t * 0.97:
                best_t, best = t, s
    kps = -(-nk // best)
    splits = -(-nk // kps)
    return dict(pair=pair, bn=bn, m_tiles=m_tiles, n_tiles=n_tiles, tiles=tiles, splits=splits, kps=kps,
                units=tiles * splits, group_m=8 if pair else 16, m_tile_rows=256 if pair else 128, nk=nk,
                grid_units=min(tiles * splits, slots))


def unit_coords(p, u):
    tile = u % p["tiles"]
    split = u // p["tiles"]
    per_group = p["group_m"] * p["n_tiles"]
    g = tile // per_group
    first_m = g * p["group_m"]
    gm = min(p["m_tiles"] - first_m, p["group_m"])
    in_g = tile - g * per_group
    m0 = (first_m + in_g % gm) * p["m_tile_rows"]
    nt = in_g // gm
    kb0 = split * p["kps"]
    kb1 = min(p["nk"], kb0 + p["kps"])
    return m0, nt, split, kb0, kb1


def gemms():
    shapes = []
    for (M, N, K) in ((16384, 4096, 2048), (16384, 2048, 2048), (16384, 12288, 2048), (16384, 2048, 6144),
                      (8192, 12288, 2048), (8192, 2048, 6144), (256, 256, 256), (512, 768, 1280),
                      (384, 640, 512), (1024, 768, 1280), (128, 128, 128)):
        shapes += [(FPROP, M, N, K), (DGRAD, M, K, N), (WGRAD, N, K, M)]
    return shapes


@pytest.mark.parametrize("forced", [0, 1, 2, 3, 5])
def test_every_tile_and_slice_is_computed_once(forced):
    for layout, M, N, K in gemms():
        p = plan(layout, M, N, K, forced)
        assert p["splits"] >= 1 and (p["splits"] - 1) * p["kps"] < p["nk"] <= p["splits"] * p["kps"]
        done = {}
        for u in range(p["units"]):
            m0, nt, split, kb0, kb1 = unit_coords(p, u)
            assert 0 <= m0 and m0 + p["m_tile_rows"] <= M and m0 % p["m_tile_rows"] == 0
            assert 0 <= nt < p["n_tiles"]
            assert 0 <= kb0 < kb1 <= p["nk"]
            for kb in range(kb0, kb1):
                key = (m0, nt, kb)
                assert key not in done, (layout, M, N, K, u, key)
                done[key] = u
        assert len(done) == p["m_tiles"] * p["n_tiles"] * p["nk"]


def test_units_walk_a_band_of_m_tiles_first():
    p = plan(FPROP, 16384, 12288, 2048)
    assert p["pair"] and p["group_m"] == 8
    first = [unit_coords(p, u) for u in range(16)]
    assert [c[0] // 256 for c in first[:8]] == list(range(8)) and all(c[1] == 0 for c in first[:8])
    assert [c[0] // 256 for c in first[8:]] == list(range(8)) and all(c[1] == 1 for c in first[8:])


@pytest.mark.parametrize("forced", [0, 3])
def test_persistent_grid_hands_out_every_unit_once(forced):
    for layout, M, N, K in gemms():
        p = plan(layout, M, N, K, forced)
        grid = p["grid_units"]  # CTAs, or CTA pairs (blockIdx.x >> 1) for the pair kernel
        owner = {}
        for b in range(grid):
            for u in range(b, p["units"], grid):
                assert u not in owner
                owner[u] = b
        assert len(owner) == p["units"]


def test_the_stack_shapes_need_no_split():
    # every GEMM of the 16384-token stack fills the GPU with whole tiles
    for layout, M, N, K in gemms()[:12]:
        assert plan(layout, M, N, K)["splits"] == 1, (layout, M, N, K)


def gemm_smem(pair, bn):
    """The GEMM's shared-memory carve-up, restated from GemmSmem."""
    stages = 4 if pair else (3 if bn == 256 else 4)
    a_bytes = 128 * 128
    b_bytes = (bn // 2 if pair else bn) * 128
    b_off = stages * a_bytes
    c_warp = 32 * (bn // 2) * 2
    c_off = b_off + stages * b_bytes
    slots, slot_floats = 8, 128 + bn
    scale_off = c_off + 8 * c_warp
    bar_off = scale_off + slots * slot_floats * 4
    bars = 2 * stages + 5 + 2 * slots + 1  # full, empty, tfull[2], tempty[2], done, sfull, sempty, stall
    tmem_slot = bar_off + bars * 8
    return dict(stages=stages, a_bytes=a_bytes, b_bytes=b_bytes, b_off=b_off, c_off=c_off, c_warp=c_warp,
                scale_off=scale_off, slot_bytes=slot_floats * 4, bar_off=bar_off, tmem_slot=tmem_slot,
                alloc=tmem_slot + 16 + 1024, tmem_cols=2 * bn)


def test_gemm_shared_memory_is_aligned_and_fits():
    for pair, bn in ((True, 256), (False, 256), (False, 128)):
        g = gemm_smem(pair, bn)
        # 128-byte-swizzled TMA tiles and the epilogue staging start on 1024-byte boundaries
        for s in range(g["stages"]):
            assert (s * g["a_bytes"]) % 1024 == 0 and (g["b_off"] + s * g["b_bytes"]) % 1024 == 0
        assert g["c_off"] % 1024 == 0 and g["c_warp"] % 1024 == 0
        # the scale ring takes 16-byte cp.async copies; barriers are 8-byte words
        assert g["scale_off"] % 16 == 0 and g["slot_bytes"] % 16 == 0
        assert g["bar_off"] % 8 == 0 and g["tmem_slot"] % 4 == 0
        assert g["alloc"] <= 232448                  # the per-CTA dynamic shared-memory limit
        assert g["tmem_cols"] <= 512 and g["tmem_cols"] & (g["tmem_cols"] - 1) == 0  # power of two, <= 512
