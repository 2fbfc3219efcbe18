// E4M3 quantisers: 1x128 activation groups (along the columns, and along
// the rows with transposed storage) and 128x128 weight blocks.
//
// Numerics follow "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within
// $5090", section 3.2: one scale per 128 consecutive values along the GEMM
// reduction dimension for activations and activation gradients, one per
// 128x128 block for weights, each computed online from its own values.
// Per group: amax = max|x| (NaN ignored); s = amax/448 in IEEE fp32 (1 when
// amax == 0); q = E4M3_rn_satfinite(fp32_rn(x / s)).  The quotient is formed
// exactly by an FMA correction step (GroupScale), so codes and scales match a
// plain CPU evaluation bit for bit.  Two other scale modes share the kernel:
// power-of-two scales (s = the smallest 2^k >= amax/448, codes from the exact
// product x * 2^-k) and the reciprocal multiply (s = amax/448 stored, codes
// E4M3(fp32_rn(x * fp32_rn(448/amax)))): both form each code from one product.
//
// Work decomposition.  The input is cut into 128x128 bf16 tiles (32 KB),
// walked in row-major order by a persistent grid (two CTAs per SM).  A CTA
// streams its tiles through a 3-deep shared-memory ring filled by TMA; its
// eight warps share each tile without any block-wide barrier (warp 0 also
// refills a slot once every warp has released it).  Warp w owns
//   * 16 rows of the tile (their 1x128 groups along the columns: q, s):
//     lane pair (2j, 2j+1) holds one row, 64 values each, as the 16-code
//     output chunks 2m+h (h = lane & 1), and
//   * columns 16w..16w+15 (their groups of 128 rows: qT, sT): each lane holds
//     4 columns over 16 consecutive rows.
// It codes the row slice first and then the column slice, holding one of
// them in registers at a time, and releases the ring slot as soon as the
// last slice it needs is in registers.  For each slice it reduces amaxes
// with in-lane packed bf16 maxima and a few shuffles, turns each amax into
// its scale and reciprocal once, forms every code from the correctly
// rounded quotient (GroupScale, written on -x so that zeros keep their
// sign), and stores codes straight to global memory in 32-byte (rows) and
// 128-byte (columns) segments.  The input is read from HBM once whichever
// outputs are requested.
//
// Shared-memory image of a tile.  The input is addressed by TMA as the 2-D
// tensor [R/16, 16 C]: its row y holds rows 16y..16y+15 of the input side by
// side, so a 64-column x 8-row box at x = l C + c0 + 64h, y = r0/16 fetches
// rows r0 + l, r0 + 16 + l, ..., r0 + 112 + l.  Thirty-two such boxes
// (l = 0..15, h = 0..1), 128-byte swizzled, place element (r, c) of the tile,
// r = 16 a + l, c = 64 h + 8 k + e, at byte
//   16384 h + 1024 l + 128 a + 16 (k XOR a) + 2 e.
// Rows 16 apart therefore sit in different swizzle phases, and the lane
// assignments below make both register views conflict-free: a quarter-warp
// of 16-byte row reads covers rows of four distinct a (0,1,4,5 or 2,3,6,7),
// and a half-warp of 8-byte column reads covers row blocks of one parity.
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace bfp8 {

struct QuantParams {
  const uint16_t* x;  // bf16 [R, C]; for the SiLU-gated prologue [R, 2C] = [g || u]
  int64_t R, C;       // the quantised tensor (h for the prologue)
  uint8_t* q;   // [R, C] or null
  float* s;     // act: [C/128, R];  weight: [R/128, C/128]
  uint8_t* qT;  // [C, R] or null
  float* sT;    // act: [R/128, C];  unused for weights
  uint64_t wait_ns;
  uint32_t ctiles, tiles;  // C/128 and (R/128)(C/128), filled in by the launcher
  uint16_t* h;             // prologue only: bf16 [R, C] copy of h, or null
  uint32_t stall;          // test hook: warp 0 first waits on a barrier nothing completes
};

// Which outputs a kernel instance writes (a template bit set).
constexpr int kQRows = 1;  // q, s: groups along the columns (or the block, rows view)
constexpr int kQCols = 2;  // qT (, sT): groups along the rows, stored transposed

constexpr int kQComputeWarps = 8;
constexpr int kQuantThreads = 32 * kQComputeWarps;
constexpr int kQStages = 3;
constexpr int kQTileBytes = 128 * 256;  // bf16 tile

// Shared memory: the ring (one tile per slot, or the g and u tiles of the
// SiLU-gated prologue), then full[3], empty[3], redbar[2], stall and
// float[2][8] (weight block amax), plus room to align the base to 1024.
template <bool kGlu>
struct QuantLayout {
  static constexpr int kSlot = (kGlu ? 2 : 1) * kQTileBytes;
  static constexpr int kBarOff = kQStages * kSlot;
  static constexpr int kRedOff = kBarOff + (2 * kQStages + 3) * 8;
  static constexpr int kSmemBytes = kRedOff + 2 * kQComputeWarps * 4 + 1024;
};
constexpr int kQuantSmemBytes = QuantLayout<false>::kSmemBytes;
constexpr int kQuantGluSmemBytes = QuantLayout<true>::kSmemBytes;

// Tile coordinates of a persistent CTA's walk (tile t = rt * ctiles + ct).
struct TileWalk {
  uint32_t t, rt, ct;
  __device__ __forceinline__ void advance(uint32_t step, uint32_t drt, uint32_t dct, uint32_t ctiles) {
    t += step;
    rt += drt;
    ct += dct;
    if (ct >= ctiles) {
      ct -= ctiles;
      ++rt;
    }
  }
};

__device__ __forceinline__ float bf16x2_absmax(uint32_t w) { return fmaxf(fabsf(bf16lo(w)), fabsf(bf16hi(w))); }

// max(|a|, |b|) per bf16 half (NaN ignored); the sign bits of the result are
// meaningless and are dropped when the halves are widened.
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The 16 values of one group slice as a warp lane holds them.  Row slices:
// value 2i + h is half h of word i.  Column slices: value k (row k) is half
// kHalf of word kWord of the 8-byte chunk v[k].  neg(i) is -x_i and pos(i)
// is x_i, widened to fp32 straight from the word that holds them.
struct RowSlice {
  const uint32_t (&w)[8];
  __device__ __forceinline__ float neg(int i) const { return (i & 1) ? neg_bf16hi(w[i >> 1]) : neg_bf16lo(w[i >> 1]); }
  __device__ __forceinline__ float pos(int i) const { return (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]); }
};
template <int kWord, int kHalf>
struct ColSlice {
  const uint2 (&v)[16];
  __device__ __forceinline__ uint32_t word(int k) const { return kWord ? v[k].y : v[k].x; }
  __device__ __forceinline__ float neg(int k) const { return kHalf ? neg_bf16hi(word(k)) : neg_bf16lo(word(k)); }
  __device__ __forceinline__ float pos(int k) const { return kHalf ? bf16hi(word(k)) : bf16lo(word(k)); }
};

// 16 codes (byte i = value i) of a slice whose group scale g is on the fast
// path: the correction step on -x (amax/448 mode) or one product with the
// group multiplier (the other modes; exact for power-of-two scales).
template <int kScale, class Slice>
__device__ __forceinline__ uint4 codes16_fast(const Slice& v, const GroupScale& g) {
  uint32_t c[4];
  if constexpr (kScale == kScaleAmax448) {
    const float2 nr2 = make_float2(-g.r, -g.r), s2 = make_float2(g.s, g.s);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = quotient_pair_neg(make_float2(v.neg(4 * i), v.neg(4 * i + 1)), nr2, s2);
      const float2 b = quotient_pair_neg(make_float2(v.neg(4 * i + 2), v.neg(4 * i + 3)), nr2, s2);
      c[i] = e4m3x4(a.x, a.y, b.x, b.y);
    }
  } else {
    const float2 r2 = make_float2(g.r, g.r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = fmul2(make_float2(v.pos(4 * i), v.pos(4 * i + 1)), r2);
      const float2 b = fmul2(make_float2(v.pos(4 * i + 2), v.pos(4 * i + 3)), r2);
      c[i] = e4m3x4(a.x, a.y, b.x, b.y);
    }
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// The same for any group: groups off the fast path (extreme or infinite
// scales) take the power-of-two pre-scaling and two correction steps.
template <int kScale, class Slice>
__device__ __forceinline__ uint4 codes16(const Slice& v, const GroupScale& g) {
  if (g.exact) return codes16_fast<kScale>(v, g);
  const ScaledGroup sg = scaled_group(g.s);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = quotient_pair_scaled(make_float2(v.neg(4 * i), v.neg(4 * i + 1)), sg);
    const float2 b = quotient_pair_scaled(make_float2(v.neg(4 * i + 2), v.neg(4 * i + 3)), sg);
    c[i] = e4m3x4(a.x, a.y, b.x, b.y);
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// 16 codes of the 16 consecutive values in (a, b) (8 bf16 each), one group.
template <bool kFast, int kScale>
__device__ __forceinline__ uint4 quant16(const uint4& a, const uint4& b, const GroupScale& g) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const RowSlice v{w};
  return kFast ? codes16_fast<kScale>(v, g) : codes16<kScale>(v, g);
}

// 16 codes of one column over 16 rows, one group.  Codes in row order.
template <int kWord, int kHalf, bool kFast, int kScale>
__device__ __forceinline__ uint4 quant_col16(const uint2 (&cv)[16], const GroupScale& g) {
  const ColSlice<kWord, kHalf> v{cv};
  return kFast ? codes16_fast<kScale>(v, g) : codes16<kScale>(v, g);
}

// Warp 0 fetches tile (rt, ct) into ring slot `buf` with 32 TMA boxes (one
// per lane; lane 0 arms the slot's barrier first).  xrow is the input's row
// length.  The SiLU-gated prologue also fetches the u tile, uoff columns to
// the right, into the slot's second half.
template <bool kGlu>
__device__ __forceinline__ void quant_fill(const CUtensorMap* tmx, uint32_t xrow, uint32_t uoff, uint32_t rt,
                                           uint32_t ct, uint8_t* buf, uint64_t* bar, int lane) {
  if (lane == 0) mbar_arrive_expect_tx(bar, QuantLayout<kGlu>::kSlot);
  __syncwarp();
  const int l = lane >> 1, h = lane & 1;
  const int32_t x0 = static_cast<int32_t>(l * xrow + ct * 128 + 64 * h);
  tma_load_2d(buf + 16384 * h + 1024 * l, tmx, x0, static_cast<int32_t>(rt * 8), bar);
  if constexpr (kGlu)
    tma_load_2d(buf + kQTileBytes + 16384 * h + 1024 * l, tmx, x0 + static_cast<int32_t>(uoff),
                static_cast<int32_t>(rt * 8), bar);
}

// Codes of this lane's row slice (4 chunks of 16) under the row group scale.
template <bool kFast, int kScale>
__device__ __forceinline__ void quant_row_codes(const uint4 (&rv)[8], const GroupScale& g, uint8_t* qrow) {
#pragma unroll
  for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4*>(qrow + 32 * m) = quant16<kFast, kScale>(rv[2 * m], rv[2 * m + 1], g);
}

// Codes of this lane's 4 columns over its 16 rows (gc: their group scales),
// column k to qcol + k R.
template <bool kFast, int kScale>
__device__ __forceinline__ void quant_col_codes(const uint2 (&cv)[16], const GroupScale (&gc)[4], uint8_t* qcol,
                                                int64_t R) {
  *reinterpret_cast<uint4*>(qcol) = quant_col16<0, 0, kFast, kScale>(cv, gc[0]);
  *reinterpret_cast<uint4*>(qcol + R) = quant_col16<0, 1, kFast, kScale>(cv, gc[1]);
  *reinterpret_cast<uint4*>(qcol + 2 * R) = quant_col16<1, 0, kFast, kScale>(cv, gc[2]);
  *reinterpret_cast<uint4*>(qcol + 3 * R) = quant_col16<1, 1, kFast, kScale>(cv, gc[3]);
}

// kWeight = false: activation groups (rows -> q/s, columns -> qT/sT).
// kWeight = true : one 128x128 block per tile (q and/or qT, one scale).
// kScale: the scale mode (kScaleAmax448, kScalePow2 or kScaleMulRecip).
// kGlu: the input is the gate+up output [g || u] and the quantised tensor is
// h = bf16_rn(SiLU(g) u) (the down projection's activation).  Each warp forms
// h for its 16 rows, writes it over g in the slot (and to p.h if given), and
// the column view reads h once every warp's rows are in place (redbar, all
// 256 threads arriving).  One CTA per SM: a slot holds two tiles.
template <bool kWeight, int kMode, int kScale, bool kGlu>
__global__ void __launch_bounds__(kQuantThreads, kGlu ? 1 : 2)
    quantize_tile_kernel(const __grid_constant__ CUtensorMap tmx, const QuantParams p) {
  static_assert(!(kGlu && kWeight), "the SiLU-gated prologue quantises an activation");
  static_assert(kScale != kScaleMx32 || (!kWeight && !kGlu), "the 1x32 recipe has no 2-D blocks or prologue");
  using L = QuantLayout<kGlu>;
  constexpr bool kRows = (kMode & kQRows) != 0, kCols = (kMode & kQCols) != 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kQStages;
  uint64_t* redbar = empty + kQStages;  // weight block amax / prologue h exchange, by tile parity
  uint64_t* stall = redbar + 2;         // never completed (test hook p.stall)
  float* red = reinterpret_cast<float*>(smem + L::kRedOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ctiles = p.ctiles, tiles = p.tiles, C = static_cast<uint32_t>(p.C);
  const uint32_t xrow = kGlu ? 2u * C : C;  // input row length
  const uint32_t step = gridDim.x, drt = step / ctiles, dct = step % ctiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQComputeWarps);
    }
    mbar_init(&redbar[0], kGlu ? kQuantThreads : kQComputeWarps);
    mbar_init(&redbar[1], kGlu ? kQuantThreads : kQComputeWarps);
    mbar_init(stall, 1);
    fence_mbar_init();
  }
  __syncthreads();

  TileWalk cur{blockIdx.x, blockIdx.x / ctiles, blockIdx.x % ctiles};
  // Warp 0 issues the first kQStages tiles of this CTA, and later (at
  // iteration j) tile j-1+kQStages into the slot tile j-1 used.
  TileWalk fill = cur;
  uint32_t issued = 0;  // tiles of this CTA issued so far (warp 0)
  // Test hook: a wait that nothing satisfies, so that it expires after the
  // wait limit; warp 0 then issues no copy and every warp's first wait on a
  // tile expires too, so the kernel ends with nothing in flight.
  const bool stalled = p.stall != 0u && warp == 0 && !mbar_wait(stall, 0, p.wait_ns, kWeight ? 0x200u : 0x100u);
  if (warp == 0 && !stalled) {
    for (; issued < kQStages && fill.t < tiles; ++issued) {
      quant_fill<kGlu>(&tmx, xrow, C, fill.rt, fill.ct, smem + issued * L::kSlot, &full[issued], lane);
      fill.advance(step, drt, dct, ctiles);
    }
  }

  // Row view: lane pair (2j, 2j+1) holds tile row 16 a + l with
  // a = j%8 with its bits 1 and 2 swapped, l = 2w + j/8; lane h = lane & 1
  // reads 16-byte chunks 4m + 2h + u (u = 0, 1) of it.
  const int jj = lane >> 1, hh = lane & 1;
  const int ra = (jj & 1) | (((jj >> 2) & 1) << 1) | (((jj >> 1) & 1) << 2);
  const int wrow = 16 * ra + 2 * warp + (jj >> 3);
  // chunk 2h of the row; chunk 4(m%2) + 2h + u differs from it in the bits
  // 4(m%2) + u of the 16-byte index, which the swizzle XOR leaves alone
  const uint32_t roff = 1024u * (2 * warp + (jj >> 3)) + 128u * ra + ((static_cast<uint32_t>(2 * hh) ^ ra) << 4);
  // Column view: lane (cq, g) holds columns 16w + 4cq..+3 over rows
  // 16 rg..16 rg + 15, rg = 2 (g % 4) + g / 4.
  const int cq = lane & 3, g = lane >> 2, rg = 2 * (g & 3) + (g >> 2);
  const uint32_t coff = 16384u * (warp >> 2) + 128u * rg +
                        ((static_cast<uint32_t>(2 * (warp & 3) + (cq >> 1)) ^ rg) << 4) + 8u * (cq & 1);

  uint32_t j = 0;
  for (; cur.t < tiles; cur.advance(step, drt, dct, ctiles), ++j) {
    const uint32_t s = j % kQStages, ph = (j / kQStages) & 1u;
    if (!mbar_wait(&full[s], ph, p.wait_ns, kWeight ? 0x201u : 0x101u)) break;
    uint8_t* buf = smem + s * L::kSlot;
    const int64_t r0 = static_cast<int64_t>(cur.rt) * 128, c0 = static_cast<int64_t>(cur.ct) * 128;

    // The row view is coded before the column view is read, so that only
    // one slice of the tile is held in registers at a time; the slot is
    // handed back once the last slice this warp needs is in registers.
    uint4 rv[8];
    if constexpr (kRows || kGlu) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        rv[2 * m] = *reinterpret_cast<const uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1))));
        rv[2 * m + 1] = *reinterpret_cast<const uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1) + 16u)));
      }
    }
    if constexpr (kGlu) {
      // h for this warp's rows: the u row slice sits at the same offsets in
      // the slot's second half.  The exponent path is chosen per warp: the
      // wide one only when some |g| of the slice exceeds 64.
      uint4 ru[8];
      uint32_t gm2 = 0u;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint8_t* ub = buf + kQTileBytes + 16384 * (m >> 1);
        ru[2 * m] = *reinterpret_cast<const uint4*>(ub + (roff ^ (64u * (m & 1))));
        ru[2 * m + 1] = *reinterpret_cast<const uint4*>(ub + (roff ^ (64u * (m & 1) + 16u)));
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        gm2 = bf16x2_maxabs(bf16x2_maxabs(gm2, bf16x2_maxabs(rv[k].x, rv[k].y)), bf16x2_maxabs(rv[k].z, rv[k].w));
      if (__any_sync(0xffffffffu, !(bf16x2_absmax(gm2) <= 64.0f))) {
#pragma unroll
        for (int k = 0; k < 8; ++k) rv[k] = swiglu_bf16x8<true>(rv[k], ru[k]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) rv[k] = swiglu_bf16x8<false>(rv[k], ru[k]);
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        *reinterpret_cast<uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1)))) = rv[2 * m];
        *reinterpret_cast<uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1) + 16u))) = rv[2 * m + 1];
      }
      if (p.h != nullptr) {
        // chunks 4m + 2h + u of the row: columns 32m + 16h + 8u
        uint16_t* hrow = p.h + (static_cast<int64_t>(r0) + wrow) * p.C + c0 + 16 * hh;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          *reinterpret_cast<uint4*>(hrow + 32 * m) = rv[2 * m];
          *reinterpret_cast<uint4*>(hrow + 32 * m + 8) = rv[2 * m + 1];
        }
      }
      // The slot is refilled by TMA after every warp releases it: order these
      // generic-proxy writes before that async-proxy write, and release them
      // to the other warps (each thread arrives for its own writes).
      fence_proxy_async_smem();
      mbar_arrive(&redbar[j & 1u]);
      if (!mbar_wait(&redbar[j & 1u], (j >> 1) & 1u, p.wait_ns, 0x131u)) break;
    }

    // Hands the slot back (every lane's reads of it are done) and lets warp 0
    // refill the slot of tile j-1 (every warp released it, usually long ago)
    // with tile j-1+kQStages.  False if that wait expired.
    auto release = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (warp == 0 && j >= 1 && fill.t < tiles) {
        const uint32_t f = j - 1, sf = f % kQStages;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[sf], (f / kQStages) & 1u, p.wait_ns, kWeight ? 0x211u : 0x111u);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        quant_fill<kGlu>(&tmx, xrow, C, fill.rt, fill.ct, smem + sf * L::kSlot, &full[sf], lane);
        fill.advance(step, drt, dct, ctiles);
        ++issued;
      }
      return true;
    };
    auto load_cols = [&](uint2 (&cv)[16]) {
#pragma unroll
      for (int k = 0; k < 16; ++k) cv[k] = *reinterpret_cast<const uint2*>(buf + coff + 1024 * k);
    };
    if constexpr (!kCols) {
      if (!release()) break;
    }

    if constexpr (kScale == kScaleMx32) {
      // MXFP8 1x32 groups.  Row view: 32-group m of a row is columns
      // 32m .. 32m + 31, whose halves 16h .. 16h + 15 sit in the two lanes of
      // the row's lane pair.  Column view: a column's 32-row group k (rows
      // 32k ..) sits in lanes (cq, k) and (cq, k + 4), 16 lanes apart.
      if constexpr (kRows) {
        uint8_t* qrow = p.q + (r0 + wrow) * p.C + c0 + 16 * hh;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint4 a = rv[2 * m], b = rv[2 * m + 1];
          const uint32_t m2 = bf16x2_maxabs(bf16x2_maxabs(bf16x2_maxabs(a.x, a.y), bf16x2_maxabs(a.z, a.w)),
                                            bf16x2_maxabs(bf16x2_maxabs(b.x, b.y), bf16x2_maxabs(b.z, b.w)));
          float am = bf16x2_absmax(m2);
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
          const GroupScale gs = make_group_scale_mx(am);
          if (hh == (m & 1)) p.s[(static_cast<int64_t>(cur.ct) * 4 + m) * p.R + r0 + wrow] = gs.s;
          *reinterpret_cast<uint4*>(qrow + 32 * m) = quant16<true, kScaleMx32>(a, b, gs);
        }
      }
      if constexpr (kCols) {
        uint2 cv[16];
        load_cols(cv);
        if (!release()) break;
        uint32_t c01 = 0u, c23 = 0u;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          c01 = bf16x2_maxabs(c01, cv[k].x);
          c23 = bf16x2_maxabs(c23, cv[k].y);
        }
        c01 = bf16x2_maxabs(c01, __shfl_xor_sync(0xffffffffu, c01, 16));
        c23 = bf16x2_maxabs(c23, __shfl_xor_sync(0xffffffffu, c23, 16));
        const GroupScale gs[4] = {make_group_scale_mx(fabsf(bf16lo(c01))), make_group_scale_mx(fabsf(bf16hi(c01))),
                                  make_group_scale_mx(fabsf(bf16lo(c23))), make_group_scale_mx(fabsf(bf16hi(c23)))};
        if (g < 4)  // the 4 scales of this lane's columns for 32-group g of the tile's rows
          *reinterpret_cast<float4*>(p.sT + (static_cast<int64_t>(cur.rt) * 4 + g) * p.C + c0 + 16 * warp + 4 * cq) =
              make_float4(gs[0].s, gs[1].s, gs[2].s, gs[3].s);
        quant_col_codes<true, kScaleMx32>(cv, gs, p.qT + (c0 + 16 * warp + 4 * cq) * p.R + r0 + 16 * rg, p.R);
      }
      continue;
    }

    // Block maximum of a weight tile: every warp's maximum meets in shared
    // memory.  Slot j%2 is reused two tiles later, when every warp has read
    // it (a warp arrives for tile j+1 only after reading slot j%2).
    auto block_max = [&](float m, bool& ok) -> float {
      m = warp_max(m);
      float* rbuf = red + (j & 1u) * kQComputeWarps;
      if (lane == 0) {
        rbuf[warp] = m;
        mbar_arrive(&redbar[j & 1u]);
      }
      ok = mbar_wait(&redbar[j & 1u], (j >> 1) & 1u, p.wait_ns, 0x221u);
      float bm = rbuf[0];
#pragma unroll
      for (int k = 1; k < kQComputeWarps; ++k) bm = fmaxf(bm, rbuf[k]);
      return bm;
    };

    GroupScale grow;  // the row group's scale (weights: the block's)
    if constexpr (kRows) {
      uint32_t m2 = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        m2 = bf16x2_maxabs(bf16x2_maxabs(m2, bf16x2_maxabs(rv[k].x, rv[k].y)), bf16x2_maxabs(rv[k].z, rv[k].w));
      float row_m = bf16x2_absmax(m2);
      row_m = fmaxf(row_m, __shfl_xor_sync(0xffffffffu, row_m, 1));
      bool fast;
      if constexpr (kWeight) {
        bool ok;
        grow = make_scale<kScale>(block_max(row_m, ok));
        if (!ok) break;
        if (threadIdx.x == 0) p.s[cur.rt * static_cast<int64_t>(ctiles) + cur.ct] = grow.s;
        fast = grow.exact;  // uniform over the block
      } else {
        grow = make_scale<kScale>(row_m);
        if (hh == 0) p.s[static_cast<int64_t>(cur.ct) * p.R + r0 + wrow] = grow.s;
        fast = kScale == kScaleMulRecip || __all_sync(0xffffffffu, grow.exact);  // no slow path for the multiplier
      }
      uint8_t* qrow = p.q + (r0 + wrow) * p.C + c0 + 16 * hh;
      if (fast)
        quant_row_codes<true, kScale>(rv, grow, qrow);
      else
        quant_row_codes<false, kScale>(rv, grow, qrow);
    }

    if constexpr (kCols) {
      uint2 cv[16];
      load_cols(cv);
      if (!release()) break;
      uint32_t m01 = 0u, m23 = 0u;
      if (!(kWeight && kRows)) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          m01 = bf16x2_maxabs(m01, cv[k].x);
          m23 = bf16x2_maxabs(m23, cv[k].y);
        }
      }
      GroupScale gc[4];  // the groups of this lane's 4 columns
      bool fast;
      if constexpr (kWeight) {
        if constexpr (!kRows) {
          bool ok;
          grow = make_scale<kScale>(block_max(fmaxf(bf16x2_absmax(m01), bf16x2_absmax(m23)), ok));
          if (!ok) break;
          if (threadIdx.x == 0) p.s[cur.rt * static_cast<int64_t>(ctiles) + cur.ct] = grow.s;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) gc[k] = grow;
        fast = grow.exact;
      } else {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          m01 = bf16x2_maxabs(m01, __shfl_xor_sync(0xffffffffu, m01, o));
          m23 = bf16x2_maxabs(m23, __shfl_xor_sync(0xffffffffu, m23, o));
        }
        // lane (cq, g) forms the scale of column 4cq + g%4; lanes cq + 4k
        // hold those of this lane's columns
        const int sel = g & 3;
        const uint32_t mw = sel < 2 ? m01 : m23;
        const GroupScale gcol = make_scale<kScale>(fabsf((sel & 1) ? bf16hi(mw) : bf16lo(mw)));
        if (g < 4) p.sT[static_cast<int64_t>(cur.rt) * p.C + c0 + 16 * warp + 4 * cq + g] = gcol.s;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          gc[k].s = __shfl_sync(0xffffffffu, gcol.s, cq + 4 * k);
          gc[k].r = __shfl_sync(0xffffffffu, gcol.r, cq + 4 * k);
          gc[k].exact = scale_fast<kScale>(gc[k].s);
        }
        fast = kScale == kScaleMulRecip || __all_sync(0xffffffffu, gcol.exact);
      }
      uint8_t* qcol = p.qT + (c0 + 16 * warp + 4 * cq) * p.R + r0 + 16 * rg;
      if (fast)
        quant_col_codes<true, kScale>(cv, gc, qcol, p.R);
      else
        quant_col_codes<false, kScale>(cv, gc, qcol, p.R);
    }
  }
  // Leave no copy in flight into this CTA's shared memory: after an early
  // exit at local tile j, warp 0 (which issues every copy) waits (bounded)
  // for the tiles >= j it issued, at most kQStages of them.  No later fill
  // of those slots can have been issued (that needs every warp to release
  // the tile), so the waited phase is the one of that tile.  After a normal
  // exit j counts all tiles of the CTA and nothing is waited for.
  if (warp == 0 && lane == 0) {
    for (uint32_t k = j; k < issued; ++k)
      mbar_wait(&full[k % kQStages], (k / kQStages) & 1u, kDrainWaitNs, kWeight ? 0x212u : 0x112u);
  }
}

// ---------------------------------------------------------------------------
// Several weights in one launch.  A Transformer layer quantises four weights
// of 8-50 MB each; one launch per weight leaves a persistent grid mostly in
// its ramp-up and drain (a 2048 x 2048 weight has 256 tiles for 296 CTAs).
// This kernel walks the 128 x 128 blocks of up to kQBatch weights as one
// sequence (job 0's tiles, then job 1's, ...), each fetched through its own
// tensor map, with the weight path of quantize_tile_kernel: one block scale
// per tile, rows coded before columns.  Every job writes the same outputs
// (kMode).
constexpr int kQBatch = 4;

struct QuantJob {
  uint8_t* q;      // [R, C] (kQRows)
  uint8_t* qT;     // [C, R] (kQCols)
  float* s;        // [R/128, C/128]
  int64_t R, C;
  uint32_t ctiles;  // C/128
  uint32_t tile0;   // first tile of this job in the walk
};

struct QuantBatchParams {
  CUtensorMap tm[kQBatch];  // bf16 [R/16, 16 C] views, as make_quant_tmap builds them
  QuantJob job[kQBatch];
  uint32_t jobs, tiles;     // jobs in use; tiles of all of them
  uint64_t wait_ns;
  uint32_t stall;           // test hook, as QuantParams::stall
};

// The job, row tile and column tile of walk position t.
struct BatchTile {
  uint32_t j, rt, ct;
};
__device__ __forceinline__ BatchTile batch_tile(const QuantBatchParams& b, uint32_t t) {
  uint32_t j = 0;
#pragma unroll
  for (int k = 1; k < kQBatch; ++k)
    if (static_cast<uint32_t>(k) < b.jobs && t >= b.job[k].tile0) j = static_cast<uint32_t>(k);
  const uint32_t lt = t - b.job[j].tile0;
  return {j, lt / b.job[j].ctiles, lt % b.job[j].ctiles};
}

template <int kMode, int kScale>
__global__ void __launch_bounds__(kQuantThreads, 2) quantize_w_batch_kernel(const __grid_constant__ QuantBatchParams b) {
  using L = QuantLayout<false>;
  constexpr bool kRows = (kMode & kQRows) != 0, kCols = (kMode & kQCols) != 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kQStages;
  uint64_t* redbar = empty + kQStages;  // block amax exchange, by tile parity
  uint64_t* stall = redbar + 2;         // never completed (test hook b.stall)
  float* red = reinterpret_cast<float*>(smem + L::kRedOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tiles = b.tiles, step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQComputeWarps);
    }
    mbar_init(&redbar[0], kQComputeWarps);
    mbar_init(&redbar[1], kQComputeWarps);
    mbar_init(stall, 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Warp 0 issues the first kQStages tiles, and later (at iteration j) tile
  // j-1+kQStages into the slot tile j-1 used.
  uint32_t fill_t = blockIdx.x, issued = 0;
  auto fill = [&](uint32_t slot) {
    const BatchTile f = batch_tile(b, fill_t);
    quant_fill<false>(&b.tm[f.j], static_cast<uint32_t>(b.job[f.j].C), 0u, f.rt, f.ct, smem + slot * L::kSlot,
                      &full[slot], lane);
    fill_t += step;
    ++issued;
  };
  const bool stalled = b.stall != 0u && warp == 0 && !mbar_wait(stall, 0, b.wait_ns, 0x240u);
  if (warp == 0 && !stalled) {
    while (issued < kQStages && fill_t < tiles) fill(issued);
  }

  // lane maps as in quantize_tile_kernel
  const int jj = lane >> 1, hh = lane & 1;
  const int ra = (jj & 1) | (((jj >> 2) & 1) << 1) | (((jj >> 1) & 1) << 2);
  const int wrow = 16 * ra + 2 * warp + (jj >> 3);
  const uint32_t roff = 1024u * (2 * warp + (jj >> 3)) + 128u * ra + ((static_cast<uint32_t>(2 * hh) ^ ra) << 4);
  const int cq = lane & 3, g = lane >> 2, rg = 2 * (g & 3) + (g >> 2);
  const uint32_t coff = 16384u * (warp >> 2) + 128u * rg +
                        ((static_cast<uint32_t>(2 * (warp & 3) + (cq >> 1)) ^ rg) << 4) + 8u * (cq & 1);

  uint32_t j = 0;
  for (uint32_t t = blockIdx.x; t < tiles; t += step, ++j) {
    const uint32_t s = j % kQStages, ph = (j / kQStages) & 1u;
    if (!mbar_wait(&full[s], ph, b.wait_ns, 0x241u)) break;
    uint8_t* buf = smem + s * L::kSlot;
    const BatchTile bt = batch_tile(b, t);
    const QuantJob& job = b.job[bt.j];
    const int64_t r0 = static_cast<int64_t>(bt.rt) * 128, c0 = static_cast<int64_t>(bt.ct) * 128;

    auto release = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (warp == 0 && j >= 1 && fill_t < tiles) {
        const uint32_t f = j - 1, sf = f % kQStages;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[sf], (f / kQStages) & 1u, b.wait_ns, 0x242u);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
        fill(sf);
      }
      return true;
    };
    auto block_max = [&](float m, bool& ok) -> float {
      m = warp_max(m);
      float* rbuf = red + (j & 1u) * kQComputeWarps;
      if (lane == 0) {
        rbuf[warp] = m;
        mbar_arrive(&redbar[j & 1u]);
      }
      ok = mbar_wait(&redbar[j & 1u], (j >> 1) & 1u, b.wait_ns, 0x243u);
      float bm = rbuf[0];
#pragma unroll
      for (int k = 1; k < kQComputeWarps; ++k) bm = fmaxf(bm, rbuf[k]);
      return bm;
    };

    GroupScale gb;  // the block's scale
    if constexpr (kRows) {
      uint4 rv[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        rv[2 * m] = *reinterpret_cast<const uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1))));
        rv[2 * m + 1] = *reinterpret_cast<const uint4*>(buf + 16384 * (m >> 1) + (roff ^ (64u * (m & 1) + 16u)));
      }
      if constexpr (!kCols) {
        if (!release()) break;
      }
      uint32_t m2 = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        m2 = bf16x2_maxabs(bf16x2_maxabs(m2, bf16x2_maxabs(rv[k].x, rv[k].y)), bf16x2_maxabs(rv[k].z, rv[k].w));
      bool ok;
      gb = make_scale<kScale>(block_max(bf16x2_absmax(m2), ok));
      if (!ok) break;
      if (threadIdx.x == 0) job.s[bt.rt * static_cast<int64_t>(job.ctiles) + bt.ct] = gb.s;
      uint8_t* qrow = job.q + (r0 + wrow) * job.C + c0 + 16 * hh;
      if (gb.exact)
        quant_row_codes<true, kScale>(rv, gb, qrow);
      else
        quant_row_codes<false, kScale>(rv, gb, qrow);
    }
    if constexpr (kCols) {
      uint2 cv[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) cv[k] = *reinterpret_cast<const uint2*>(buf + coff + 1024 * k);
      if (!release()) break;
      if constexpr (!kRows) {
        uint32_t m01 = 0u, m23 = 0u;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          m01 = bf16x2_maxabs(m01, cv[k].x);
          m23 = bf16x2_maxabs(m23, cv[k].y);
        }
        bool ok;
        gb = make_scale<kScale>(block_max(fmaxf(bf16x2_absmax(m01), bf16x2_absmax(m23)), ok));
        if (!ok) break;
        if (threadIdx.x == 0) job.s[bt.rt * static_cast<int64_t>(job.ctiles) + bt.ct] = gb.s;
      }
      const GroupScale gc[4] = {gb, gb, gb, gb};
      uint8_t* qcol = job.qT + (c0 + 16 * warp + 4 * cq) * job.R + r0 + 16 * rg;
      if (gb.exact)
        quant_col_codes<true, kScale>(cv, gc, qcol, job.R);
      else
        quant_col_codes<false, kScale>(cv, gc, qcol, job.R);
    }
  }
  // No copy left in flight into shared memory (see quantize_tile_kernel).
  if (warp == 0 && lane == 0) {
    for (uint32_t k = j; k < issued; ++k)
      mbar_wait(&full[k % kQStages], (k / kQStages) & 1u, kDrainWaitNs, 0x244u);
  }
}

}  // namespace bfp8
