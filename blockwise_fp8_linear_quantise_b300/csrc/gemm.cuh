// Block-scaled E4M3 GEMM with fp32 promotion of every 128-deep slice.
//
// Computes C[i, j] = bf16( sum_kb P_kb[i, j] * sa(i, kb) * sb(j, kb) ) with
// P_kb the E4M3 x E4M3 product over the 128 reduction indices of slice kb,
// the GEMM of the Transformer linear layers in "Puro-2B: Poor Lab's
// Qwen2-1.5B Trained on RTX 5090 within $5090", section 3.2 (E4M3 operands,
// one scale per 1x128 activation group and per 128x128 weight block).
//
// The per-group scales are arbitrary fp32 values, which the tensor cores'
// own block-scale path (power-of-two or E4M3 scale factors per 16/32
// elements) cannot express, so every slice's partial product leaves the
// tensor core and is promoted in fp32 by CUDA cores:
//
//   warp 8      producer: per slice, lane 0 loads a 128x128 A tile and a
//               BNx128 B tile (both 128-byte swizzled, TMA) into a
//               STAGES-deep shared-memory ring, and all 32 lanes copy the
//               slice's scales (sa of the CTA's rows, sb) into an 8-slot
//               scale ring with cp.async, so no promotion warp ever waits on
//               a global load.
//   warp 9      MMA issuer: 4 x tcgen05.mma (K=32 each) write the slice's
//               partial P_kb into one of two TMEM buffers (BN fp32 columns
//               each); commits release the smem stage and signal the buffer.
//   warps 0..7  promotion: warp w reads TMEM lanes 32*(w%4).. (its 32 rows)
//               and columns 128*(w/4).. of the buffer, multiplies by the
//               slice's scale product (from the scale ring) and adds into
//               128 fp32 accumulators per thread held in registers, then
//               frees the buffer.  While they promote slice kb the tensor
//               core already computes kb+1.  At the end of a tile the
//               epilogue (EpiKind) converts to bf16 and hands the tile to TMA
//               stores through shared memory, adds it into an fp32 output by
//               TMA reduce-add stores, or (E4M3 codes, split-K partials)
//               stores directly.
//
// The kernel is persistent: one CTA (or CTA pair, 256 x 256 tiles with
// tcgen05 cta_group::2 MMAs) per SM walks work units (tile, split) in a
// grouped order that keeps a band of A rows and B rows hot in L2.
// With split-K, each split writes fp32 partial sums to a workspace and a
// separate kernel adds them in a fixed order (deterministic).
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace bfp8 {

// What the epilogue writes.
enum EpiKind : int {
  kEpiPlain = 0,  // bf16 C by TMA stores (or fp32 split-K partials)
  kEpiCodes = 1,  // bf16 C and its E4M3 codes (one split, BN = 256), direct stores
  kEpiAccum = 2   // C_f32 += result by TMA reduce-add stores (or fp32 split-K partials)
};

enum SbMode : int {
  kSbBlock = 0,   // sb [N/128, K/128]: FPROP weight blocks
  kSbBlockT = 1,  // sb [K/128, N/128]: DGRAD weight blocks (transposed use)
  kSbCol = 2      // sb [K/128, N]:     WGRAD per-column token groups
};

struct GemmParams {
  int M, N, K;
  int m_tiles, n_tiles, tiles;  // tiles = m_tiles * n_tiles
  int splits, kps;              // split-K count and slices per split
  int units;                    // tiles * splits
  int group_m;                  // tile rasterisation band height (in m tiles)
  int m_tile_rows;              // rows per m tile: 128, or 256 for a CTA pair
  const float* sa;              // [K/128, M]
  const float* sb;              // see SbMode
  uint16_t* C;                  // bf16 [M, N] (splits == 1)
  float* Cpart;                 // fp32 [splits, M, N] (splits > 1)
  uint8_t* Cq;                  // optional E4M3 [M, N] (splits == 1)
  float* sCq;                   // optional [N/128, M]
  float* Cacc;                  // fp32 [M, N] accumulated into instead of C (kEpiAccum, or the split-K reduction)
  uint64_t wait_ns;
  uint32_t stall;               // test hook: the producer first waits on a barrier nothing completes
};

// Three warpgroups: 0 and 1 promote, 2 holds the producer (warp 8) and the
// MMA issuer (warp 9); warps 10 and 11 only give their registers away.
// At launch every thread has kLaunchRegs registers (65536 / 384, rounded
// down to a multiple of 8); warpgroup 2 then drops to kSmallRegs and the
// promotion warpgroups rise to kBigRegs.  The split adds up exactly:
// 128 * 56 + 256 * 224 = 384 * 168.
constexpr int kGemmThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kLaunchRegs = 168;
constexpr int kSmallRegs = 56;
constexpr int kBigRegs = 224;
static_assert(128 * kSmallRegs + 256 * kBigRegs <= kGemmThreads * kLaunchRegs, "register split exceeds the launch");
// Shared memory of the GEMM: a ring of A (128x128) and B (BNx128) E4M3
// tiles, the bf16 output staging for the TMA-store epilogue (each promotion
// warp owns 32 rows x BN/2 columns, in boxes of 64 columns, 128-byte
// swizzled), the scale ring and the barriers.  Scale slot i holds the scales
// of one slice: sa of this CTA's 128 rows, then sb (the slice's block
// scalars of the tile's column blocks, or its BN per-column scales).
// With kPair the CTA is one of a pair sharing a 256 x BN tile: it holds its
// own 128 rows of A and half (BN/2 rows) of B per stage.
// kCol: the per-column (WGRAD) promotion layout (see gemm_body): a 2 KB
// staging area per warp, drained in passes of 32 bf16 (or 16 fp32) columns,
// leaves room for a deeper operand ring, and sb sits in each slot in the
// order the promotion threads read it.
template <int BN, bool kPair = false, bool kCol = false>
struct GemmSmem {
  static constexpr int kStages = kCol ? (kPair ? 6 : (BN == 256 ? 4 : 6)) : (kPair ? 4 : (BN == 256 ? 3 : 4));
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = (kPair ? BN / 2 : BN) * 128;
  static constexpr int kAOff = 0;
  static constexpr int kBOff = kStages * kABytes;
  static constexpr int kCWarpBytes = kCol ? 2048 : 32 * (BN / 2) * 2;  // one promotion warp's staging
  static constexpr int kCOff = kBOff + kStages * kBBytes;            // 1024-aligned
  // At least kStages + 2: the producer's lead (operand ring + two TMEM
  // buffers) never waits on a scale slot.
  static constexpr int kScaleSlots = kCol ? kStages + 2 : 8;
  // kCol: sb is stored as 8 runs (warp half x thread column pair) of BN/8
  // scales, each run padded by 4 floats so that the 4 runs a warp reads at
  // once start in different banks.
  static constexpr int kSbStride = BN / 8 + 4;
  static constexpr int kScaleSlotFloats = 128 + (kCol ? 8 * kSbStride : BN);
  static constexpr int kScaleOff = kCOff + 8 * kCWarpBytes;
  static constexpr int kBarOff = kScaleOff + kScaleSlots * kScaleSlotFloats * 4;
  // barriers: full[S], empty[S], tfull[2], tempty[2], done, sfull[slots], sempty[slots], stall
  static constexpr int kNumBars = 2 * kStages + 5 + 2 * kScaleSlots + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kTmemSlotOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
  static constexpr uint32_t kTmemCols = 2 * BN;
  static_assert(kAlloc <= 232448, "GEMM shared memory exceeds the per-CTA limit");
};

struct UnitCoords {
  int m0;     // first output row
  int nt;     // output column tile index (columns nt*BN ..)
  int split;  // split-K index
  int kb0, kb1;  // slice range [kb0, kb1)
};

__device__ __forceinline__ UnitCoords unit_coords(const GemmParams& p, int u) {
  UnitCoords c;
  const int tile = u % p.tiles;
  c.split = u / p.tiles;
  const int per_group = p.group_m * p.n_tiles;
  const int g = tile / per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.m_tiles - first_m, p.group_m);
  const int in_g = tile - g * per_group;
  c.m0 = (first_m + in_g % gm) * p.m_tile_rows;
  c.nt = in_g / gm;
  const int nk = p.K / 128;
  c.kb0 = c.split * p.kps;
  c.kb1 = min(nk, c.kb0 + p.kps);
  return c;
}

// acc[0..31] += v[0..31] * scale: one scale s2 for the block modes, sa times
// the 32 per-column scales at sbc for kSbCol.
template <int SBMODE>
__device__ __forceinline__ void promote32(float* acc, const uint32_t (&v)[32], float2 s2, float2 sa2,
                                          const float* sbc) {
  if constexpr (SBMODE != kSbCol) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 a2 = ffma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), s2,
                              make_float2(acc[i], acc[i + 1]));
      acc[i] = a2.x;
      acc[i + 1] = a2.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 sb4 = *reinterpret_cast<const float4*>(sbc + i);
      const float2 sc0 = fmul2(sa2, make_float2(sb4.x, sb4.y));
      const float2 sc1 = fmul2(sa2, make_float2(sb4.z, sb4.w));
      const float2 a0 = ffma2(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), sc0,
                              make_float2(acc[i], acc[i + 1]));
      const float2 a1 = ffma2(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])), sc1,
                              make_float2(acc[i + 2], acc[i + 3]));
      acc[i] = a0.x;
      acc[i + 1] = a0.y;
      acc[i + 2] = a1.x;
      acc[i + 3] = a1.y;
    }
  }
}

// The GEMM body.  kPair: this CTA and its cluster peer compute a 256 x BN
// tile together with tcgen05 pair MMAs (cta_group::2): each loads its own
// 128 rows of A and BN/2 rows of B (so each SM moves 32 KB per slice instead
// of 48 KB), the first CTA of the pair issues the MMAs, whose results land in
// both CTAs' tensor memory (each CTA its own 128 rows x BN columns), and each
// CTA promotes and stores its own rows.
//
// Promotion layouts.  With one scale per row (FPROP, DGRAD) each promotion
// thread owns one tile row (TMEM lane) and BN/2 consecutive columns, read
// with the 32x32b shape.  With the WGRAD outer product sa(i) sb(j), a thread
// so placed needs all BN/2 column scales of every slice, and those
// warp-uniform shared-memory reads (two wavefronts per 16 bytes) held the
// kernel back.  The column layout (kCol) reads TMEM with the 16x256b shape
// instead: thread t of a warp owns rows 16h + 8i + t/4 (h, i in {0, 1}) of its
// 32 and columns 8j + 2 (t%4) + {0, 1} of its BN/2, so it needs BN/8 column
// scales per slice, which the producer stores in that order (4 threads read 4
// different 16-byte pieces per load).  The fused E4M3 epilogue keeps the row
// layout (it needs whole 128-column groups per thread).
template <int SBMODE, int kEpi>
__host__ __device__ constexpr bool gemm_col_layout() {
  return SBMODE == kSbCol && kEpi != kEpiCodes;
}

// Shared-memory bytes a GEMM kernel instance needs.
template <int BN, bool kPair, int SBMODE, int kEpi>
__host__ __device__ constexpr int gemm_smem_alloc() {
  return GemmSmem<BN, kPair, gemm_col_layout<SBMODE, kEpi>()>::kAlloc;
}

// The promotion warps in the column layout (WGRAD), with their epilogues.
// Warp w owns TMEM lanes 32 (w%4) .. +31 and columns (w/4) BN/2 .. +BN/2-1
// of the CTA's tile; its thread t owns, for h, i in {0, 1}, row
// 16h + 8i + t/4 of those 32 and, for every 8-column group j, columns
// 8j + 2 (t%4) + {0, 1}.  acc holds them in the register order of the
// 16x256b loads: acc[32 (h kChunks + ch) + 4 jj + 2 i + e] is row
// 16h + 8i + t/4, column 8 (8 ch + jj) + 2 (t%4) + e.
template <int BN, bool kPair, int kEpi, typename L>
__device__ __forceinline__ void promote_col(const CUtensorMap& tmC, const GemmParams& p, uint8_t* smem,
                                            const float* scales, uint64_t* tfull, uint64_t* tempty, uint64_t* sfull,
                                            uint64_t* sempty, uint32_t tmem_base, uint32_t rank, int unit0,
                                            int unit_step, int warp, int lane) {
  constexpr int kCols = BN / 2;        // columns of this warp
  constexpr int kJ = kCols / 8;        // 8-column groups of a thread
  constexpr int kChunks = kCols / 64;  // 16x256b.x8 loads (64 columns) per 16-lane half
  constexpr int kSlots = L::kScaleSlots, kSlotFloats = L::kScaleSlotFloats;
  const int quad = warp & 3, half = warp >> 2;
  const int tq = lane & 3, tr = lane >> 2;
  uint32_t it = 0;
  bool ok = true;
  float acc[8 * kJ];
  const uint32_t tempty_leader0 = kPair ? mapa_shared(&tempty[0], 0) : 0u;
  const uint32_t tempty_leader1 = kPair ? mapa_shared(&tempty[1], 0) : 0u;
  for (int u = unit0; u < p.units && ok; u += unit_step) {
    UnitCoords c = unit_coords(p, u);
    c.m0 += 128 * static_cast<int>(rank);  // this CTA's rows of a pair tile
    const int row0 = c.m0 + quad * 32;     // first output row of this warp
    const int col0 = c.nt * BN + half * kCols;
#pragma unroll
    for (int i = 0; i < 8 * kJ; ++i) acc[i] = 0.0f;

    for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
      const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
      const uint32_t q = it % kSlots, qph = (it / kSlots) & 1u;
      if (!mbar_wait(&sfull[q], qph, p.wait_ns, 0x332u) || !mbar_wait(&tfull[b], bph, p.wait_ns, 0x331u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the slice's scales of this thread's 4 rows and 2 kJ columns (the
      // producer stored the columns in this thread's order)
      const float* slot = scales + q * kSlotFloats;
      float sa_r[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) sa_r[rr] = slot[quad * 32 + 16 * (rr >> 1) + 8 * (rr & 1) + tr];
      const float4* sb4 = reinterpret_cast<const float4*>(slot + 128 + (half * 4 + tq) * L::kSbStride);
      // 64 columns at a time (both 16-lane halves, one 16x256b.x8 load each),
      // so that only their 16 column scales are live next to the
      // accumulators; the buffer is handed back once its last chunk is in
      // registers.
      const uint32_t tbase = tmem_base + b * BN + half * kCols;
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        float2 sbp[8];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float4 t = sb4[4 * ch + jj];
          sbp[2 * jj] = make_float2(t.x, t.y);
          sbp[2 * jj + 1] = make_float2(t.z, t.w);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld16x256b_x8(tbase + (static_cast<uint32_t>(quad * 32 + 16 * h) << 16) + 64 * ch, v);
          tmem_wait_ld32(v);
          if (h == 1 && ch + 1 == kChunks) {  // the buffer is in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (kPair && rank != 0)
                mbar_arrive_cluster(b ? tempty_leader1 : tempty_leader0);
              else
                mbar_arrive(&tempty[b]);
            }
          }
          const uint32_t* cur = v;
          float* a = acc + 32 * (h * kChunks + ch);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float2 sc = fmul2(make_float2(sa_r[2 * h + i], sa_r[2 * h + i]), sbp[jj]);
              const float2 r = ffma2(make_float2(__uint_as_float(cur[4 * jj + 2 * i]), __uint_as_float(cur[4 * jj + 2 * i + 1])),
                                     sc, make_float2(a[4 * jj + 2 * i], a[4 * jj + 2 * i + 1]));
              a[4 * jj + 2 * i] = r.x;
              a[4 * jj + 2 * i + 1] = r.y;
            }
          }
          reg_fence32(a);
        }
      }
      // the slot's scales have been read
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[q]);
    }
    if (!ok) break;

    // ------------------------------------------------------------ epilogue
    // acc index of row 16h + 8i + t/4, column pair (8j + 2 (t%4)) of the warp
    auto at = [&](int h, int i, int j) -> float* { return acc + 32 * (h * kChunks + j / 8) + 4 * (j % 8) + 2 * i; };
    if (p.splits > 1) {
      // fp32 partial sums of this split, 8 bytes per store
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float* prow = p.Cpart + (static_cast<int64_t>(c.split) * p.M + row0 + 16 * h + 8 * i + tr) * p.N + col0 + 2 * tq;
#pragma unroll
          for (int j = 0; j < kJ; ++j) {
            const float* a = at(h, i, j);
            *reinterpret_cast<float2*>(prow + 8 * j) = make_float2(a[0], a[1]);
          }
        }
    } else {
      // Through this warp's 2 KB staging area (rows of 64 bytes, 64-byte
      // swizzle: 16-byte chunk k of row r at chunk k ^ ((r >> 1) & 3)), one
      // TMA box of 32 rows per pass: 32 bf16 columns (plain) or 16 fp32
      // columns added into the output (accumulate).
      constexpr bool kAcc = kEpi == kEpiAccum;
      constexpr int kPassCols = kAcc ? 16 : 32;
      uint8_t* stg = smem + L::kCOff + warp * L::kCWarpBytes;
#pragma unroll
      for (int ps = 0; ps < kCols / kPassCols; ++ps) {
        if (lane == 0) bulk_wait_group_read<0>();  // the previous pass's box has been read
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t r = 16 * h + 8 * i + tr, sw = (r >> 1) & 3u;
#pragma unroll
            for (int g = 0; g < kPassCols / 8; ++g) {  // 8-column group g of the pass
              const float* a = at(h, i, ps * (kPassCols / 8) + g);
              if constexpr (kAcc) {
                // columns 8g' + 2tq, +1: byte 4 (8g' + 2tq) = chunk 2g' + tq/2,
                // offset 8 (tq%2).  Lanes 8..15 and 24..31 (rows with bit 1
                // set) store the other group g' = g ^ 1 first, which puts the
                // 4 rows of each 16-lane phase in different banks.
                const float* o = at(h, i, ps * (kPassCols / 8) + (g ^ 1));
                const bool flip = (lane >> 3) & 1;
                const float2 val = flip ? make_float2(o[0], o[1]) : make_float2(a[0], a[1]);
                const uint32_t chunk = static_cast<uint32_t>(2 * (g ^ static_cast<int>(flip)) + (tq >> 1));
                *reinterpret_cast<float2*>(stg + r * 64 + ((chunk ^ sw) << 4) + 8 * (tq & 1)) = val;
              } else {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(a[0], a[1]);
                *reinterpret_cast<uint32_t*>(stg + r * 64 + ((static_cast<uint32_t>(g) ^ sw) << 4) + 4 * tq) =
                    *reinterpret_cast<const uint32_t*>(&h2);
              }
            }
          }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kAcc)
            tma_reduce_add_2d(&tmC, stg, col0 + kPassCols * ps, row0);
          else
            tma_store_2d(&tmC, stg, col0 + kPassCols * ps, row0);
          bulk_commit_group();
        }
      }
    }
  }
}

template <int BN, int SBMODE, bool kPair, int kEpi>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                                          const GemmParams& p) {
  constexpr bool kCol = gemm_col_layout<SBMODE, kEpi>();
  using L = GemmSmem<BN, kPair, kCol>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint64_t* done = bars + 2 * kStages + 4;
  uint64_t* sfull = bars + 2 * kStages + 5;  // scale slot landed (32 producer lanes)
  uint64_t* sempty = sfull + L::kScaleSlots;  // scale slot read (8 promotion warps)
  uint64_t* stall = sempty + L::kScaleSlots;  // never completed (test hook p.stall)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOff);
  float* scales = reinterpret_cast<float*>(smem + L::kScaleOff);
  constexpr int kSlots = L::kScaleSlots, kSlotFloats = L::kScaleSlotFloats;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0: this CTA issues the MMAs
  const int unit0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kPair ? 16 : 8);  // one arrival per promotion warp (of both CTAs)
    }
    mbar_init(done, 1);
    mbar_init(stall, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sfull[i], 32);
      mbar_init(&sempty[i], 8);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, L::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, L::kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers must be initialised before either CTA signals them
  if constexpr (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= kProducerWarp) {
    setmaxnreg_dec<kSmallRegs>();
    if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the operand tiles (TMA); every lane copies its share of
    // the slice's scales into the scale ring (cp.async, completion counted
    // on the slot's barrier), so the promotion warps never wait on global
    // memory for a scale.
    const int nkb = p.K / 128;
    uint32_t it = 0;
    bool ok = true;
    // Test hook: a wait that nothing satisfies, so that it expires after the
    // wait limit and the kernel takes its early-exit path before any copy.
    if (p.stall != 0u) ok = mbar_wait(stall, 0, p.wait_ns, 0x300u);
    for (int u = unit0; u < p.units && ok; u += unit_step) {
      UnitCoords c = unit_coords(p, u);
      const int m_rows = c.m0 + 128 * static_cast<int>(rank);  // this CTA's rows
      for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
        const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
        const uint32_t q = it % kSlots, qph = (it / kSlots) & 1u;
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1u, p.wait_ns, 0x301u);
        w_ok = mbar_wait(&sempty[q], qph ^ 1u, p.wait_ns, 0x303u) && w_ok;
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        float* slot = scales + q * kSlotFloats;
        cp_async16(slot + 4 * lane, p.sa + static_cast<int64_t>(kb) * p.M + m_rows + 4 * lane);
        if constexpr (kCol) {
          // columns (col, col + 1) of the tile, col = 2 (32 r + lane), go to
          // the run of warp half col / (BN/2) and thread column pair
          // (col % 8) / 2, at position 2 (col % (BN/2)) / 8 of the run
          constexpr int kHalfCols = BN / 2;
#pragma unroll
          for (int r = 0; r < BN / 64; ++r) {
            const int col = 2 * (32 * r + lane);
            const int cc = col % kHalfCols;
            const int dst = ((col / kHalfCols) * 4 + (cc % 8) / 2) * L::kSbStride + 2 * (cc / 8);
            cp_async8(slot + 128 + dst, p.sb + static_cast<int64_t>(kb) * p.N + c.nt * BN + col);
          }
        } else if constexpr (SBMODE == kSbCol) {
#pragma unroll
          for (int r = 0; r < BN / 128; ++r)
            cp_async16(slot + 128 + 128 * r + 4 * lane,
                       p.sb + static_cast<int64_t>(kb) * p.N + c.nt * BN + 128 * r + 4 * lane);
        } else {
          if (lane < BN / 128) {
            const int nb = c.nt * (BN / 128) + lane;  // column block
            const float* src = SBMODE == kSbBlock ? p.sb + static_cast<int64_t>(nb) * nkb + kb
                                                  : p.sb + static_cast<int64_t>(kb) * (p.N / 128) + nb;
            cp_async4(slot + 128 + lane, src);
          }
        }
        cp_async_arrive(&sfull[q]);
        if (lane == 0) {
          if constexpr (kPair) {
            // both CTAs' copies are counted on the first CTA's full[s]
            const uint32_t leader_full = mapa_shared(&full[s], 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (L::kABytes + L::kBBytes));
            tma_load_2d_pair(smem + L::kAOff + s * L::kABytes, &tmA, kb * 128, m_rows, leader_full);
            tma_load_2d_pair(smem + L::kBOff + s * L::kBBytes, &tmB, kb * 128,
                             c.nt * BN + (BN / 2) * static_cast<int>(rank), leader_full);
          } else {
            mbar_arrive_expect_tx(&full[s], L::kABytes + L::kBBytes);
            tma_load_2d(smem + L::kAOff + s * L::kABytes, &tmA, kb * 128, c.m0, &full[s]);
            tma_load_2d(smem + L::kBOff + s * L::kBBytes, &tmB, kb * 128, c.nt * BN, &full[s]);
          }
        }
        __syncwarp();
      }
    }
    // Do not leave while copies into this CTA's shared memory are in flight:
    // this lane's scale copies, and the last fill of every operand stage (for
    // a pair, the first CTA's full barriers count both CTAs' copies; the
    // second CTA is held by the cluster barrier at the end until the first
    // is done).
    cp_async_wait_all();
    if (lane == 0 && (!kPair || rank == 0)) {
      for (uint32_t j = 0; j < kStages && j < it; ++j) {
        const uint32_t f = it - 1 - j;
        mbar_wait(&full[f % kStages], (f / kStages) & 1u, kDrainWaitNs, 0x302u);
      }
    }
    } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kPair ? 256 : 128, BN);
      uint32_t it = 0;
      bool ok = true;
      for (int u = unit0; u < p.units && ok; u += unit_step) {
        const UnitCoords c = unit_coords(p, u);
        for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
          if (!mbar_wait(&tempty[b], bph ^ 1u, p.wait_ns, 0x311u) || !mbar_wait(&full[s], ph, p.wait_ns, 0x312u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + L::kAOff + s * L::kABytes);
          const uint32_t b_addr = smem_u32(smem + L::kBOff + s * L::kBBytes);
          const uint32_t d = tmem_base + b * BN;
          if constexpr (kPair) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_e4m3_pair(d, sw128_kmajor_desc(a_addr + 32 * k), sw128_kmajor_desc(b_addr + 32 * k), idesc, k > 0);
            mma_commit_pair_mc(&empty[s], 0x3);
            mma_commit_pair_mc(&tfull[b], 0x3);
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_e4m3(d, sw128_kmajor_desc(a_addr + 32 * k), sw128_kmajor_desc(b_addr + 32 * k), idesc, k > 0);
            mma_commit(&empty[s]);
            mma_commit(&tfull[b]);
          }
        }
      }
      // Every MMA this thread issued has completed once `done` fires.
      if constexpr (kPair) {
        mma_commit_pair_mc(done, 0x1);
      } else {
        mma_commit(done);
      }
      mbar_wait(done, 0, kDrainWaitNs, 0x313u);
    }
    }
  } else {
    setmaxnreg_inc<kBigRegs>();
    if constexpr (kCol) {
      promote_col<BN, kPair, kEpi, L>(tmC, p, smem, scales, tfull, tempty, sfull, sempty, tmem_base, rank, unit0,
                                      unit_step, warp, lane);
    } else {
    // ------------------------------------------------------------ promotion
    constexpr int kCols = BN / 2;  // output columns per promotion thread
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    float acc[kCols];
    // where this warp reports a freed TMEM buffer: the first CTA's tempty
    const uint32_t tempty_leader0 = kPair ? mapa_shared(&tempty[0], 0) : 0u;
    const uint32_t tempty_leader1 = kPair ? mapa_shared(&tempty[1], 0) : 0u;
    for (int u = unit0; u < p.units && ok; u += unit_step) {
      UnitCoords c = unit_coords(p, u);
      c.m0 += 128 * static_cast<int>(rank);  // this CTA's rows of a pair tile
      const int gm = c.m0 + row;
      const int col0 = c.nt * BN + half * kCols;  // first output column of this thread
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0.0f;

      for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
        const uint32_t b = it & 1u, bph = (it >> 1) & 1u;
        const uint32_t q = it % kSlots, qph = (it / kSlots) & 1u;
        if (!mbar_wait(&sfull[q], qph, p.wait_ns, 0x322u) || !mbar_wait(&tfull[b], bph, p.wait_ns, 0x321u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this slice's scales: sa of this thread's row; sb of its column
        // block (block modes) or its columns (kSbCol)
        const float* slot = scales + q * kSlotFloats;
        const float sa_cur = slot[row];
        const float sb_cur = SBMODE == kSbCol ? 1.0f : slot[128 + (BN == 256 ? half : 0)];
        const float* sbc = slot + 128 + half * kCols;
        const uint32_t taddr = tmem_base + lane_base + b * BN + half * kCols;
        // acc[j] += P[j] * scale(j) over this thread's kCols columns, read
        // from TMEM 64 columns at a time: each tcgen05.ld round trip is
        // long next to the FMAs it feeds, and tcgen05.wait::ld drains every
        // outstanding load, so fewer, wider loads shorten the chain.  The
        // buffer is released as soon as its last chunk is in registers.
        const float sc = sa_cur * sb_cur;
        const float2 s2 = make_float2(sc, sc);
        const float2 sa2 = make_float2(sa_cur, sa_cur);
#pragma unroll
        for (int ch = 0; ch < kCols / 64; ++ch) {
          uint32_t v[64];
          tmem_ld64(taddr + ch * 64, v);
          tmem_wait_ld64(v);
          if (ch + 1 == kCols / 64) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (kPair && rank != 0)
                mbar_arrive_cluster(b ? tempty_leader1 : tempty_leader0);
              else
                mbar_arrive(&tempty[b]);
            }
          }
          promote32<SBMODE>(acc + ch * 64, *reinterpret_cast<const uint32_t(*)[32]>(v), s2, sa2, sbc + ch * 64);
          promote32<SBMODE>(acc + ch * 64 + 32, *reinterpret_cast<const uint32_t(*)[32]>(v + 32), s2, sa2,
                            sbc + ch * 64 + 32);
          reg_fence64(acc + ch * 64);
        }
        // the slot's scales have been read
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[q]);
      }
      if (!ok) break;

      // ------------------------------------------------------------ epilogue
      if constexpr (kEpi == kEpiCodes) {
        // One split, BN = 256, codes requested: bf16 and E4M3 outputs are
        // stored directly (each thread owns whole 128-column groups).
        // bf16 output, 8 columns (16 bytes) per store.
        uint16_t* crow = p.C + static_cast<int64_t>(gm) * p.N + col0;
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < kCols / 8; ++i) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[8 * i + 2 * j], acc[8 * i + 2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h2);
            m = fmaxf(m, fmaxf(fabsf(bf16lo(w[j])), fabsf(bf16hi(w[j]))));
          }
          *reinterpret_cast<uint4*>(crow + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        {
          // E4M3 codes of the bf16 values of this thread's 128-column group,
          // with the activation quantiser's rule (m is their amax).
          const GroupScale g = make_group_scale(m);
          uint8_t* qrow = p.Cq + static_cast<int64_t>(gm) * p.N + col0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = 16 * i + 4 * j;
              const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[c], acc[c + 1]);
              const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[c + 2], acc[c + 3]);
              const uint32_t l = *reinterpret_cast<const uint32_t*>(&lo), h = *reinterpret_cast<const uint32_t*>(&hi);
              w[j] = quant_pair(bf16lo(l), bf16hi(l), g) | (quant_pair(bf16lo(h), bf16hi(h), g) << 16);
            }
            *reinterpret_cast<uint4*>(qrow + 16 * i) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          p.sCq[static_cast<int64_t>(col0 / 128) * p.M + gm] = g.s;
        }
      } else if (kEpi == kEpiAccum && p.splits == 1) {
        // C_f32 += acc: this warp's 32 rows x kCols fp32 values go through
        // its staging area in passes of kPass columns (boxes of 32 columns,
        // 128-byte swizzle), each added into global memory by TMA
        // reduce-add stores, one fp32 addition per element.
        constexpr int kPass = L::kCWarpBytes / (32 * 4);  // columns per pass: 64 (BN 256) or 32 (BN 128)
        uint8_t* stg = smem + L::kCOff + warp * L::kCWarpBytes;
#pragma unroll
        for (int ps = 0; ps < kCols / kPass; ++ps) {
          if (lane == 0) bulk_wait_group_read<0>();  // the staging area has been read
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kPass / 4; ++i) {
            const float* a = acc + kPass * ps + 4 * i;
            *reinterpret_cast<float4*>(stg + (i / 8) * 4096 + lane * 128 + (((i % 8) ^ (lane & 7)) << 4)) =
                make_float4(a[0], a[1], a[2], a[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int bx = 0; bx < kPass / 32; ++bx)
              tma_reduce_add_2d(&tmC, stg + bx * 4096, col0 + kPass * ps + 32 * bx, c.m0 + quad * 32);
            bulk_commit_group();
          }
        }
      } else if (p.splits == 1) {
        // bf16 output through shared memory and TMA stores: this warp's 32
        // rows x kCols columns go to its staging boxes (64 columns, 128-byte
        // swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)), then lane
        // 0 issues the stores and the warp moves on to the next tile.
        uint8_t* stg = smem + L::kCOff + warp * L::kCWarpBytes;
        if (lane == 0) bulk_wait_group_read<0>();  // the previous tile's stores have read it
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kCols / 8; ++i) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[8 * i + 2 * j], acc[8 * i + 2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(stg + (i / 8) * 4096 + lane * 128 + (((i % 8) ^ (lane & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int bx = 0; bx < kCols / 64; ++bx) tma_store_2d(&tmC, stg + bx * 4096, col0 + 64 * bx, c.m0 + quad * 32);
          bulk_commit_group();
        }
      } else {
        float* prow = p.Cpart + (static_cast<int64_t>(c.split) * p.M + gm) * p.N + col0;
#pragma unroll
        for (int i = 0; i < kCols / 4; ++i)
          *reinterpret_cast<float4*>(prow + 4 * i) = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
    }
    }
  }

  // the staged output must have been read (and written) before the CTA ends
  if (warp < kProducerWarp && lane == 0) bulk_wait_group<0>();
  tc_fence_before();
  __syncthreads();
  // neither CTA of a pair may leave (or free tensor memory) while the other
  // can still signal its barriers or read its shared memory
  if constexpr (kPair) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, L::kTmemCols);
    else
      tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// kEpi selects the epilogue (EpiKind).  Each kind is its own instance so
// that the plain GEMM holds none of the others' code: the E4M3 epilogue's
// IEEE division fallbacks, for one, would otherwise sit (unused) in every
// GEMM kernel and take part in its register allocation.  tmC describes the
// bf16 output for kEpiPlain and the fp32 output for kEpiAccum.
template <int BN, int SBMODE, int kEpi = kEpiPlain>
__global__ void __launch_bounds__(kGemmThreads, 1)
    block_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  static_assert(kEpi != kEpiCodes || BN == 256, "the E4M3 epilogue needs whole 128-column groups per thread");
  gemm_body<BN, SBMODE, false, kEpi>(tmA, tmB, tmC, p);
}

// 256 x 256 output tiles on CTA pairs (clusters of two).
template <int SBMODE, int kEpi = kEpiPlain>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    block_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  gemm_body<256, SBMODE, true, kEpi>(tmA, tmB, tmC, p);
}

// Adds the fp32 split-K partials in split order, rounds to bf16 and,
// optionally, quantises each 128-column group of the bf16 result exactly as
// the activation quantiser does.  One warp per 128-column group of a row.
// With Cacc the sum is instead added into the fp32 output (one addition per
// element) and C, Cq are not written.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part, int splits, int M, int N,
                                                            uint16_t* __restrict__ C, uint8_t* __restrict__ Cq,
                                                            float* __restrict__ sCq, float* __restrict__ Cacc) {
  const int64_t groups = static_cast<int64_t>(M) * (N / 128);
  const int lane = threadIdx.x & 31;
  for (int64_t g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; g < groups;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x / 32) {
    const int64_t r = g / (N / 128), cg = g % (N / 128);
    const int64_t off = r * N + cg * 128 + lane * 4;
    float4 a = *reinterpret_cast<const float4*>(part + off);
    for (int s = 1; s < splits; ++s) {
      const float4 b = *reinterpret_cast<const float4*>(part + static_cast<int64_t>(s) * M * N + off);
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (Cacc != nullptr) {
      float4 m = *reinterpret_cast<const float4*>(Cacc + off);
      m.x += a.x;
      m.y += a.y;
      m.z += a.z;
      m.w += a.w;
      *reinterpret_cast<float4*>(Cacc + off) = m;
      continue;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&lo);
    v.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(C + off) = v;
    if (Cq != nullptr) {
      const GroupScale gs = make_group_scale(warp_max(fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))),
                                                            fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))))));
      const uint32_t q = quant_pair(bf16lo(v.x), bf16hi(v.x), gs) | (quant_pair(bf16lo(v.y), bf16hi(v.y), gs) << 16);
      *reinterpret_cast<uint32_t*>(Cq + off) = q;
      if (lane == 0) sCq[cg * M + r] = gs.s;
    }
  }
}

}  // namespace bfp8
