// E4M3 quantisers: 1x128 activation groups (along the columns, and along
// the rows with transposed storage) and 128x128 weight blocks.
//
// Numerics follow "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within
// $5090", section 3.2: one scale per 128 consecutive values along the GEMM
// reduction dimension for activations and activation gradients, one per
// 128x128 block for weights, each computed online from its own values.
// Per group: amax = max|x| (NaN ignored); s = amax/448 in IEEE fp32 (1 when
// amax == 0); q = E4M3_rn_satfinite(fp32_rn(x / s)).  The quotient is formed
// exactly by FMA correction steps (GroupScale), so codes and scales match a
// plain CPU evaluation bit for bit.
//
// Work decomposition.  The input is cut into 128x128 bf16 tiles (32 KB),
// walked in row-major order by a persistent grid (two CTAs per SM).  A CTA
// streams its tiles through a 3-deep shared-memory ring filled by bulk
// copies; its eight warps share each tile without any block-wide barrier
// (warp 0 also refills a slot once every warp has released it).  Warp w owns
//   * rows 16w..16w+15 (their 1x128 groups along the columns: q, s): lane
//     pair (2j, 2j+1) holds row 16w+j, 64 values each, as the 16-code output
//     chunks 2m+h (h = lane & 1), and
//   * columns 16w..16w+15 (their groups of 128 rows: qT, sT): lane l holds
//     columns 16w+4(l%4)..+3 over rows 16(l/4)..16(l/4)+15.
// It copies both slices into registers, releases the ring slot, reduces
// amaxes with in-lane packed bf16 maxima and a few shuffles, turns each
// amax into its scale and reciprocal once per warp instruction stream, forms
// every code from the correctly rounded quotient (GroupScale), and stores codes
// straight to global memory in 32-byte (rows) and 128-byte (columns)
// segments.  The input is read from HBM once whichever outputs are requested.
//
// Shared-memory image of a tile: row r (256 bytes) starts at byte
// 272 r + 32 ((r / 16) % 8).  The 16-byte stride padding and the per-block
// offset make both register views conflict-free: in the row view 16
// consecutive rows cover the eight 16-byte bank groups twice per half-warp;
// in the column view rows 16 apart start 32 bytes (8 banks) apart, so eight
// of them tile the 32 banks in two wavefronts, the minimum for 256 bytes.
#pragma once

#include "common.cuh"

namespace bfp8 {

struct QuantParams {
  const uint16_t* x;  // bf16 [R, C]
  int64_t R, C;
  uint8_t* q;   // [R, C] or null
  float* s;     // act: [C/128, R];  weight: [R/128, C/128]
  uint8_t* qT;  // [C, R] or null
  float* sT;    // act: [R/128, C];  unused for weights
  uint64_t wait_ns;
};

constexpr int kQComputeWarps = 8;
constexpr int kQuantThreads = 32 * kQComputeWarps;
constexpr int kQStages = 3;
constexpr int kQTileBytes = 128 * 256;                     // bf16 payload of a tile
constexpr int kQBufBytes = 35072;                          // padded image, >= 272*127 + 32*7 + 256
constexpr int kQBarOff = kQStages * kQBufBytes;            // full[3], empty[3], redbar[2]
constexpr int kQRedOff = kQBarOff + (2 * kQStages + 2) * 8;  // float[2][8] (weight block amax)
constexpr int kQuantSmemBytes = kQRedOff + 2 * kQComputeWarps * 4;
static_assert(272 * 127 + 32 * 7 + 256 <= kQBufBytes, "tile image overflows its buffer");

__device__ __forceinline__ uint32_t qrow_off(int r) { return 272u * r + 32u * ((r >> 4) & 7); }

__device__ __forceinline__ float bf16x2_absmax(uint32_t w) { return fmaxf(fabsf(bf16lo(w)), fabsf(bf16hi(w))); }

// max(|a|, |b|) per bf16 half (NaN ignored); the sign bits of the result are
// meaningless and are dropped when the halves are widened.
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 16 codes of 8 words of bf16 pairs (value 2i in the low half of word i),
// one group.  Groups with extreme scales (g.exact false) take the IEEE
// division; the branch is uniform over the group.
__device__ __forceinline__ uint4 quant16w(const uint32_t (&w)[8], const GroupScale& g) {
  if (g.exact) {
    const float2 r2 = make_float2(g.r, g.r), ns2 = make_float2(-g.s, -g.s);
    return make_uint4(quant4_exact(w[0], w[1], r2, ns2), quant4_exact(w[2], w[3], r2, ns2),
                      quant4_exact(w[4], w[5], r2, ns2), quant4_exact(w[6], w[7], r2, ns2));
  }
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = quant_pair_div(bf16lo(w[i]), bf16hi(w[i]), g.s, g.s);
  return make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16), c[6] | (c[7] << 16));
}

// 16 codes of the 16 consecutive values in (a, b) (8 bf16 each), one group.
__device__ __forceinline__ uint4 quant16(const uint4& a, const uint4& b, const GroupScale& g) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  return quant16w(w, g);
}

// Values k and k+1 of one column (element kHalf of word kWord of row slices
// k and k+1 in v[]) packed as one bf16 pair, row k in the low half.
template <int kWord, int kHalf>
__device__ __forceinline__ uint32_t col_pair(const uint2 (&v)[16], int k) {
  const uint32_t w0 = kWord ? v[k].y : v[k].x, w1 = kWord ? v[k + 1].y : v[k + 1].x;
  return kHalf ? __byte_perm(w0, w1, 0x7632) : __byte_perm(w0, w1, 0x5410);
}

// 16 codes of one column over 16 rows, one group.  Codes in row order.
template <int kWord, int kHalf>
__device__ __forceinline__ uint4 quant_col16(const uint2 (&v)[16], const GroupScale& g) {
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 16; k += 2) w[k / 2] = col_pair<kWord, kHalf>(v, k);
  return quant16w(w, g);
}

// kWeight = false: activation groups (rows -> q/s, columns -> qT/sT).
// kWeight = true : one 128x128 block per tile (q and/or qT, one scale).
// Issues the bulk copies of tile t into ring slot `buf` (one whole warp;
// lane 0 arms the slot's barrier).
__device__ __forceinline__ void quant_fill(const QuantParams& p, int64_t t, int64_t ctiles, uint8_t* buf,
                                           uint64_t* bar, int lane) {
  const int64_t r0 = (t / ctiles) * 128, c0 = (t % ctiles) * 128;
  if (lane == 0) mbar_arrive_expect_tx(bar, kQTileBytes);
  __syncwarp();
  for (int r = lane; r < 128; r += 32) bulk_g2s(buf + qrow_off(r), p.x + (r0 + r) * p.C + c0, 256, bar);
}

// kWeight = false: activation groups (rows -> q/s, columns -> qT/sT).
// kWeight = true : one 128x128 block per tile (q and/or qT, one scale).
template <bool kWeight>
__global__ void __launch_bounds__(kQuantThreads, 2) quantize_tile_kernel(const QuantParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQBarOff);
  uint64_t* empty = full + kQStages;
  uint64_t* redbar = empty + kQStages;  // weight block amax exchange, by tile parity
  float* red = reinterpret_cast<float*>(smem + kQRedOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ctiles = p.C / 128;
  const int64_t tiles = (p.R / 128) * ctiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kQComputeWarps);
    }
    mbar_init(&redbar[0], kQComputeWarps);
    mbar_init(&redbar[1], kQComputeWarps);
    fence_mbar_init();
  }
  __syncthreads();
  // prologue: warp 0 issues the first kQStages tiles of this CTA, and later
  // each tile j-1+kQStages at iteration j.
  int64_t last_issued = -1;  // latest tile (local index) this warp issued after the prologue
  uint32_t prologue = 0;     // tiles issued by the prologue (warp 0)
  if (warp == 0) {
    int64_t t = blockIdx.x;
    for (; prologue < kQStages && t < tiles; ++prologue, t += gridDim.x)
      quant_fill(p, t, ctiles, smem + prologue * kQBufBytes, &full[prologue], lane);
  }

  const bool rows = p.q != nullptr, cols = p.qT != nullptr;
  const int rj = lane >> 1, rh = lane & 1;   // row view: row 16w + rj, chunks 2m + rh
  const int cq = lane & 3, rg = lane >> 2;   // column view: columns 16w + 4cq.., rows 16rg..
  const int wrow = 16 * warp + rj;
  uint32_t j = 0;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, ++j) {
    const uint32_t s = j % kQStages, ph = (j / kQStages) & 1u;
    if (!mbar_wait(&full[s], ph, p.wait_ns, kWeight ? 0x201u : 0x101u)) break;
    const uint8_t* buf = smem + s * kQBufBytes;
    const int64_t r0 = (t / ctiles) * 128, c0 = (t % ctiles) * 128;

    // both slices into registers, then hand the slot back
    uint4 rv[8];
    uint2 cv[16];
    if (rows) {
      const uint8_t* rp = buf + qrow_off(wrow);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        rv[2 * m] = *reinterpret_cast<const uint4*>(rp + (2 * (2 * m + rh)) * 16);
        rv[2 * m + 1] = *reinterpret_cast<const uint4*>(rp + (2 * (2 * m + rh) + 1) * 16);
      }
    }
    if (cols) {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        cv[k] = *reinterpret_cast<const uint2*>(buf + qrow_off(16 * rg + k) + 32 * warp + 8 * cq);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0 && j >= 1) {
      // Refill the slot of tile j-1 (every warp released it, usually long
      // ago) with tile j-1+kQStages.
      const int64_t tn = t + (kQStages - 1) * static_cast<int64_t>(gridDim.x);
      if (tn < tiles) {
        const uint32_t f = j - 1, sf = f % kQStages;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[sf], (f / kQStages) & 1u, p.wait_ns, kWeight ? 0x211u : 0x111u);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        quant_fill(p, tn, ctiles, smem + sf * kQBufBytes, &full[sf], lane);
        last_issued = f + kQStages;
      }
    }

    // amaxes (packed bf16, NaN ignored)
    float row_m = 0.0f;
    uint32_t m01 = 0u, m23 = 0u;
    if (rows) {
      uint32_t m2 = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        m2 = bf16x2_maxabs(bf16x2_maxabs(m2, bf16x2_maxabs(rv[k].x, rv[k].y)), bf16x2_maxabs(rv[k].z, rv[k].w));
      row_m = bf16x2_absmax(m2);
      row_m = fmaxf(row_m, __shfl_xor_sync(0xffffffffu, row_m, 1));
    }
    if (cols) {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        m01 = bf16x2_maxabs(m01, cv[k].x);
        m23 = bf16x2_maxabs(m23, cv[k].y);
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        m01 = bf16x2_maxabs(m01, __shfl_xor_sync(0xffffffffu, m01, o));
        m23 = bf16x2_maxabs(m23, __shfl_xor_sync(0xffffffffu, m23, o));
      }
    }

    GroupScale grow, gcol;  // this lane's row group; column 4cq + rg%4 (scales of the other columns by shuffle)
    if constexpr (kWeight) {
      // one block: every warp's maxima meet in shared memory.  Slot j%2 is
      // reused two tiles later, when every warp has read it (a warp arrives
      // for tile j+1 only after reading slot j%2).
      float m = rows ? row_m : fmaxf(bf16x2_absmax(m01), bf16x2_absmax(m23));
      m = warp_max(m);
      float* rbuf = red + (j & 1u) * kQComputeWarps;
      if (lane == 0) {
        rbuf[warp] = m;
        mbar_arrive(&redbar[j & 1u]);
      }
      if (!mbar_wait(&redbar[j & 1u], (j >> 1) & 1u, p.wait_ns, 0x221u)) break;
      float bm = rbuf[0];
#pragma unroll
      for (int k = 1; k < kQComputeWarps; ++k) bm = fmaxf(bm, rbuf[k]);
      grow = make_group_scale(bm);
      gcol = grow;
      if (threadIdx.x == 0) p.s[(r0 / 128) * (p.C / 128) + c0 / 128] = grow.s;
    } else {
      if (rows) {
        grow = make_group_scale(row_m);
        if (rh == 0) p.s[(c0 / 128) * p.R + r0 + wrow] = grow.s;
      }
      if (cols) {
        const int sel = rg & 3;
        const uint32_t mw = sel < 2 ? m01 : m23;
        gcol = make_group_scale(fabsf((sel & 1) ? bf16hi(mw) : bf16lo(mw)));
        if (rg < 4) p.sT[(r0 / 128) * p.C + c0 + 16 * warp + 4 * cq + rg] = gcol.s;
      }
    }

    // codes
    if (rows) {
      uint8_t* qrow = p.q + (r0 + wrow) * p.C + c0;
#pragma unroll
      for (int m = 0; m < 4; ++m)
        *reinterpret_cast<uint4*>(qrow + (2 * m + rh) * 16) = quant16(rv[2 * m], rv[2 * m + 1], grow);
    }
    if (cols) {
      // the scales of this lane's 4 columns live in lanes cq + 4k
      GroupScale gc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (kWeight) {
          gc[k] = gcol;
        } else {
          gc[k].s = __shfl_sync(0xffffffffu, gcol.s, cq + 4 * k);
          gc[k].r = __shfl_sync(0xffffffffu, gcol.r, cq + 4 * k);
          gc[k].exact = __shfl_sync(0xffffffffu, gcol.exact, cq + 4 * k);
        }
      }
      uint8_t* qcol = p.qT + (c0 + 16 * warp + 4 * cq) * p.R + r0 + 16 * rg;
      *reinterpret_cast<uint4*>(qcol) = quant_col16<0, 0>(cv, gc[0]);
      *reinterpret_cast<uint4*>(qcol + p.R) = quant_col16<0, 1>(cv, gc[1]);
      *reinterpret_cast<uint4*>(qcol + 2 * p.R) = quant_col16<1, 0>(cv, gc[2]);
      *reinterpret_cast<uint4*>(qcol + 3 * p.R) = quant_col16<1, 1>(cv, gc[3]);
    }
  }
  // Leave no copy in flight into this CTA's shared memory: after an early
  // exit at local tile j, warp 0 (which issues every copy) waits (bounded)
  // for the tiles >= j it issued, at most kQStages of them.  No later fill
  // of those slots can have been issued (that needs every warp to release
  // the tile), so the waited phase is the one of that tile.  After a normal
  // exit j counts all tiles of the CTA and nothing is waited for.
  if (warp == 0 && lane == 0) {
    const int64_t last = last_issued > static_cast<int64_t>(prologue) - 1 ? last_issued : static_cast<int64_t>(prologue) - 1;
    for (int64_t k = j; k <= last; ++k)
      mbar_wait(&full[k % kQStages], (k / kQStages) & 1u, p.wait_ns, kWeight ? 0x212u : 0x112u);
  }
}

}  // namespace bfp8
