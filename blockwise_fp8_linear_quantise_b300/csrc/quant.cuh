// E4M3 quantisers: 1x128 activation groups (along the columns, and along
// the rows with transposed storage) and 128x128 weight blocks.
//
// Numerics follow "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within
// $5090", section 3.2: one scale per 128 consecutive values along the GEMM
// reduction dimension for activations and activation gradients, one per
// 128x128 block for weights, each computed online from its own values.
// Per group: amax = max|x| (fmaxf, NaN ignored); s = amax/448 in IEEE fp32
// (1 when amax == 0); q = E4M3_rn_satfinite(fp32_rn(x / s)).  The codes are
// taken from x times the rounded reciprocal of s wherever that provably gives
// the same code, else from the IEEE division (GroupScale / quant_pair), so
// codes and scales are fully determined and match a plain CPU evaluation bit
// for bit.
//
// Work decomposition: one CTA per 128x128 tile of the bf16 input.  The tile
// (32 KB) arrives in shared memory by 128 bulk copies of one 256-byte row
// each; the CTA then
//   * row pass:    each warp takes whole tile rows; a lane holds 4 values,
//                  a 5-step shuffle gives the row-group amax; codes leave as
//                  one coalesced 128-byte store per row;
//   * column pass: each thread holds a column pair over 32 rows in registers;
//                  4 partial amaxes per column meet in shared memory; the
//                  transposed codes are staged in a swizzled [128][128] byte
//                  tile and leave as coalesced 16-byte stores.
// The input is read from HBM once whichever outputs are requested, so the
// dual quantiser moves 2 B in + 2 B out (+ scales) per element.
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

constexpr int kQuantThreads = 256;
constexpr int kQTileBytes = 128 * 256;                       // bf16 tile
constexpr int kQTileTOff = kQTileBytes;                      // [128][128] codes
constexpr int kQColMaxOff = kQTileTOff + 128 * 128;          // float[4][128]
constexpr int kQColScaleOff = kQColMaxOff + 4 * 128 * 4;     // float[128]
constexpr int kQRowScaleOff = kQColScaleOff + 128 * 4;       // float[128]
constexpr int kQRedOff = kQRowScaleOff + 128 * 4;            // float[8]
constexpr int kQBarOff = kQRedOff + 8 * 4;                   // uint64
constexpr int kQuantSmemBytes = kQBarOff + 16;

// Writes the 32 codes of one column (32 consecutive rows of the tile) into
// row `trow` of the transposed staging tile.  16-byte chunk c of a staging
// row is stored at chunk c ^ ((trow >> 1) & 7), which keeps both the writes
// here (8 lanes -> 8 rows 2 apart) and the row-wise reads conflict-free.
__device__ __forceinline__ void stage_t_row(uint8_t* tileT, int trow, int rq, const uint32_t (&pk)[8]) {
  const int sw = (trow >> 1) & 7;
  uint8_t* row = tileT + trow * 128;
  *reinterpret_cast<uint4*>(row + (((2 * rq) ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  *reinterpret_cast<uint4*>(row + (((2 * rq + 1) ^ sw) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// Quantises the column pair held in w[] (32 rows, low half = column 2cp,
// high half = column 2cp+1) with group scales g0/g1 and stages both code rows.
__device__ __forceinline__ void quant_column_pair(uint8_t* tileT, int cp, int rq, const uint32_t (&w)[32],
                                                  const GroupScale& g0, const GroupScale& g1) {
  uint32_t pk0[8], pk1[8];
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const uint32_t a01 = quant_pair(bf16lo(w[i]), bf16lo(w[i + 1]), g0);
    const uint32_t a23 = quant_pair(bf16lo(w[i + 2]), bf16lo(w[i + 3]), g0);
    const uint32_t b01 = quant_pair(bf16hi(w[i]), bf16hi(w[i + 1]), g1);
    const uint32_t b23 = quant_pair(bf16hi(w[i + 2]), bf16hi(w[i + 3]), g1);
    pk0[i / 4] = a01 | (a23 << 16);
    pk1[i / 4] = b01 | (b23 << 16);
  }
  stage_t_row(tileT, 2 * cp, rq, pk0);
  stage_t_row(tileT, 2 * cp + 1, rq, pk1);
}

// Copies the staged transposed codes to out[(c0 + row) * ld + r0 + ...].
__device__ __forceinline__ void store_t_tile(const uint8_t* tileT, uint8_t* out, int64_t ld, int64_t c0, int64_t r0,
                                             int tid) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = tid + kQuantThreads * j;
    const int row = idx >> 3, ch = idx & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(tileT + row * 128 + ((ch ^ ((row >> 1) & 7)) << 4));
    *reinterpret_cast<uint4*>(out + (c0 + row) * ld + r0 + ch * 16) = v;
  }
}

// Quantises one tile row (128 values) held as 4 values per lane; returns
// the 4 codes packed.  The group scale is already known.
__device__ __forceinline__ uint32_t quant4(uint2 v, const GroupScale& g) {
  return quant_pair(bf16lo(v.x), bf16hi(v.x), g) | (quant_pair(bf16lo(v.y), bf16hi(v.y), g) << 16);
}

__device__ __forceinline__ float amax4(uint2 v) {
  return fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))), fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))));
}

// kWeight = false: activation groups (rows -> q/s, columns -> qT/sT).
// kWeight = true : one 128x128 block per tile (q and/or qT, one scale).
template <bool kWeight>
__global__ void __launch_bounds__(kQuantThreads) quantize_tile_kernel(const QuantParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tile = smem;
  uint8_t* tileT = smem + kQTileTOff;
  float* colmax = reinterpret_cast<float*>(smem + kQColMaxOff);
  float* colscale = reinterpret_cast<float*>(smem + kQColScaleOff);  // column amax
  float* rowscale = reinterpret_cast<float*>(smem + kQRowScaleOff);
  float* red = reinterpret_cast<float*>(smem + kQRedOff);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kQBarOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) mbar_arrive_expect_tx(bar, kQTileBytes);
    __syncwarp();
    for (int i = lane; i < 128; i += 32) bulk_g2s(tile + i * 256, p.x + (r0 + i) * p.C + c0, 256, bar);
  }
  const bool ok = mbar_wait(bar, 0, p.wait_ns, kWeight ? 0x201u : 0x101u);
  if (__syncthreads_or(!ok)) return;

  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(tile);
  const int cp = tid & 63, rq = tid >> 6;

  if constexpr (!kWeight) {
    if (p.q != nullptr) {
      for (int rr = warp; rr < 128; rr += kQuantThreads / 32) {
        const uint2 v = *reinterpret_cast<const uint2*>(tile + rr * 256 + lane * 8);
        const GroupScale g = make_group_scale(warp_max(amax4(v)));
        *reinterpret_cast<uint32_t*>(p.q + (r0 + rr) * p.C + c0 + lane * 4) = quant4(v, g);
        if (lane == 0) rowscale[rr] = g.s;
      }
    }
    if (p.qT != nullptr) {
      uint32_t w[32];
      float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        w[i] = t32[(rq * 32 + i) * 64 + cp];
        m0 = fmaxf(m0, fabsf(bf16lo(w[i])));
        m1 = fmaxf(m1, fabsf(bf16hi(w[i])));
      }
      colmax[rq * 128 + 2 * cp] = m0;
      colmax[rq * 128 + 2 * cp + 1] = m1;
      __syncthreads();
      if (tid < 128) {
        // colscale holds the column amax; every thread derives the same scale from it
        const float m = fmaxf(fmaxf(colmax[tid], colmax[128 + tid]), fmaxf(colmax[256 + tid], colmax[384 + tid]));
        colscale[tid] = m;
        p.sT[(r0 / 128) * p.C + c0 + tid] = group_scale(m);
      }
      __syncthreads();
      quant_column_pair(tileT, cp, rq, w, make_group_scale(colscale[2 * cp]), make_group_scale(colscale[2 * cp + 1]));
    }
    __syncthreads();
    if (p.q != nullptr && tid < 128) p.s[(c0 / 128) * p.R + r0 + tid] = rowscale[tid];
    if (p.qT != nullptr) store_t_tile(tileT, p.qT, p.R, c0, r0, tid);
  } else {
    uint32_t w[32];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      w[i] = t32[(rq * 32 + i) * 64 + cp];
      m = fmaxf(m, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    }
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float bm = red[0];
#pragma unroll
    for (int i = 1; i < kQuantThreads / 32; ++i) bm = fmaxf(bm, red[i]);
    const GroupScale g = make_group_scale(bm);
    if (tid == 0) p.s[(r0 / 128) * (p.C / 128) + c0 / 128] = g.s;
    if (p.q != nullptr) {
      for (int rr = warp; rr < 128; rr += kQuantThreads / 32) {
        const uint2 v = *reinterpret_cast<const uint2*>(tile + rr * 256 + lane * 8);
        *reinterpret_cast<uint32_t*>(p.q + (r0 + rr) * p.C + c0 + lane * 4) = quant4(v, g);
      }
    }
    if (p.qT != nullptr) {
      quant_column_pair(tileT, cp, rq, w, g, g);
      __syncthreads();
      store_t_tile(tileT, p.qT, p.R, c0, r0, tid);
    }
  }
}

}  // namespace bfp8
