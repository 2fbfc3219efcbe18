// GEMM of the MXFP8 1x32 recipe: C = A . B^T with E4M3 operands whose
// scales belong to groups of 32 consecutive reduction indices, one per row of
// A and one per row of B (bloombook.cn tutorial, FP8 paragraph and MXFP
// concept figure: every 32 elements share one scale X, V_i = Q_i X):
//
//   C[i, j] = bf16( sum over 32-deep slices t of P_t[i, j] * sa(i, t) * sb(j, t) )
//
// with P_t the exact-order-free tensor-core fp32 sum of the slice's 32
// products, promoted in fp32 slice by slice, as the 1x128 GEMM promotes its
// 128-deep slices.  It is the comparison workload of the blockwise recipe;
// with these power-of-two scales the tensor core's own block-scaled MMA could
// apply them, but its instruction-descriptor and scale-factor layouts are not
// documented where this library was written, so each 32-deep partial leaves
// the tensor core and is promoted on CUDA cores (four times the promotion
// work of the 1x128 GEMM per element).
//
// Structure: the 1x128 kernel's warp roles on single-CTA 128 x 128 tiles.
// Each TMA stage holds a 128-deep slice of A and B; the MMA warp issues its
// four K = 32 sub-slices into four separate TMEM buffers of 128 columns (the
// whole 512 columns), and the promotion warps take them in order with the
// column layout of the WGRAD promotion (16x256b loads; thread t owns rows
// 16h + 8i + t/4 and columns 8j + 2 (t%4) + {0, 1} of its warp's 32 x 64),
// both 16-lane halves loaded before the buffer is handed back.  The producer
// stores each stage's 4 x 128 row scales and 4 x 128 column scales (the latter
// in the threads' reading order) in a scale slot.
#pragma once

#include <cuda.h>
#include "common.cuh"
#include "gemm.cuh"

namespace bfp8 {

struct MxSmem {
  static constexpr int kStages = 4;
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = 128 * 128;
  static constexpr int kAOff = 0;
  static constexpr int kBOff = kStages * kABytes;
  static constexpr int kCOff = kBOff + kStages * kBBytes;  // 1024-aligned
  static constexpr int kCWarpBytes = 2048;                 // 32 rows x 32 bf16, 64-byte swizzle
  static constexpr int kSbStride = 128 / 8 + 4;            // a thread column pair's 16 scales, padded
  static constexpr int kSubSaFloats = 128;
  static constexpr int kSubSbFloats = 8 * kSbStride;
  static constexpr int kSlotFloats = 4 * (kSubSaFloats + kSubSbFloats);
  static constexpr int kScaleSlots = kStages + 2;
  static constexpr int kScaleOff = kCOff + 8 * kCWarpBytes;
  static constexpr int kBarOff = kScaleOff + kScaleSlots * kSlotFloats * 4;
  // full[S], empty[S], tfull[4], tempty[4], done, sfull[slots], sempty[slots], stall
  static constexpr int kNumBars = 2 * kStages + 9 + 2 * kScaleSlots + 1;
  static constexpr int kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kTmemSlotOff + 16;
  static constexpr int kAlloc = kBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;  // four 128-column buffers
  static_assert(kAlloc <= 232448, "MX GEMM shared memory exceeds the per-CTA limit");
};

// p.sa: [K/32, M] (row scales of A); p.sb: [K/32, N] (row scales of B); C bf16
// [M, N]; p.kps = K/128 (one work unit per 128 x 128 output tile).
__global__ void __launch_bounds__(kGemmThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  using L = MxSmem;
  constexpr int kStages = L::kStages, kSlots = L::kScaleSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;        // TMEM buffer t % 4 holds sub-slice t
  uint64_t* tempty = bars + 2 * kStages + 4;
  uint64_t* done = bars + 2 * kStages + 8;
  uint64_t* sfull = bars + 2 * kStages + 9;
  uint64_t* sempty = sfull + kSlots;
  uint64_t* stall = sempty + kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOff);
  float* scales = reinterpret_cast<float*>(smem + L::kScaleOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit0 = blockIdx.x, unit_step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);
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
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp >= kProducerWarp) {
    setmaxnreg_dec<kSmallRegs>();
    if (warp == kProducerWarp) {
      // ---------------------------------------------------------- producer
      uint32_t it = 0;
      bool ok = true;
      if (p.stall != 0u) ok = mbar_wait(stall, 0, p.wait_ns, 0x500u);
      for (int u = unit0; u < p.units && ok; u += unit_step) {
        const UnitCoords c = unit_coords(p, u);
        for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
          const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
          const uint32_t q = it % kSlots, qph = (it / kSlots) & 1u;
          bool w_ok = true;
          if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1u, p.wait_ns, 0x501u);
          w_ok = mbar_wait(&sempty[q], qph ^ 1u, p.wait_ns, 0x503u) && w_ok;
          if (!__all_sync(0xffffffffu, w_ok)) {
            ok = false;
            break;
          }
          float* slot = scales + q * L::kSlotFloats;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int64_t t = 4 * static_cast<int64_t>(kb) + jj;  // 32-deep slice
            float* sa_sub = slot + jj * (L::kSubSaFloats + L::kSubSbFloats);
            cp_async16(sa_sub + 4 * lane, p.sa + t * p.M + c.m0 + 4 * lane);
            // columns (col, col + 1) go to the run of warp half col / 64 and
            // thread column pair (col % 8) / 2, position 2 (col % 64) / 8
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const int col = 2 * (32 * r + lane);
              const int cc = col % 64;
              const int dst = ((col / 64) * 4 + (cc % 8) / 2) * L::kSbStride + 2 * (cc / 8);
              cp_async8(sa_sub + L::kSubSaFloats + dst, p.sb + t * p.N + c.nt * 128 + col);
            }
          }
          cp_async_arrive(&sfull[q]);
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], L::kABytes + L::kBBytes);
            tma_load_2d(smem + L::kAOff + s * L::kABytes, &tmA, kb * 128, c.m0, &full[s]);
            tma_load_2d(smem + L::kBOff + s * L::kBBytes, &tmB, kb * 128, c.nt * 128, &full[s]);
          }
          __syncwarp();
        }
      }
      cp_async_wait_all();
      if (lane == 0) {
        for (uint32_t j = 0; j < kStages && j < it; ++j) {
          const uint32_t f = it - 1 - j;
          mbar_wait(&full[f % kStages], (f / kStages) & 1u, kDrainWaitNs, 0x502u);
        }
      }
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------- MMA issue
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_e4m3_f32(128, 128);
        uint32_t it = 0;
        bool ok = true;
        for (int u = unit0; u < p.units && ok; u += unit_step) {
          const UnitCoords c = unit_coords(p, u);
          for (int kb = c.kb0; kb < c.kb1 && ok; ++kb, ++it) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
            if (!mbar_wait(&full[s], ph, p.wait_ns, 0x512u)) {
              ok = false;
              break;
            }
            const uint32_t a_addr = smem_u32(smem + L::kAOff + s * L::kABytes);
            const uint32_t b_addr = smem_u32(smem + L::kBOff + s * L::kBBytes);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              // sub-slice t = 4 it + jj into buffer jj; its previous use was t - 4
              if (!mbar_wait(&tempty[jj], (it & 1u) ^ 1u, p.wait_ns, 0x511u)) {
                ok = false;
                break;
              }
              tc_fence_after();
              mma_e4m3(tmem_base + 128 * jj, sw128_kmajor_desc(a_addr + 32 * jj), sw128_kmajor_desc(b_addr + 32 * jj),
                       idesc, 0u);
              mma_commit(&tfull[jj]);
            }
            if (!ok) break;
            mma_commit(&empty[s]);
          }
        }
        mma_commit(done);
        mbar_wait(done, 0, kDrainWaitNs, 0x513u);
      }
    }
  } else {
    setmaxnreg_inc<kBigRegs>();
    // ------------------------------------------------------------ promotion
    const int quad = warp & 3, half = warp >> 2;
    const int tq = lane & 3, tr = lane >> 2;
    uint32_t it = 0;
    bool ok = true;
    float acc[64];  // acc[32 h + 4 j + 2 i + e]: row 16h + 8i + t/4, column 8j + 2 (t%4) + e
    for (int u = unit0; u < p.units && ok; u += unit_step) {
      const UnitCoords c = unit_coords(p, u);
      const int row0 = c.m0 + quad * 32;
      const int col0 = c.nt * 128 + half * 64;
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      for (int kb = c.kb0; kb < c.kb1 && ok; ++kb, ++it) {
        const uint32_t q = it % kSlots, qph = (it / kSlots) & 1u;
        if (!mbar_wait(&sfull[q], qph, p.wait_ns, 0x522u)) {
          ok = false;
          break;
        }
        const float* slot = scales + q * L::kSlotFloats;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (!mbar_wait(&tfull[jj], it & 1u, p.wait_ns, 0x521u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t v[2][32];
          const uint32_t ta = tmem_base + 128 * jj + half * 64;
          tmem_ld16x256b_x8(ta + (static_cast<uint32_t>(quad * 32) << 16), v[0]);
          tmem_ld16x256b_x8(ta + (static_cast<uint32_t>(quad * 32 + 16) << 16), v[1]);
          tmem_wait_ld32(v[0]);
          tmem_wait_ld32(v[1]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[jj]);  // both halves are in registers
          const float* sub = slot + jj * (L::kSubSaFloats + L::kSubSbFloats);
          float sa_r[4];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) sa_r[rr] = sub[quad * 32 + 16 * (rr >> 1) + 8 * (rr & 1) + tr];
          const float4* sb4 = reinterpret_cast<const float4*>(sub + L::kSubSaFloats + (half * 4 + tq) * L::kSbStride);
          float2 sbp[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 t = sb4[k];
            sbp[2 * k] = make_float2(t.x, t.y);
            sbp[2 * k + 1] = make_float2(t.z, t.w);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const float2 sc = fmul2(make_float2(sa_r[2 * h + i], sa_r[2 * h + i]), sbp[j]);
                float* a = acc + 32 * h + 4 * j + 2 * i;
                const float2 r = ffma2(make_float2(__uint_as_float(v[h][4 * j + 2 * i]),
                                                   __uint_as_float(v[h][4 * j + 2 * i + 1])),
                                       sc, make_float2(a[0], a[1]));
                a[0] = r.x;
                a[1] = r.y;
              }
            }
            reg_fence32(acc + 32 * h);
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[q]);
      }
      if (!ok) break;

      // epilogue: bf16 through the warp's 2 KB staging area (64-byte swizzle),
      // one TMA box of 32 rows x 32 columns per pass
      uint8_t* stg = smem + L::kCOff + warp * L::kCWarpBytes;
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t r = 16 * h + 8 * i + tr, sw = (r >> 1) & 3u;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const float* a = acc + 32 * h + 4 * (4 * ps + g) + 2 * i;
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(a[0], a[1]);
              *reinterpret_cast<uint32_t*>(stg + r * 64 + ((static_cast<uint32_t>(g) ^ sw) << 4) + 4 * tq) =
                  *reinterpret_cast<const uint32_t*>(&h2);
            }
          }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmC, stg, col0 + 32 * ps, row0);
          bulk_commit_group();
        }
      }
    }
  }

  if (warp < kProducerWarp && lane == 0) bulk_wait_group<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

}  // namespace bfp8
