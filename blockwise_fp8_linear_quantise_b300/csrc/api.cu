// C ABI of the blockwise-FP8 linear layer: argument validation, tensor-map
// encoding, launch configuration and the fused linear forward/backward.
// All kernels live in this single translation unit (quant.cuh, gemm.cuh) so
// the device error word has one definition per loaded module.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/bfp8.h"
#include "common.cuh"
#include "gemm.cuh"
#include "quant.cuh"
#include "gemm_mx.cuh"

namespace {

using namespace bfp8;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int pair_clusters = 0;  // co-resident clusters of the CTA-pair GEMM (0: not usable)
  uint64_t wait_ns = kDefaultWaitNs;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
// Process-wide tuning knobs: read by every planning call, possibly from
// several host threads at once, so they are atomics.
std::atomic<int> g_forced_splits{0};  // 0 = automatic
std::atomic<int> g_gemm_kind{0};      // 0 = CTA pairs where the shape allows, 1 = single-CTA tiles only
std::atomic<uint64_t> g_launches{0};  // kernels launched by this library
std::atomic<int> g_stall_next{0};     // test hook: the next quantiser or GEMM launch stalls (bounded)

uint32_t take_stall() { return g_stall_next.exchange(0, std::memory_order_relaxed) != 0 ? 1u : 0u; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bfp8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BFP8_OK : BFP8_ECUDA; }

// Looks up the current device, checks it is an sm_103 part and sets the
// kernels' shared-memory limits once.
bfp8_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BFP8_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return BFP8_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return BFP8_ECUDA;
    if (major != 10 || minor != 3) return BFP8_EUNSUPPORTED;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return BFP8_ECUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    cudaError_t e = cudaSuccess;
    // two quantiser CTAs per SM need the largest shared-memory carveout
#define BFP8_SET_QUANT_SMEM_GLU(W, MODE, SCALE, GLU, BYTES)                                               \
  if (e == cudaSuccess)                                                                                     \
    e = cudaFuncSetAttribute(quantize_tile_kernel<W, MODE, SCALE, GLU>,                                     \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES);                           \
  if (e == cudaSuccess)                                                                                     \
    e = cudaFuncSetAttribute(quantize_tile_kernel<W, MODE, SCALE, GLU>,                                     \
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
#define BFP8_SET_QUANT_SMEM(W, MODE, SCALE) BFP8_SET_QUANT_SMEM_GLU(W, MODE, SCALE, false, kQuantSmemBytes)
#define BFP8_SET_QUANT_SMEM_ALL(SCALE)                  \
  BFP8_SET_QUANT_SMEM(false, kQRows, SCALE)             \
  BFP8_SET_QUANT_SMEM(false, kQCols, SCALE)             \
  BFP8_SET_QUANT_SMEM(false, kQRows | kQCols, SCALE)    \
  BFP8_SET_QUANT_SMEM(true, kQRows, SCALE)              \
  BFP8_SET_QUANT_SMEM(true, kQCols, SCALE)              \
  BFP8_SET_QUANT_SMEM(true, kQRows | kQCols, SCALE)
    BFP8_SET_QUANT_SMEM_ALL(kScaleAmax448)
    BFP8_SET_QUANT_SMEM_ALL(kScalePow2)
    BFP8_SET_QUANT_SMEM_ALL(kScaleMulRecip)
    BFP8_SET_QUANT_SMEM(false, kQRows, kScaleMx32)
    BFP8_SET_QUANT_SMEM(false, kQCols, kScaleMx32)
    BFP8_SET_QUANT_SMEM(false, kQRows | kQCols, kScaleMx32)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MxSmem::kAlloc);
#undef BFP8_SET_QUANT_SMEM_ALL
#define BFP8_SET_WBATCH_SMEM(MODE, SCALE)                                                                \
  if (e == cudaSuccess)                                                                                  \
    e = cudaFuncSetAttribute(quantize_w_batch_kernel<MODE, SCALE>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             kQuantSmemBytes);                                                           \
  if (e == cudaSuccess)                                                                                  \
    e = cudaFuncSetAttribute(quantize_w_batch_kernel<MODE, SCALE>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
#define BFP8_SET_WBATCH_SMEM_ALL(SCALE)        \
  BFP8_SET_WBATCH_SMEM(kQRows, SCALE)          \
  BFP8_SET_WBATCH_SMEM(kQCols, SCALE)          \
  BFP8_SET_WBATCH_SMEM(kQRows | kQCols, SCALE)
    BFP8_SET_WBATCH_SMEM_ALL(kScaleAmax448)
    BFP8_SET_WBATCH_SMEM_ALL(kScalePow2)
    BFP8_SET_WBATCH_SMEM_ALL(kScaleMulRecip)
#undef BFP8_SET_WBATCH_SMEM_ALL
#undef BFP8_SET_WBATCH_SMEM
    // the SiLU-gated prologue#undef BFP8_SET_QUANT_SMEM_ALL
    // the SiLU-gated prologue: one CTA per SM with two tiles per ring slot
#define BFP8_SET_GLU_SMEM_ALL(SCALE)                                                      \
  BFP8_SET_QUANT_SMEM_GLU(false, kQRows, SCALE, true, kQuantGluSmemBytes)                 \
  BFP8_SET_QUANT_SMEM_GLU(false, kQCols, SCALE, true, kQuantGluSmemBytes)                 \
  BFP8_SET_QUANT_SMEM_GLU(false, kQRows | kQCols, SCALE, true, kQuantGluSmemBytes)
    BFP8_SET_GLU_SMEM_ALL(kScaleAmax448)
    BFP8_SET_GLU_SMEM_ALL(kScalePow2)
    BFP8_SET_GLU_SMEM_ALL(kScaleMulRecip)
#undef BFP8_SET_GLU_SMEM_ALL
#undef BFP8_SET_QUANT_SMEM
#undef BFP8_SET_QUANT_SMEM_GLU
#define BFP8_SET_GEMM_SMEM(BN, MODE, EPI)                                                                     \
  if (e == cudaSuccess)                                                                                        \
    e = cudaFuncSetAttribute(block_gemm_kernel<BN, MODE, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             gemm_smem_alloc<BN, false, MODE, EPI>());
    BFP8_SET_GEMM_SMEM(256, kSbBlock, kEpiPlain)
    BFP8_SET_GEMM_SMEM(256, kSbBlockT, kEpiPlain)
    BFP8_SET_GEMM_SMEM(256, kSbCol, kEpiPlain)
    BFP8_SET_GEMM_SMEM(256, kSbBlock, kEpiCodes)
    BFP8_SET_GEMM_SMEM(256, kSbBlockT, kEpiCodes)
    BFP8_SET_GEMM_SMEM(256, kSbCol, kEpiCodes)
    BFP8_SET_GEMM_SMEM(256, kSbBlock, kEpiAccum)
    BFP8_SET_GEMM_SMEM(256, kSbBlockT, kEpiAccum)
    BFP8_SET_GEMM_SMEM(256, kSbCol, kEpiAccum)
    BFP8_SET_GEMM_SMEM(128, kSbBlock, kEpiPlain)
    BFP8_SET_GEMM_SMEM(128, kSbBlockT, kEpiPlain)
    BFP8_SET_GEMM_SMEM(128, kSbCol, kEpiPlain)
    BFP8_SET_GEMM_SMEM(128, kSbBlock, kEpiAccum)
    BFP8_SET_GEMM_SMEM(128, kSbBlockT, kEpiAccum)
    BFP8_SET_GEMM_SMEM(128, kSbCol, kEpiAccum)
#undef BFP8_SET_GEMM_SMEM
#define BFP8_SET_PAIR_SMEM(MODE, EPI)                                                                        \
  if (e == cudaSuccess)                                                                                       \
    e = cudaFuncSetAttribute(block_gemm_pair_kernel<MODE, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             gemm_smem_alloc<256, true, MODE, EPI>());
    BFP8_SET_PAIR_SMEM(kSbBlock, kEpiPlain)
    BFP8_SET_PAIR_SMEM(kSbBlockT, kEpiPlain)
    BFP8_SET_PAIR_SMEM(kSbCol, kEpiPlain)
    BFP8_SET_PAIR_SMEM(kSbBlock, kEpiCodes)
    BFP8_SET_PAIR_SMEM(kSbBlockT, kEpiCodes)
    BFP8_SET_PAIR_SMEM(kSbCol, kEpiCodes)
    BFP8_SET_PAIR_SMEM(kSbBlock, kEpiAccum)
    BFP8_SET_PAIR_SMEM(kSbBlockT, kEpiAccum)
    BFP8_SET_PAIR_SMEM(kSbCol, kEpiAccum)
#undef BFP8_SET_PAIR_SMEM
    if (e != cudaSuccess) return BFP8_ECUDA;
    // The GEMM moves registers between warpgroups with setmaxnreg; that is
    // only safe if each thread really starts with kLaunchRegs registers.
    // Refuse to run a build where it does not (it would wait forever).
#define BFP8_CHECK_REGS(BN, MODE, EPI)                                                  \
  {                                                                                      \
    cudaFuncAttributes fa;                                                               \
    if (cudaFuncGetAttributes(&fa, block_gemm_kernel<BN, MODE, EPI>) != cudaSuccess) \
      return BFP8_ECUDA;                                                                 \
    if (fa.numRegs != kLaunchRegs) return BFP8_EUNSUPPORTED;                             \
  }
    BFP8_CHECK_REGS(256, kSbBlock, kEpiPlain)
    BFP8_CHECK_REGS(256, kSbBlockT, kEpiPlain)
    BFP8_CHECK_REGS(256, kSbCol, kEpiPlain)
    BFP8_CHECK_REGS(256, kSbBlock, kEpiCodes)
    BFP8_CHECK_REGS(256, kSbBlockT, kEpiCodes)
    BFP8_CHECK_REGS(256, kSbCol, kEpiCodes)
    BFP8_CHECK_REGS(256, kSbBlock, kEpiAccum)
    BFP8_CHECK_REGS(256, kSbBlockT, kEpiAccum)
    BFP8_CHECK_REGS(256, kSbCol, kEpiAccum)
    BFP8_CHECK_REGS(128, kSbBlock, kEpiPlain)
    BFP8_CHECK_REGS(128, kSbBlockT, kEpiPlain)
    BFP8_CHECK_REGS(128, kSbCol, kEpiPlain)
    BFP8_CHECK_REGS(128, kSbBlock, kEpiAccum)
    BFP8_CHECK_REGS(128, kSbBlockT, kEpiAccum)
    BFP8_CHECK_REGS(128, kSbCol, kEpiAccum)
#undef BFP8_CHECK_REGS
#define BFP8_CHECK_PAIR_REGS(MODE, EPI)                                                   \
  {                                                                                        \
    cudaFuncAttributes fa;                                                                 \
    if (cudaFuncGetAttributes(&fa, block_gemm_pair_kernel<MODE, EPI>) != cudaSuccess) \
      return BFP8_ECUDA;                                                                   \
    if (fa.numRegs != kLaunchRegs) return BFP8_EUNSUPPORTED;                               \
  }
    BFP8_CHECK_PAIR_REGS(kSbBlock, kEpiPlain)
    BFP8_CHECK_PAIR_REGS(kSbBlockT, kEpiPlain)
    BFP8_CHECK_PAIR_REGS(kSbCol, kEpiPlain)
    BFP8_CHECK_PAIR_REGS(kSbBlock, kEpiCodes)
    BFP8_CHECK_PAIR_REGS(kSbBlockT, kEpiCodes)
    BFP8_CHECK_PAIR_REGS(kSbCol, kEpiCodes)
    BFP8_CHECK_PAIR_REGS(kSbBlock, kEpiAccum)
    BFP8_CHECK_PAIR_REGS(kSbBlockT, kEpiAccum)
    BFP8_CHECK_PAIR_REGS(kSbCol, kEpiAccum)
    {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, mx_gemm_kernel) != cudaSuccess) return BFP8_ECUDA;
      if (fa.numRegs != kLaunchRegs) return BFP8_EUNSUPPORTED;
    }
#undef BFP8_CHECK_PAIR_REGS
    // How many CTA pairs can be resident at once (the persistent pair grid).
    {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(sms - (sms & 1)), 1, 1);
      cfg.blockDim = dim3(kGemmThreads, 1, 1);
      cfg.dynamicSmemBytes = gemm_smem_alloc<256, true, kSbBlock, kEpiPlain>();
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, block_gemm_pair_kernel<kSbBlock>, &cfg) != cudaSuccess) {
        cudaGetLastError();  // clear; the pair GEMM is then not used
        clusters = 0;
      }
      st.pair_clusters = clusters;
    }
    st.sms = sms;
    st.ready = true;
  }
  *out = &st;
  return BFP8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int64_t d) { return d > 0 && d % 128 == 0 && d <= (int64_t(1) << 30); }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// 2-D K-contiguous E4M3 tensor [rows, K], box 128 (K bytes) x box_rows,
// 128-byte swizzle: the shared-memory image is the canonical K-major
// layout the MMA descriptors describe.
bfp8_status make_kmajor_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BFP8_OK : BFP8_ECUDA;
}

// The quantisers' input x [R, C] bf16 seen as the 2-D tensor [R/16, 16 C]
// (row y = input rows 16y..16y+15 side by side), box 64 elements x 8 rows,
// 128-byte swizzle: one box brings 64 columns of 8 input rows 16 apart.
bfp8_status make_quant_tmap(CUtensorMap* map, const void* x, int64_t R, int64_t C) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(16 * C), static_cast<cuuint64_t>(R / 16)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(32 * C)};
  cuuint32_t box[2] = {64, 8};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BFP8_OK : BFP8_ECUDA;
}

// The GEMM epilogue's output tensor maps: 32-row boxes of one 128-byte
// swizzled row each (row layout), or of one 64-byte swizzled row each (the
// column layout's 2 KB staging areas).
//   fp32 [rows, cols] accumulation target: 32 (row layout) or 16 columns;
//   bf16 [rows, cols] output: 64 (row layout) or 32 columns.
bfp8_status make_f32_acc_tmap(CUtensorMap* map, float* base, int64_t rows, int64_t cols, bool col_layout) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {col_layout ? 16u : 32u, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        col_layout ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BFP8_OK : BFP8_ECUDA;
}

bfp8_status make_bf16_store_tmap(CUtensorMap* map, void* base, int64_t rows, int64_t cols, bool col_layout) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {col_layout ? 32u : 64u, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        col_layout ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BFP8_OK : BFP8_ECUDA;
}

struct GemmPlan {
  bool pair;                 // 256 x 256 tiles on CTA pairs
  int bn;
  int m_tiles, n_tiles, tiles;
  int splits, kps;
  int slots;                 // work units that run at once
  size_t ws_bytes;
};

// Picks the tile kind and the split-K factor.  CTA pairs (256 x 256 tiles)
// are used for FPROP and DGRAD when both output dimensions allow them; WGRAD,
// whose per-column scales double the promotion work, runs faster on
// single-CTA 128 x BN tiles, as does any other shape.  Split-K only pays when the tile count leaves SMs idle and
// the extra fp32 partial traffic is small next to the GEMM time; estimate both
// with nominal B300 rates.
GemmPlan plan_gemm(bfp8_layout layout, int64_t M, int64_t N, int64_t K, const DeviceState& d) {
  GemmPlan g;
  const int forced_splits = g_forced_splits.load(std::memory_order_relaxed);
  const int kind = g_gemm_kind.load(std::memory_order_relaxed);
  g.pair = kind != 1 && (layout != BFP8_WGRAD || kind == 2) && d.pair_clusters > 0 && M % 256 == 0 &&
           N % 256 == 0;
  g.bn = (N % 256 == 0) ? 256 : 128;
  g.m_tiles = static_cast<int>(M / (g.pair ? 256 : 128));
  g.n_tiles = static_cast<int>(N / g.bn);
  g.tiles = g.m_tiles * g.n_tiles;
  g.slots = g.pair ? d.pair_clusters : d.sms;
  const int nk = static_cast<int>(K / 128);
  int best = 1;
  if (forced_splits > 0) {
    best = std::min(forced_splits, nk);
  } else if (g.slots > 0) {
    const double t_gemm = 2.0 * M * N * K / 4.0e15;
    double best_t = 1e30;
    for (int s = 1; s <= std::min(nk, 16); ++s) {
      const int units = g.tiles * s;
      const double waves = std::ceil(static_cast<double>(units) / g.slots);
      const double eff = units / (waves * g.slots);
      const double t = t_gemm / eff + (s > 1 ? (static_cast<double>(s) * M * N * 4 * 2 + M * N * 2) / 6.0e12 : 0.0);
      if (t < best_t * 0.97) {
        best_t = t;
        best = s;
      }
    }
  }
  g.kps = (nk + best - 1) / best;
  g.splits = (nk + g.kps - 1) / g.kps;
  g.ws_bytes = g.splits > 1 ? static_cast<size_t>(g.splits) * M * N * sizeof(float) : 0;
  return g;
}

template <int BN, int kEpi>
void launch_gemm_bn_mode(int mode, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const GemmParams& p, int grid, cudaStream_t st) {
  switch (mode) {
    case kSbBlock:
      block_gemm_kernel<BN, kSbBlock, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<BN, false, kSbBlock, kEpi>(), st>>>(ta, tb, tc, p);
      break;
    case kSbBlockT:
      block_gemm_kernel<BN, kSbBlockT, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<BN, false, kSbBlockT, kEpi>(), st>>>(ta, tb, tc, p);
      break;
    default:
      block_gemm_kernel<BN, kSbCol, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<BN, false, kSbCol, kEpi>(), st>>>(ta, tb, tc, p);
      break;
  }
}

// The epilogue kind of a launch: fp32 accumulate with p.Cacc and one split,
// the E4M3 codes with p.Cq (one split, BN = 256 only), bf16 C (or split-K
// partials) otherwise.
int epi_kind(const GemmParams& p) {
  if (p.Cacc != nullptr && p.splits == 1) return kEpiAccum;
  if (p.Cq != nullptr) return kEpiCodes;
  return kEpiPlain;
}

template <int BN>
bfp8_status launch_gemm_bn(int mode, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                           const GemmParams& p, int grid, cudaStream_t st) {
  const int epi = epi_kind(p);
  if (epi == kEpiAccum) {
    launch_gemm_bn_mode<BN, kEpiAccum>(mode, ta, tb, tc, p, grid, st);
  } else if (epi == kEpiCodes) {
    if constexpr (BN == 256)
      launch_gemm_bn_mode<BN, kEpiCodes>(mode, ta, tb, tc, p, grid, st);
    else
      return BFP8_EINVAL;
  } else {
    launch_gemm_bn_mode<BN, kEpiPlain>(mode, ta, tb, tc, p, grid, st);
  }
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError());
}

template <int kEpi>
void launch_gemm_pair_mode(int mode, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                           const GemmParams& p, int grid, cudaStream_t st) {
  switch (mode) {
    case kSbBlock:
      block_gemm_pair_kernel<kSbBlock, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<256, true, kSbBlock, kEpi>(), st>>>(ta, tb, tc, p);
      break;
    case kSbBlockT:
      block_gemm_pair_kernel<kSbBlockT, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<256, true, kSbBlockT, kEpi>(), st>>>(ta, tb, tc, p);
      break;
    default:
      block_gemm_pair_kernel<kSbCol, kEpi>
          <<<grid, kGemmThreads, gemm_smem_alloc<256, true, kSbCol, kEpi>(), st>>>(ta, tb, tc, p);
      break;
  }
}

bfp8_status launch_gemm_pair(int mode, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                             const GemmParams& p, int grid, cudaStream_t st) {
  const int epi = epi_kind(p);
  if (epi == kEpiAccum)
    launch_gemm_pair_mode<kEpiAccum>(mode, ta, tb, tc, p, grid, st);
  else if (epi == kEpiCodes)
    launch_gemm_pair_mode<kEpiCodes>(mode, ta, tb, tc, p, grid, st);
  else
    launch_gemm_pair_mode<kEpiPlain>(mode, ta, tb, tc, p, grid, st);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError());
}

// Persistent quantiser grid: two CTAs per SM (each streams its tiles
// through a 3-deep shared-memory ring).  The tile walk and the TMA
// coordinates are 32-bit: C up to 2^27 and fewer than 2^31 tiles.
template <bool kWeight, int kScale, bool kGlu>
bfp8_status launch_quant_mode(const CUtensorMap& tm, const QuantParams& p, unsigned grid, cudaStream_t st) {
  constexpr int kSmem = kGlu ? kQuantGluSmemBytes : kQuantSmemBytes;
  const int mode = (p.q ? kQRows : 0) | (p.qT ? kQCols : 0);
  if (mode == kQRows)
    quantize_tile_kernel<kWeight, kQRows, kScale, kGlu><<<grid, kQuantThreads, kSmem, st>>>(tm, p);
  else if (mode == kQCols)
    quantize_tile_kernel<kWeight, kQCols, kScale, kGlu><<<grid, kQuantThreads, kSmem, st>>>(tm, p);
  else
    quantize_tile_kernel<kWeight, kQRows | kQCols, kScale, kGlu><<<grid, kQuantThreads, kSmem, st>>>(tm, p);
  return BFP8_OK;
}

template <bool kWeight, bool kGlu>
bfp8_status launch_quant_scale(const CUtensorMap& tm, const QuantParams& p, unsigned grid, int scale_mode,
                               cudaStream_t st) {
  if (scale_mode == kScalePow2) return launch_quant_mode<kWeight, kScalePow2, kGlu>(tm, p, grid, st);
  if (scale_mode == kScaleMulRecip) return launch_quant_mode<kWeight, kScaleMulRecip, kGlu>(tm, p, grid, st);
  if constexpr (!kWeight && !kGlu) {
    if (scale_mode == kScaleMx32) return launch_quant_mode<false, kScaleMx32, false>(tm, p, grid, st);
  }
  if (scale_mode == kScaleMx32) return BFP8_EINVAL;
  return launch_quant_mode<kWeight, kScaleAmax448, kGlu>(tm, p, grid, st);
}

// glu: p.x is the gate+up output [R, 2C] and the kernel quantises
// h = bf16(SiLU(g) u) [R, C] (one CTA per SM; row length 2C up to 2^27).
bfp8_status launch_quant(QuantParams p, bool weight, int scale_mode, cudaStream_t st, bool glu = false) {
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  if (p.q == nullptr && p.qT == nullptr) return BFP8_EINVAL;
  if (glu && weight) return BFP8_EINVAL;
  const int64_t tiles = (p.R / 128) * (p.C / 128);
  if (p.C > (int64_t(1) << (glu ? 26 : 27)) || tiles >= (int64_t(1) << 31)) return BFP8_EINVAL;
  p.ctiles = static_cast<uint32_t>(p.C / 128);
  p.tiles = static_cast<uint32_t>(tiles);
  p.stall = take_stall();
  CUtensorMap tm;
  if ((s = make_quant_tmap(&tm, p.x, p.R, glu ? 2 * p.C : p.C)) != BFP8_OK) return s;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, int64_t(dev->sms) * (glu ? 1 : 2)));
  if (glu)
    s = launch_quant_scale<false, true>(tm, p, grid, scale_mode, st);
  else
    s = weight ? launch_quant_scale<true, false>(tm, p, grid, scale_mode, st)
               : launch_quant_scale<false, false>(tm, p, grid, scale_mode, st);
  if (s != BFP8_OK) return s;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError());
}

// C (bf16) is written, or (with Cacc, C null) the result is added into the
// fp32 Cacc; exactly one of the two.
bfp8_status gemm_impl(bfp8_layout layout, const uint8_t* A, const float* sa, const uint8_t* B, const float* sb,
                      int64_t M, int64_t N, int64_t K, void* C, uint8_t* Cq, float* sCq, void* ws, size_t ws_bytes,
                      cudaStream_t stream, float* Cacc = nullptr) {
  if (layout != BFP8_FPROP && layout != BFP8_DGRAD && layout != BFP8_WGRAD) return BFP8_EINVAL;
  if (!A || !sa || !B || !sb || ((C == nullptr) == (Cacc == nullptr))) return BFP8_EINVAL;
  if ((Cq == nullptr) != (sCq == nullptr) || (Cacc && Cq)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(sa) || !aligned16(sb) || (C && !aligned16(C)) ||
      (Cacc && !aligned16(Cacc)) || (Cq && (!aligned16(Cq) || !aligned16(sCq))))
    return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  const GemmPlan g = plan_gemm(layout, M, N, K, *dev);
  if (g.ws_bytes > 0) {
    if (ws == nullptr || ws_bytes < g.ws_bytes) return BFP8_EWORKSPACE;
    if (!aligned16(ws)) return BFP8_EALIGN;
  }
  // The fused quantised epilogue needs a whole 128-column group per thread,
  // which the 256-column tile gives; otherwise the codes come from the
  // split-K reduction or from the row quantiser run on C afterwards.
  const bool fused_here = g.splits == 1 && g.bn == 256;
  // WGRAD promotes in the column layout, except with the fused codes (the
  // kernels' gemm_col_layout()), and its output boxes follow that layout.
  const bool col_layout = layout == BFP8_WGRAD && !(Cq != nullptr && fused_here);
  CUtensorMap ta, tb, tc;
  if ((s = make_kmajor_tmap(&ta, A, M, K, 128)) != BFP8_OK) return s;
  if ((s = make_kmajor_tmap(&tb, B, N, K, g.pair ? g.bn / 2 : g.bn)) != BFP8_OK) return s;
  if ((s = Cacc ? make_f32_acc_tmap(&tc, Cacc, M, N, col_layout) : make_bf16_store_tmap(&tc, C, M, N, col_layout)) !=
      BFP8_OK)
    return s;

  GemmParams p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = g.m_tiles;
  p.n_tiles = g.n_tiles;
  p.tiles = g.tiles;
  p.splits = g.splits;
  p.kps = g.kps;
  p.units = g.tiles * g.splits;
  p.group_m = g.pair ? 8 : 16;
  p.m_tile_rows = g.pair ? 256 : 128;
  p.sa = sa;
  p.sb = sb;
  p.C = static_cast<uint16_t*>(C);
  p.Cacc = Cacc;
  p.Cpart = g.splits > 1 ? static_cast<float*>(ws) : nullptr;
  p.Cq = fused_here ? Cq : nullptr;
  p.sCq = fused_here ? sCq : nullptr;
  p.wait_ns = dev->wait_ns;
  p.stall = take_stall();
  const int mode = layout == BFP8_FPROP ? kSbBlock : (layout == BFP8_DGRAD ? kSbBlockT : kSbCol);
  if (g.pair) {
    s = launch_gemm_pair(mode, ta, tb, tc, p, 2 * std::min(p.units, g.slots), stream);
  } else {
    const int grid = std::min(p.units, dev->sms);
    s = g.bn == 256 ? launch_gemm_bn<256>(mode, ta, tb, tc, p, grid, stream)
                    : launch_gemm_bn<128>(mode, ta, tb, tc, p, grid, stream);
  }
  if (s != BFP8_OK) return s;
  if (g.splits == 1) {
    if (Cq == nullptr || fused_here) return BFP8_OK;  // (Cacc: added by the epilogue)
    QuantParams qp{static_cast<const uint16_t*>(C), M, N, Cq, sCq, nullptr, nullptr, dev->wait_ns, 0u, 0u};
    return launch_quant(qp, false, kScaleAmax448, stream);
  }
  const int64_t groups = M * (N / 128);
  const int rgrid = static_cast<int>(std::min<int64_t>((groups + 7) / 8, int64_t(dev->sms) * 16));
  splitk_reduce_kernel<<<rgrid, 256, 0, stream>>>(static_cast<const float*>(ws), g.splits, p.M, p.N,
                                                   static_cast<uint16_t*>(C), Cq, sCq, Cacc);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError());
}

static_assert(kScaleAmax448 == BFP8_SCALE_AMAX448 && kScalePow2 == BFP8_SCALE_POW2 &&
                  kScaleMulRecip == BFP8_SCALE_MUL_RECIP,
              "kernel scale modes are numbered as the ABI's");
bool scale_mode_ok(int mode) {
  return mode == BFP8_SCALE_AMAX448 || mode == BFP8_SCALE_POW2 || mode == BFP8_SCALE_MUL_RECIP;
}

bfp8_status quant_act_impl(const void* x, int64_t M, int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                           int scale_mode, cudaStream_t stream) {
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!x || (!q && !qT)) return BFP8_EINVAL;
  if ((q && !s) || (qT && !sT)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(K)) return BFP8_EINVAL;
  if (!aligned16(x) || (q && (!aligned16(q) || !aligned16(s))) || (qT && (!aligned16(qT) || !aligned16(sT))))
    return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status st = device_state(&dev);
  if (st != BFP8_OK) return st;
  QuantParams p{static_cast<const uint16_t*>(x), M, K, q, s, qT, sT, dev->wait_ns, 0u, 0u};
  return launch_quant(p, false, scale_mode, stream);
}

bfp8_status swiglu_quant_impl(const void* gu, int64_t M, int64_t F, void* h, uint8_t* q, float* s, uint8_t* qT,
                              float* sT, int scale_mode, cudaStream_t stream) {
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!gu || (!q && !qT)) return BFP8_EINVAL;
  if ((q && !s) || (qT && !sT)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(F)) return BFP8_EINVAL;
  if (!aligned16(gu) || (h && !aligned16(h)) || (q && (!aligned16(q) || !aligned16(s))) ||
      (qT && (!aligned16(qT) || !aligned16(sT))))
    return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status st = device_state(&dev);
  if (st != BFP8_OK) return st;
  QuantParams p{static_cast<const uint16_t*>(gu), M, F, q, s, qT, sT, dev->wait_ns, 0u, 0u,
                static_cast<uint16_t*>(h)};
  return launch_quant(p, false, scale_mode, stream, true);
}

bfp8_status quant_w_impl(const void* w, int64_t N, int64_t K, uint8_t* q, uint8_t* qT, float* s, int scale_mode,
                         cudaStream_t stream) {
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!w || !s || (!q && !qT)) return BFP8_EINVAL;
  if (!dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  if (!aligned16(w) || !aligned16(s) || (q && !aligned16(q)) || (qT && !aligned16(qT))) return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status st = device_state(&dev);
  if (st != BFP8_OK) return st;
  QuantParams p{static_cast<const uint16_t*>(w), N, K, q, s, qT, nullptr, dev->wait_ns, 0u, 0u};
  return launch_quant(p, true, scale_mode, stream);
}

// Launches of the batched weight quantiser, kQBatch jobs at a time; every
// job is checked before the first launch.
template <int kScale>
void launch_quant_w_batch(int mode, const QuantBatchParams& b, unsigned grid, cudaStream_t st) {
  if (mode == kQRows)
    quantize_w_batch_kernel<kQRows, kScale><<<grid, kQuantThreads, kQuantSmemBytes, st>>>(b);
  else if (mode == kQCols)
    quantize_w_batch_kernel<kQCols, kScale><<<grid, kQuantThreads, kQuantSmemBytes, st>>>(b);
  else
    quantize_w_batch_kernel<kQRows | kQCols, kScale><<<grid, kQuantThreads, kQuantSmemBytes, st>>>(b);
}

bfp8_status quant_w_batch_impl(const bfp8_w_job* jobs, int count, int scale_mode, cudaStream_t stream) {
  if (!scale_mode_ok(scale_mode) || jobs == nullptr || count < 1) return BFP8_EINVAL;
  const bool rows = jobs[0].q != nullptr, cols = jobs[0].qT != nullptr;
  for (int i = 0; i < count; ++i) {
    const bfp8_w_job& jb = jobs[i];
    if (!jb.w || !jb.s || (jb.q != nullptr) != rows || (jb.qT != nullptr) != cols || (!rows && !cols))
      return BFP8_EINVAL;
    if (!dim_ok(jb.n) || !dim_ok(jb.k) || jb.k > (int64_t(1) << 27)) return BFP8_EINVAL;
    if (!aligned16(jb.w) || !aligned16(jb.s) || (rows && !aligned16(jb.q)) || (cols && !aligned16(jb.qT)))
      return BFP8_EALIGN;
  }
  DeviceState* dev = nullptr;
  bfp8_status st = device_state(&dev);
  if (st != BFP8_OK) return st;
  const int mode = (rows ? kQRows : 0) | (cols ? kQCols : 0);
  for (int i0 = 0; i0 < count; i0 += kQBatch) {
    QuantBatchParams b{};
    const int n = std::min(kQBatch, count - i0);
    int64_t tiles = 0;
    for (int k = 0; k < n; ++k) {
      const bfp8_w_job& jb = jobs[i0 + k];
      if ((st = make_quant_tmap(&b.tm[k], jb.w, jb.n, jb.k)) != BFP8_OK) return st;
      QuantJob& q = b.job[k];
      q.q = jb.q;
      q.qT = jb.qT;
      q.s = jb.s;
      q.R = jb.n;
      q.C = jb.k;
      q.ctiles = static_cast<uint32_t>(jb.k / 128);
      q.tile0 = static_cast<uint32_t>(tiles);
      tiles += (jb.n / 128) * (jb.k / 128);
      if (tiles >= (int64_t(1) << 31)) return BFP8_EINVAL;
    }
    b.jobs = static_cast<uint32_t>(n);
    b.tiles = static_cast<uint32_t>(tiles);
    b.wait_ns = dev->wait_ns;
    b.stall = take_stall();
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, int64_t(dev->sms) * 2));
    if (scale_mode == kScalePow2)
      launch_quant_w_batch<kScalePow2>(mode, b, grid, stream);
    else if (scale_mode == kScaleMulRecip)
      launch_quant_w_batch<kScaleMulRecip>(mode, b, grid, stream);
    else
      launch_quant_w_batch<kScaleAmax448>(mode, b, grid, stream);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if ((st = cuda_status(cudaGetLastError())) != BFP8_OK) return st;
  }
  return BFP8_OK;
}

// Workspace carving for the fused linear calls: consecutive 256-byte aligned
// regions.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t bytes) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = round_up(off + bytes, 256);
    return p;
  }
};

size_t fwd_ws(int64_t M, int64_t N, int64_t K, const DeviceState& sms, Carver* c, uint8_t** Wq, uint8_t** Xq, float** sX,
              void** gws) {
  Carver local(nullptr);
  Carver& cv = c ? *c : local;
  uint8_t* wq = cv.take<uint8_t>(static_cast<size_t>(N) * K);
  uint8_t* xq = cv.take<uint8_t>(static_cast<size_t>(M) * K);
  float* sx = cv.take<float>(static_cast<size_t>(K / 128) * M * sizeof(float));
  const GemmPlan g = plan_gemm(BFP8_FPROP, M, N, K, sms);
  void* gw = cv.take<uint8_t>(g.ws_bytes);
  if (Wq) *Wq = wq;
  if (Xq) *Xq = xq;
  if (sX) *sX = sx;
  if (gws) *gws = gw;
  return cv.off;
}

size_t bwd_ws(int64_t M, int64_t N, int64_t K, const DeviceState& sms, Carver* c, uint8_t** dYq, float** sdY, uint8_t** dYqT,
              float** sdYT, void** gws) {
  Carver local(nullptr);
  Carver& cv = c ? *c : local;
  uint8_t* a = cv.take<uint8_t>(static_cast<size_t>(M) * N);
  float* b = cv.take<float>(static_cast<size_t>(N / 128) * M * sizeof(float));
  uint8_t* cT = cv.take<uint8_t>(static_cast<size_t>(N) * M);
  float* d = cv.take<float>(static_cast<size_t>(M / 128) * N * sizeof(float));
  const GemmPlan gd = plan_gemm(BFP8_DGRAD, M, K, N, sms);  // dgrad: [M, K], reduction N
  const GemmPlan gw = plan_gemm(BFP8_WGRAD, N, K, M, sms);  // wgrad: [N, K], reduction M
  void* w = cv.take<uint8_t>(std::max(gd.ws_bytes, gw.ws_bytes));
  if (dYq) *dYq = a;
  if (sdY) *sdY = b;
  if (dYqT) *dYqT = cT;
  if (sdYT) *sdYT = d;
  if (gws) *gws = w;
  return cv.off;
}

// The current device's state, or a nominal B300 when it cannot be read (the
// *_workspace_bytes() queries then still answer).
DeviceState current_state() {
  DeviceState* dev = nullptr;
  if (device_state(&dev) == BFP8_OK) return *dev;
  DeviceState d;
  d.sms = 148;
  d.pair_clusters = 74;
  return d;
}

}  // namespace

// ----------------------------------------------------------------------------
// GEMM entry point that allocates nothing: its split-K scratch is a static
// device array of this module.  The array's name in host code is only a
// host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and passed
// to the kernels like any other workspace pointer.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BFP8_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device).
bfp8_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BFP8_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return BFP8_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return BFP8_ECUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return BFP8_OK;
}

}  // namespace

extern "C" {

bfp8_status bfp8_fp8_block_gemm_noalloc(bfp8_layout layout, const uint8_t* A, const float* sa, const uint8_t* B,
                                        const float* sb, int64_t M, int64_t N, int64_t K, void* C, uint8_t* Cq,
                                        float* sCq, bfp8_stream_t stream) {
  if (layout != BFP8_FPROP && layout != BFP8_DGRAD && layout != BFP8_WGRAD) return BFP8_EINVAL;
  if (!A || !sa || !B || !sb || !C || (Cq == nullptr) != (sCq == nullptr)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != BFP8_OK) return s;
  // The split-K partials of these sizes must fit in the static array.
  if (plan_gemm(layout, M, N, K, *dev).ws_bytes > static_cast<size_t>(BFP8_NOALLOC_SCRATCH_BYTES))
    return BFP8_EWORKSPACE;
  return gemm_impl(layout, A, sa, B, sb, M, N, K, C, Cq, sCq, scratch, BFP8_NOALLOC_SCRATCH_BYTES,
                   reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

extern "C" {

bfp8_status bfp8_quantize_act_1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                                    bfp8_stream_t stream) {
  return quant_act_impl(x, M, K, q, s, qT, sT, BFP8_SCALE_AMAX448, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_quantize_w_128x128(const void* w, int64_t N, int64_t K, uint8_t* q, uint8_t* qT, float* s,
                                    bfp8_stream_t stream) {
  return quant_w_impl(w, N, K, q, qT, s, BFP8_SCALE_AMAX448, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_quantize_act_1x128_ex(const void* x, int64_t M, int64_t K, uint8_t* q, float* s, uint8_t* qT,
                                       float* sT, bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  return quant_act_impl(x, M, K, q, s, qT, sT, scale_mode, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_quantize_w_128x128_ex(const void* w, int64_t N, int64_t K, uint8_t* q, uint8_t* qT, float* s,
                                       bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  return quant_w_impl(w, N, K, q, qT, s, scale_mode, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_quantize_w_128x128_batch(const bfp8_w_job* jobs, int count, bfp8_scale_mode scale_mode,
                                          bfp8_stream_t stream) {
  return quant_w_batch_impl(jobs, count, scale_mode, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_swiglu_quantize_1x128(const void* gu, int64_t M, int64_t F, void* h, uint8_t* q, float* s,
                                       uint8_t* qT, float* sT, bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  return swiglu_quant_impl(gu, M, F, h, q, s, qT, sT, scale_mode, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_fp8_block_gemm(bfp8_layout layout, const uint8_t* A, const float* sa, const uint8_t* B,
                                const float* sb, int64_t M, int64_t N, int64_t K, void* C, uint8_t* Cq, float* sCq,
                                void* workspace, size_t ws_bytes, bfp8_stream_t stream) {
  return gemm_impl(layout, A, sa, B, sb, M, N, K, C, Cq, sCq, workspace, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_fp8_block_gemm_accumulate(bfp8_layout layout, const uint8_t* A, const float* sa, const uint8_t* B,
                                           const float* sb, int64_t M, int64_t N, int64_t K, float* C_f32, void* ws,
                                           size_t ws_bytes, bfp8_stream_t stream) {
  if (C_f32 == nullptr) return BFP8_EINVAL;
  return gemm_impl(layout, A, sa, B, sb, M, N, K, nullptr, nullptr, nullptr, ws, ws_bytes,
                   reinterpret_cast<cudaStream_t>(stream), C_f32);
}

bfp8_status bfp8_quantize_mx_1x32(const void* x, int64_t M, int64_t K, uint8_t* q, float* s, uint8_t* qT, float* sT,
                                  bfp8_stream_t stream) {
  if (!x || (!q && !qT) || (q && !s) || (qT && !sT)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(K)) return BFP8_EINVAL;
  if (!aligned16(x) || (q && (!aligned16(q) || !aligned16(s))) || (qT && (!aligned16(qT) || !aligned16(sT))))
    return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status st = device_state(&dev);
  if (st != BFP8_OK) return st;
  QuantParams p{static_cast<const uint16_t*>(x), M, K, q, s, qT, sT, dev->wait_ns, 0u, 0u};
  return launch_quant(p, false, kScaleMx32, reinterpret_cast<cudaStream_t>(stream));
}

bfp8_status bfp8_mx_gemm(const uint8_t* A, const float* sa, const uint8_t* B, const float* sb, int64_t M, int64_t N,
                         int64_t K, void* C, bfp8_stream_t stream) {
  if (!A || !sa || !B || !sb || !C) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(sa) || !aligned16(sb) || !aligned16(C)) return BFP8_EALIGN;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  CUtensorMap ta, tb, tc;
  if ((s = make_kmajor_tmap(&ta, A, M, K, 128)) != BFP8_OK) return s;
  if ((s = make_kmajor_tmap(&tb, B, N, K, 128)) != BFP8_OK) return s;
  if ((s = make_bf16_store_tmap(&tc, C, M, N, true)) != BFP8_OK) return s;
  GemmParams p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>(M / 128);
  p.n_tiles = static_cast<int>(N / 128);
  p.tiles = p.m_tiles * p.n_tiles;
  p.splits = 1;
  p.kps = static_cast<int>(K / 128);
  p.units = p.tiles;
  p.group_m = 16;
  p.m_tile_rows = 128;
  p.sa = sa;
  p.sb = sb;
  p.C = static_cast<uint16_t*>(C);
  p.wait_ns = dev->wait_ns;
  p.stall = take_stall();
  const int grid = std::min(p.units, dev->sms);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  mx_gemm_kernel<<<grid, kGemmThreads, MxSmem::kAlloc, st>>>(ta, tb, tc, p);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cuda_status(cudaGetLastError());
}

size_t bfp8_gemm_workspace_bytes(bfp8_layout layout, int64_t M, int64_t N, int64_t K) {
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return 0;
  return plan_gemm(layout, M, N, K, current_state()).ws_bytes;
}

size_t bfp8_linear_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return 0;
  return fwd_ws(M, N, K, current_state(), nullptr, nullptr, nullptr, nullptr, nullptr);
}

size_t bfp8_linear_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return 0;
  return bwd_ws(M, N, K, current_state(), nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
}

bfp8_status bfp8_linear_fwd_ex(const void* X, const void* W, int64_t M, int64_t N, int64_t K, void* Y, uint8_t* WqT,
                               float* sW, uint8_t* XqT, float* sXT, void* ws, size_t ws_bytes,
                               bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  if (!X || !W || !Y || !WqT || !sW || !XqT || !sXT) return BFP8_EINVAL;
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  const size_t need = fwd_ws(M, N, K, *dev, nullptr, nullptr, nullptr, nullptr, nullptr);
  if (ws == nullptr || ws_bytes < need) return BFP8_EWORKSPACE;
  if (!aligned16(ws)) return BFP8_EALIGN;
  Carver cv(ws);
  uint8_t *Wq, *Xq;
  float* sX;
  void* gws;
  fwd_ws(M, N, K, *dev, &cv, &Wq, &Xq, &sX, &gws);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = quant_w_impl(W, N, K, Wq, WqT, sW, scale_mode, st)) != BFP8_OK) return s;
  if ((s = quant_act_impl(X, M, K, Xq, sX, XqT, sXT, scale_mode, st)) != BFP8_OK) return s;
  const size_t gws_bytes = ws_bytes - (static_cast<uint8_t*>(gws) - static_cast<uint8_t*>(ws));
  return gemm_impl(BFP8_FPROP, Xq, sX, Wq, sW, M, N, K, Y, nullptr, nullptr, gws, gws_bytes, st);
}

bfp8_status bfp8_linear_fwd_prequantised(const void* X, const uint8_t* Wq, const float* sW, int64_t M, int64_t N,
                                         int64_t K, void* Y, uint8_t* XqT, float* sXT, void* ws, size_t ws_bytes,
                                         bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  if (!X || !Wq || !sW || !Y || !XqT || !sXT) return BFP8_EINVAL;
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  const size_t need = fwd_ws(M, N, K, *dev, nullptr, nullptr, nullptr, nullptr, nullptr);
  if (ws == nullptr || ws_bytes < need) return BFP8_EWORKSPACE;
  if (!aligned16(ws)) return BFP8_EALIGN;
  Carver cv(ws);
  uint8_t* Xq;
  float* sX;
  void* gws;
  fwd_ws(M, N, K, *dev, &cv, nullptr, &Xq, &sX, &gws);  // the weight-code region stays unused
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = quant_act_impl(X, M, K, Xq, sX, XqT, sXT, scale_mode, st)) != BFP8_OK) return s;
  const size_t gws_bytes = ws_bytes - (static_cast<uint8_t*>(gws) - static_cast<uint8_t*>(ws));
  return gemm_impl(BFP8_FPROP, Xq, sX, Wq, sW, M, N, K, Y, nullptr, nullptr, gws, gws_bytes, st);
}

bfp8_status bfp8_linear_fwd(const void* X, const void* W, int64_t M, int64_t N, int64_t K, void* Y, uint8_t* WqT,
                            float* sW, uint8_t* XqT, float* sXT, void* ws, size_t ws_bytes, bfp8_stream_t stream) {
  return bfp8_linear_fwd_ex(X, W, M, N, K, Y, WqT, sW, XqT, sXT, ws, ws_bytes, BFP8_SCALE_AMAX448, stream);
}

// The backward pass; dW bf16 is written, or (dW null) the weight gradient
// is added into the fp32 dW_main.
static bfp8_status linear_bwd_impl(const void* dY, const uint8_t* WqT, const float* sW, const uint8_t* XqT, const float* sXT,
                            int64_t M, int64_t N, int64_t K, void* dX, void* dW, float* dW_main, void* ws,
                            size_t ws_bytes, int scale_mode, bfp8_stream_t stream) {
  if (!dY || !WqT || !sW || !XqT || !sXT || !dX || ((dW == nullptr) == (dW_main == nullptr))) return BFP8_EINVAL;
  if (!scale_mode_ok(scale_mode)) return BFP8_EINVAL;
  if (!dim_ok(M) || !dim_ok(N) || !dim_ok(K)) return BFP8_EINVAL;
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  const size_t need = bwd_ws(M, N, K, *dev, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  if (ws == nullptr || ws_bytes < need) return BFP8_EWORKSPACE;
  if (!aligned16(ws)) return BFP8_EALIGN;
  Carver cv(ws);
  uint8_t *dYq, *dYqT;
  float *sdY, *sdYT;
  void* gws;
  bwd_ws(M, N, K, *dev, &cv, &dYq, &sdY, &dYqT, &sdYT, &gws);
  const size_t gws_bytes = ws_bytes - (static_cast<uint8_t*>(gws) - static_cast<uint8_t*>(ws));
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((s = quant_act_impl(dY, M, N, dYq, sdY, dYqT, sdYT, scale_mode, st)) != BFP8_OK) return s;
  if ((s = gemm_impl(BFP8_DGRAD, dYq, sdY, WqT, sW, M, K, N, dX, nullptr, nullptr, gws, gws_bytes, st)) != BFP8_OK)
    return s;
  return gemm_impl(BFP8_WGRAD, dYqT, sdYT, XqT, sXT, N, K, M, dW, nullptr, nullptr, gws, gws_bytes, st, dW_main);
}

bfp8_status bfp8_linear_bwd_ex(const void* dY, const uint8_t* WqT, const float* sW, const uint8_t* XqT,
                               const float* sXT, int64_t M, int64_t N, int64_t K, void* dX, void* dW, void* ws,
                               size_t ws_bytes, bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  if (dW == nullptr) return BFP8_EINVAL;
  return linear_bwd_impl(dY, WqT, sW, XqT, sXT, M, N, K, dX, dW, nullptr, ws, ws_bytes, scale_mode, stream);
}

bfp8_status bfp8_linear_bwd_main_grad(const void* dY, const uint8_t* WqT, const float* sW, const uint8_t* XqT,
                                      const float* sXT, int64_t M, int64_t N, int64_t K, void* dX, float* dW_main,
                                      void* ws, size_t ws_bytes, bfp8_scale_mode scale_mode, bfp8_stream_t stream) {
  if (dW_main == nullptr) return BFP8_EINVAL;
  return linear_bwd_impl(dY, WqT, sW, XqT, sXT, M, N, K, dX, nullptr, dW_main, ws, ws_bytes, scale_mode, stream);
}

bfp8_status bfp8_linear_bwd(const void* dY, const uint8_t* WqT, const float* sW, const uint8_t* XqT, const float* sXT,
                            int64_t M, int64_t N, int64_t K, void* dX, void* dW, void* ws, size_t ws_bytes,
                            bfp8_stream_t stream) {
  return bfp8_linear_bwd_ex(dY, WqT, sW, XqT, sXT, M, N, K, dX, dW, ws, ws_bytes, BFP8_SCALE_AMAX448, stream);
}

bfp8_status bfp8_sync_status(bfp8_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return BFP8_ECUDA;
  unsigned int flags = 0;
  if (cudaMemcpyFromSymbol(&flags, bfp8::g_error_flags, sizeof(flags)) != cudaSuccess) return BFP8_ECUDA;
  if (flags != 0u) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(bfp8::g_error_flags, &zero, sizeof(zero)) != cudaSuccess) return BFP8_ECUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return BFP8_ECUDA;
  }
  return (flags & bfp8::kErrTimeout) ? BFP8_ETIMEOUT : BFP8_OK;
}

bfp8_status bfp8_set_wait_limit_ns(uint64_t ns) {
  DeviceState* dev = nullptr;
  bfp8_status s = device_state(&dev);
  if (s != BFP8_OK) return s;
  std::lock_guard<std::mutex> lk(g_mu);
  dev->wait_ns = ns == 0 ? kDefaultWaitNs : ns;
  return BFP8_OK;
}

bfp8_status bfp8_set_gemm_kernel(int kind) {
  if (kind < 0 || kind > 2) return BFP8_EINVAL;
  g_gemm_kind.store(kind, std::memory_order_relaxed);
  return BFP8_OK;
}

bfp8_status bfp8_set_gemm_splits(int splits) {
  if (splits < 0) return BFP8_EINVAL;
  g_forced_splits.store(splits, std::memory_order_relaxed);
  return BFP8_OK;
}

uint64_t bfp8_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

bfp8_status bfp8_test_stall_next_launch(void) {
  g_stall_next.store(1, std::memory_order_relaxed);
  return BFP8_OK;
}

const char* bfp8_status_string(bfp8_status status) {
  switch (status) {
    case BFP8_OK: return "ok";
    case BFP8_EINVAL: return "invalid argument (null pointer, bad enum, or a dimension not a positive multiple of 128)";
    case BFP8_EALIGN: return "pointer not 16-byte aligned";
    case BFP8_EUNSUPPORTED: return "unsupported device or size";
    case BFP8_ECUDA: return "CUDA runtime or driver error";
    case BFP8_ETIMEOUT: return "device-side bounded wait expired";
    case BFP8_EWORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

}  // extern "C"
