// Shared device helpers: inline PTX for mbarriers, bulk/tensor copies
// (TMA), tcgen05 (tensor memory and MMA), bounded waits and the device error
// word.  Everything here is sm_103a-only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace bfp8 {

constexpr int kGroup = 128;  // scale group length / block edge

// Device error word (one per device, in this translation unit).  Bits:
//   1 : a bounded wait expired.
// The first failing site is stored in g_error_site for debugging.
__device__ unsigned int g_error_flags;
__device__ unsigned int g_error_site;

constexpr unsigned int kErrTimeout = 1u;

// Limit of the waits a kernel makes, on its way out, for its own operations
// still in flight: TMA copies into its shared memory, and tensor-core MMAs
// into tensor memory it is about to free.  Hardware completes those whatever
// else has failed, so the limit is long and fixed: bfp8_set_wait_limit_ns,
// which bounds every other wait, does not shorten it.
constexpr uint64_t kDrainWaitNs = 5000000000ull;  // 5 s

__device__ __forceinline__ void raise_error(unsigned int flag, unsigned int site) {
  if (atomicOr(&g_error_flags, flag) == 0u) atomicExch(&g_error_site, site);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31u) == 0u; }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One potentially blocking test of the phase with the given parity: the
// thread may be suspended (up to kSuspendHintNs) until the phase completes,
// so a waiting warp does not spin on the issue slots.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns nanoseconds: raises kErrTimeout (with `site`) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, uint32_t site) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      raise_error(kErrTimeout, site);
      return false;
    }
  }
}

// ------------------------------------------------------------- bulk copies
// Non-tensor bulk copy global -> shared, completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor copy global -> shared (TMA).  c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t c0, int32_t c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor copy shared -> global (TMA store), tracked by bulk groups.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap),
               "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}

// 2-D tensor reduce-add shared -> global (TMA): each element of the box is
// added into the global tensor (type from the tensor map), tracked by bulk
// groups.
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, const void* src, int32_t c0, int32_t c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   tmap),
               "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------ non-bulk async copies
// cp.async of 16 (or 4) bytes global -> shared; both addresses aligned to
// the size.  Completion is reported to an mbarrier by cp_async_arrive.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has landed
// (.noinc: the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Makes generic-proxy writes to shared memory visible to the async proxy
// (needed before a TMA store reads what threads wrote).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Packed fp32 pair arithmetic (sm_100 family builtins, round to nearest).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// ------------------------------------------------------------ conversions
// Two fp32 -> two E4M3 codes (round to nearest even, saturate to +-448);
// lo lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scale of a group from its amax: fp32_rn(amax / 448), or 1 for amax 0.
// amax is the largest magnitude of bf16 values, so it has at most 8
// significant bits.  For such amax with a normal quotient the quotient is
// taken as q0 = rn(amax * c), c = rn(1/448), corrected once with the exact
// residual amax - 448 q0 (Markstein's FMA correction step); checking every
// positive finite bf16 value against the IEEE quotient shows the result is
// the correctly rounded one.  Any other input takes the IEEE division.
__device__ __forceinline__ float group_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  const bool bf16_valued = (__float_as_uint(amax) & 0xFFFFu) == 0u;
  if (bf16_valued && amax >= 448.0f * 0x1p-126f && amax <= 0x1.FEp+127f) {
    constexpr float c = 1.0f / 448.0f;
    const float q0 = __fmul_rn(amax, c);
    const float r = __fmaf_rn(-q0, 448.0f, amax);
    return __fmaf_rn(r, c, q0);
  }
  return __fdiv_rn(amax, 448.0f);
}

// Per-group quantisation state.  A code is E4M3_rn_satfinite(fp32_rn(x / s)).
// A division per element would dominate the quantisers' instruction count,
// so the correctly rounded quotient Q = fp32_rn(x / s) is formed from the
// group's reciprocal with one FMA correction (Markstein's step: P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev., 1990; as stated in Muller et al., Handbook of
// Floating-Point Arithmetic):
//   r  = RN(1/s)                     once per group (IEEE reciprocal);
//   y0 = RN(x r)                     within 1.5 ulp of x/s;
//   Q  = RN(y0 + r RN(x - s y0)).
// For arbitrary x and s the theorem needs a faithful y (one more refinement
// before the last step).  The inputs here are narrower: x is bf16, and s is
// RN(amax/448) for a bf16 amax >= |x|.  Scaling x and amax by one power of two
// leaves y0 and Q unchanged while s stays in [2^-80, 2^100] (r is then
// normal, and a remainder that rounds is a normal fp32: it has more than 24
// bits above its quantum ulp(s) ulp(y0) >= 2^-137), so one binade of amax
// with every bf16 x covers all cases; evaluated exactly there (all 128
// mantissas, every x in (0, amax]), Q equals fp32_rn(x / s) every time, and y0
// alone misses some codes.  Quotients below 2^-11 (codes +-0) stay below the
// smallest E4M3 rounding boundary (2^-10) whatever the remainder's rounding.
// The quantisers write the step on -x, which keeps the sign of a zero
// quotient (quotient_pair_neg); the GEMM's quantised epilogue restores it
// from x.  A group whose scale lies outside [2^-80, 2^100] (or is not
// finite) takes the power-of-two pre-scaling in the quantisers
// (scaled_group) and the IEEE division in the epilogue.
struct GroupScale {
  float s;     // dequantisation scale amax/448 (1 for an all-zero group)
  float r;     // RN(1/s)
  bool exact;  // s within [2^-80, 2^100]: the FMA path applies
};

__device__ __forceinline__ GroupScale make_group_scale(float amax) {
  GroupScale g;
  g.s = group_scale(amax);
  g.exact = g.s >= 0x1p-80f && g.s <= 0x1p+100f;
  g.r = g.exact ? __frcp_rn(g.s) : 0.0f;
  return g;
}

// Power-of-two scale mode: s = 2^k, the smallest power of two with
// s >= amax/448 (1 for an all-zero group), the reading taken for the paper's
// SM120 power-of-two scales ("Puro-2B ...", section 3.2).  With
// amax = (1 + m) 2^e (m the 23-bit fraction, fp32 subnormals normalised),
// 2^k >= amax/448 = (1 + m)/1.75 * 2^(e-8) holds from k = e - 8 when
// 1 + m <= 1.75 and from k = e - 7 otherwise.  Then x/s = x * 2^-k is an
// exact scaling: when 2^-k is a normal fp32 (k >= -127) the product is the
// IEEE quotient, sign of zero included; smaller scales (only for groups with
// amax below about 2^-118) take the IEEE division.
__device__ __forceinline__ GroupScale make_group_scale_pow2(float amax) {
  GroupScale g;
  if (!(amax > 0.0f)) {
    g.s = 1.0f;
    g.r = 1.0f;
    g.exact = true;
    return g;
  }
  const uint32_t b = __float_as_uint(amax);
  int e;
  uint32_t m;
  if (b >= 0x00800000u) {
    e = static_cast<int>(b >> 23) - 127;
    m = b & 0x007FFFFFu;
  } else {  // subnormal: amax = b 2^-149
    const int p = 31 - __clz(static_cast<int>(b));
    e = p - 149;
    m = (b << (23 - p)) & 0x007FFFFFu;
  }
  const int k = e - 8 + (m > 0x00600000u ? 1 : 0);  // in [-141, 120]
  g.s = k >= -126 ? __uint_as_float(static_cast<uint32_t>(k + 127) << 23)
                  : __uint_as_float(1u << (k + 149));
  g.exact = k >= -127;
  g.r = g.exact ? __uint_as_float(static_cast<uint32_t>(127 - k) << 23) : 0.0f;
  return g;
}

// Reciprocal-multiply mode: the stored scale is amax/448 as above, and the
// codes are E4M3(fp32_rn(x * m)) with one multiplier per group,
// m = fp32_rn(448 / amax) (one IEEE division per group), saturated at the
// largest finite fp32 (reached only for amax below about 2^-119); 1 for an
// all-zero group.  GroupScale::r carries m; every group is on the multiply
// path.
__device__ __forceinline__ GroupScale make_group_scale_recip(float amax) {
  GroupScale g;
  g.s = group_scale(amax);
  g.r = amax == 0.0f ? 1.0f : fminf(__fdiv_rn(448.0f, amax), 0x1.FFFFFEp+127f);
  g.exact = true;
  return g;
}

// Scale modes, numbered as the C ABI's bfp8_scale_mode.
constexpr int kScaleAmax448 = 0;
constexpr int kScalePow2 = 1;
constexpr int kScaleMulRecip = 2;
// MXFP8 1x32 recipe (bloombook.cn tutorial, FP8 paragraph and MXFP concept
// figure: one shared scale per 32 consecutive values): groups of 32 instead
// of 128, each with the power-of-two scale above clamped to the E8M0 range
// [2^-127, 2^127].  Not a mode of the C ABI's bfp8_scale_mode: its scales
// have their own layout ([C/32, R]), so it has its own entry point.
constexpr int kScaleMx32 = 3;

// The power-of-two scale clamped to 2^-127 from below (the upper end, 2^127,
// lies beyond any bf16 amax / 448).  2^-127 is an fp32 subnormal whose
// reciprocal 2^127 is normal, so every group is on the multiply path.
__device__ __forceinline__ GroupScale make_group_scale_mx(float amax) {
  GroupScale g = make_group_scale_pow2(amax);
  if (g.s < 0x1p-127f) {
    g.s = 0x1p-127f;
    g.r = 0x1p+127f;
    g.exact = true;
  }
  return g;
}

// Whether a group scale of the given mode is on the fast (multiply or FMA)
// path; restates GroupScale::exact from s alone.
template <int kScale>
__device__ __forceinline__ bool scale_fast(float s) {
  if constexpr (kScale == kScalePow2) return s >= 0x1p-127f;
  if constexpr (kScale == kScaleMulRecip || kScale == kScaleMx32) return true;
  return s >= 0x1p-80f && s <= 0x1p+100f;
}

template <int kScale>
__device__ __forceinline__ GroupScale make_scale(float amax) {
  if constexpr (kScale == kScalePow2) return make_group_scale_pow2(amax);
  if constexpr (kScale == kScaleMx32) return make_group_scale_mx(amax);
  if constexpr (kScale == kScaleMulRecip) return make_group_scale_recip(amax);
  return make_group_scale(amax);
}

// |v| with the sign of x.
__device__ __forceinline__ float with_sign_of(float v, float x) {
  return __uint_as_float((__float_as_uint(v) & 0x7FFFFFFFu) | (__float_as_uint(x) & 0x80000000u));
}

// RN(x / s) for a pair of bf16 values x of a group with s = RN(amax/448), by
// the correction step above (r2 = RN(1/s), ns2 = -s, for each component),
// except that the sign of a zero result may be lost (the correction's sum
// turns -0 into +0).
__device__ __forceinline__ float2 quotient_pair_unsigned_zero(float2 x, float2 r2, float2 ns2) {
  const float2 y0 = fmul2(x, r2);
  return ffma2(ffma2(y0, ns2, x), r2, y0);
}

// -x, widened to fp32, for the bf16 value in the low / high half of w: the
// sign bit is flipped by the same integer operation that places the value.
__device__ __forceinline__ float neg_bf16lo(uint32_t w) { return __uint_as_float((w << 16) + 0x80000000u); }
__device__ __forceinline__ float neg_bf16hi(uint32_t w) { return __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u); }

// The correction step written on nx = -x, with nr2 = -RN(1/s) and s2 = s in
// both components:
//   y0 = RN(nx nr)        = RN(x r), the same product;
//   e  = RN(s y0 + nx)    = -(x - s y0), exact as before;
//   Q  = RN(e nr + y0)    = RN(y0 + r (x - s y0)), the same sum.
// So Q is RN(x / s) wherever the step on x gives it, and for x = -0 the last
// sum adds two zeros of x's sign (-0 + -0), so Q keeps the sign of every
// zero without a separate restore.
__device__ __forceinline__ float2 quotient_pair_neg(float2 nx, float2 nr2, float2 s2) {
  const float2 y0 = fmul2(nx, nr2);
  return ffma2(ffma2(y0, s2, nx), nr2, y0);
}

// Four E4M3 codes (byte i from q_i) in one register: two paired casts and
// one pack.
__device__ __forceinline__ uint32_t e4m3x4(float q0, float q1, float q2, float q3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(q0), "f"(q1), "f"(q2), "f"(q3));
  return r;
}

// State of a group whose scale is off the FMA path (s outside [2^-80, 2^100]
// or not finite).  x / s = (x p) / (s p) for a power of two p, and s p lies
// well inside that range: p = 2^100 for small s, 2^-64 for large.  x p is
// exact unless it underflows, which happens only for s > 2^100 and
// |x| < 2^-62, where |x / s| < 2^-162 and the code is a signed zero either
// way.  The scaled pair takes two correction steps (a faithful quotient,
// then Markstein's step), which give RN(x p / (s p)) for any normal s p.  An
// infinite s (an infinite amax) takes p = 0: x p is then a signed zero for
// finite x (code +-0, as x / inf) and NaN for infinite or NaN x (code NaN,
// as inf / inf), and s p = 1 leaves it as it is.
struct ScaledGroup {
  float p;   // the power of two (0 for an infinite s)
  float s;   // s p (1 for an infinite s)
  float nr;  // -RN(1 / (s p))
};

__device__ __forceinline__ ScaledGroup scaled_group(float s) {
  ScaledGroup g;
  if (!(s <= 0x1.FFFFFEp+127f)) {
    g.p = 0.0f;
    g.s = 1.0f;
    g.nr = -1.0f;
    return g;
  }
  g.p = s < 1.0f ? 0x1p+100f : 0x1p-64f;
  g.s = s * g.p;
  g.nr = -__frcp_rn(g.s);
  return g;
}

// RN(x / s) for the pair nx = -x of a group off the FMA path (see above).
__device__ __forceinline__ float2 quotient_pair_scaled(float2 nx, const ScaledGroup& g) {
  const float2 p2 = make_float2(g.p, g.p), s2 = make_float2(g.s, g.s), nr2 = make_float2(g.nr, g.nr);
  const float2 nxp = fmul2(nx, p2);
  const float2 y0 = fmul2(nxp, nr2);
  const float2 y1 = ffma2(ffma2(y0, s2, nxp), nr2, y0);
  return ffma2(ffma2(y1, s2, nxp), nr2, y1);
}

// Codes of the pair (x0, x1) (x0 in the low byte), one group on the FMA path.
__device__ __forceinline__ uint32_t quant_pair_exact(float x0, float x1, float2 r2, float2 ns2) {
  const float2 q = quotient_pair_unsigned_zero(make_float2(x0, x1), r2, ns2);
  return e4m3x2(with_sign_of(q.x, x0), with_sign_of(q.y, x1));
}

// Reference path: the IEEE quotient, then the cast.
__device__ __forceinline__ uint32_t quant_pair_div(float x0, float x1, float s0, float s1) {
  return e4m3x2(__fdiv_rn(x0, s0), __fdiv_rn(x1, s1));
}

// Two codes (lo byte = a) of the values a, b under one group scale g.
__device__ __forceinline__ uint32_t quant_pair(float a, float b, const GroupScale& g) {
  if (g.exact) return quant_pair_exact(a, b, make_float2(g.r, g.r), make_float2(-g.s, -g.s));
  return quant_pair_div(a, b, g.s, g.s);
}

// ---- SiLU-gated FFN activation, h = SiLU(g) u = g u / (1 + e^-g) ----------
// The down projection of the FFN takes h, a bf16 tensor; its quantiser can
// form h itself from the gate+up output.  e^-|g| = 2^(-|g| log2 e) comes from
// the PTX instruction ex2.approx.f32 (relative error about 2^-22, subnormal
// results kept) and 1 / (1 + e^-|g|) from rcp.approx.ftz.f32 on [1, 2], so h
// is within a few fp32 ulp of the exact value before its bf16 rounding.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// SiLU(g) u for |g| <= 64, where p = e^-|g| >= 2^-93 is a normal fp32:
// sigma(g) = 1 / (1 + p) for g >= 0 and p / (1 + p) for g < 0.
__device__ __forceinline__ float silu_mul(float g, float u) {
  const float p = ex2_approx(fabsf(g) * -kLog2e);
  const float r = rcp_approx(1.0f + p);
  return (g * u) * (g < 0.0f ? p * r : r);
}

// The same for any finite g.  Beyond |g| = 64, 1 + e^-|g| rounds to 1, and
// for g < 0 the factor e^-|g| is formed as 2^64 e^-|g| (a normal fp32 down to
// |g| of about 131) and the 2^-64 is applied last, so h keeps its precision
// until it is itself below the fp32 normal range.
__device__ __forceinline__ float silu_mul_wide(float g, float u) {
  const float a = fabsf(g);
  const bool big = a > 64.0f;
  const float p = ex2_approx(fmaf(a, -kLog2e, big ? 64.0f : 0.0f));
  const float r = rcp_approx(1.0f + (big ? 0.0f : p));
  const float h = (g * u) * (g < 0.0f ? p * r : r);
  return (big && g < 0.0f) ? h * 0x1p-64f : h;
}

// bf16_rn(SiLU(g) u) for the two bf16 values of each word (low half first).
template <bool kWide>
__device__ __forceinline__ uint32_t swiglu_bf16x2(uint32_t g, uint32_t u) {
  const float lo = kWide ? silu_mul_wide(bf16lo(g), bf16lo(u)) : silu_mul(bf16lo(g), bf16lo(u));
  const float hi = kWide ? silu_mul_wide(bf16hi(g), bf16hi(u)) : silu_mul(bf16hi(g), bf16hi(u));
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h2);
}

template <bool kWide>
__device__ __forceinline__ uint4 swiglu_bf16x8(const uint4& g, const uint4& u) {
  return make_uint4(swiglu_bf16x2<kWide>(g.x, u.x), swiglu_bf16x2<kWide>(g.y, u.y), swiglu_bf16x2<kWide>(g.z, u.z),
                    swiglu_bf16x2<kWide>(g.w, u.w));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace bfp8

namespace bfp8 {

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] . B[smem]^T, E4M3 x E4M3 -> fp32, one instruction
// covers M=128, N from the instruction descriptor, K=32.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address / 16
  d |= static_cast<uint64_t>(1) << 16;                   // leading offset (unused for this layout)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride offset: next 8-row atom
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128 B
  return d;
}

// Instruction descriptor: E4M3 x E4M3 -> F32, both operands K-major, no
// negation, dense, shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                  // D format F32
         | (0u << 7) | (0u << 10)                   // A, B: E4M3
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

#define BFP8_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define BFP8_W8(i) "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]), "+r"(v[i + 4]), "+r"(v[i + 5]), "+r"(v[i + 6]), "+r"(v[i + 7])

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : BFP8_R8(0), BFP8_R8(8), BFP8_R8(16), BFP8_R8(24)
      : "r"(taddr));
}

#define BFP8_R8X(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])

// 64 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : BFP8_R8X(0), BFP8_R8X(8), BFP8_R8X(16), BFP8_R8X(24), BFP8_R8X(32), BFP8_R8X(40), BFP8_R8X(48), BFP8_R8X(56)
      : "r"(taddr));
}

// 16 TMEM lanes x 64 consecutive fp32 columns (16x256b shape, 8 repeats
// along the columns): thread t receives, for repeat i, v[4i + 0..1] = lane
// L + t/4, columns 8i + 2 (t%4) + 0..1, and v[4i + 2..3] = lane L + t/4 + 8,
// the same columns (L = the lane field of taddr).
__device__ __forceinline__ void tmem_ld16x256b_x8(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : BFP8_R8(0), BFP8_R8(8), BFP8_R8(16), BFP8_R8(24)
      : "r"(taddr));
}

// The same shape over 128 consecutive columns (16 repeats, 64 registers).
__device__ __forceinline__ void tmem_ld16x256b_x16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : BFP8_R8X(0), BFP8_R8X(8), BFP8_R8X(16), BFP8_R8X(24), BFP8_R8X(32), BFP8_R8X(40), BFP8_R8X(48), BFP8_R8X(56)
      : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld; the registers are tied to
// the wait so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld64(uint32_t* v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : BFP8_W8(0), BFP8_W8(8), BFP8_W8(16), BFP8_W8(24), BFP8_W8(32), BFP8_W8(40), BFP8_W8(48),
                 BFP8_W8(56)::"memory");
}

// Waits for this thread's outstanding tcgen05.ld; ties the 32 registers of
// the last load to the wait.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t* v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : BFP8_W8(0), BFP8_W8(8), BFP8_W8(16), BFP8_W8(24)::"memory");
}

#define BFP8_F8(i) "+f"(a[i]), "+f"(a[i + 1]), "+f"(a[i + 2]), "+f"(a[i + 3]), "+f"(a[i + 4]), "+f"(a[i + 5]), "+f"(a[i + 6]), "+f"(a[i + 7])

// Emits nothing; makes the 64 values a[0..63] final at this point in program
// order, so the arithmetic producing them cannot be moved below a later
// tcgen05.ld (which would keep two staging buffers live at once).
__device__ __forceinline__ void reg_fence64(float* a) {
  asm volatile("" : BFP8_F8(0), BFP8_F8(8), BFP8_F8(16), BFP8_F8(24), BFP8_F8(32), BFP8_F8(40), BFP8_F8(48), BFP8_F8(56));
}
__device__ __forceinline__ void reg_fence32(float* a) {
  asm volatile("" : BFP8_F8(0), BFP8_F8(8), BFP8_F8(16), BFP8_F8(24));
}

// ------------------------------------------------ CTA pairs (cluster of 2)
// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address, in the cluster's shared window, of the shared variable at the
// same offset as `p` in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Arrive on an mbarrier of another CTA of the cluster (default semantics:
// release at CTA scope).  Used to hand a tensor-memory buffer back, whose
// ordering comes from tcgen05.fence::before_thread_sync; a cluster-scope
// release here would add a full memory fence to every slice.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of both CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// 2-D tensor copy into this CTA's shared memory whose completion is counted
// on an mbarrier that may belong to either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar_cluster_addr)
      : "memory");
}

// Tensor memory of a CTA pair: allocated, relinquished and freed by one warp
// in each of the two CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (both CTAs' TMEM) (+)= A . B^T over the pair: A and B come from the same
// shared-memory offsets in both CTAs (each CTA holds half of the M rows of A
// and half of the N rows of B).  Issued by the first CTA of the pair only.
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at `bar`'s offset in every CTA of `cta_mask`
// when all pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Register reallocation between warpgroups (all 4 warps of a warpgroup
// execute the same one).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace bfp8
