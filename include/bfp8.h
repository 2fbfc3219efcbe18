/*
 * bfp8.h -- C ABI of the blockwise-FP8 Transformer linear layer for B300 (sm_103a).
 *
 * What the library computes is the linear-layer numerics of "Puro-2B: Poor
 * Lab's Qwen2-1.5B Trained on RTX 5090 within $5090" (papers.lianghsun.dev
 * translation), section 3.2 "FP8 mixed-precision training":
 *   - linear-layer GEMM operands are E4M3 (Micikevicius et al. 2022 format);
 *   - activations and activation gradients are quantised in 1-D groups of 128
 *     consecutive values along the GEMM reduction dimension;
 *   - weights are quantised in 2-D 128x128 blocks;
 *   - every group/block scale is computed online from that group's values.
 * The decoded value of a code is code * scale (bloombook.cn tutorial, MXFP
 * figure, "V_i = Q_i x X"), so every scale below is a dequantisation
 * multiplier.  The scale value is amax/448 in fp32 (1.0 for an all-zero
 * group) and codes are E4M3(x / scale) rounded to nearest-even with
 * saturation to +-448.
 *
 * Conventions for every entry point
 *   - All matrices are row-major and contiguous.  "bf16" is IEEE bfloat16.
 *   - Every dimension must be a positive multiple of 128 (BFP8_EINVAL).
 *   - Every device pointer must be 16-byte aligned (BFP8_EALIGN).
 *   - The caller owns all memory.  The library allocates no device memory.
 *     What it keeps between calls is a per-device error word, per-device
 *     set-up done on first use (kernel attributes, device queries, the
 *     device address of the static scratch array below) and that array:
 *     BFP8_NOALLOC_SCRATCH_BYTES of device memory in the loaded module,
 *     used only by bfp8_fp8_block_gemm_noalloc, whose contents persist
 *     between its calls.  The set-up does not survive cudaDeviceReset():
 *     do not call the library on a device after resetting it.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  The return value reports argument and
 *     launch errors only; bfp8_sync_status() reports errors raised on the
 *     device (an expired bounded wait).
 *   - Input and output buffers must not overlap.
 *
 * Scale layouts ("group-major": the scales of one group index are contiguous)
 *   - 1x128 groups along the columns of an [R, C] tensor: s is [C/128, R],
 *     s[g*R + r] scales elements (r, 128g .. 128g+127).
 *   - 128x128 weight blocks of W [N, K]: s is [N/128, K/128].
 */
#ifndef BFP8_H
#define BFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* bfp8_stream_t;

typedef enum {
  BFP8_OK = 0,
  BFP8_EINVAL = 1,       /* null pointer, bad enum, or a dimension that is not a positive multiple of 128 */
  BFP8_EALIGN = 2,       /* a pointer is not 16-byte aligned */
  BFP8_EUNSUPPORTED = 3, /* no usable sm_103a device, or a size beyond what a kernel indexes */
  BFP8_ECUDA = 4,        /* a CUDA runtime or driver call failed (launch, tensor-map encode, sync) */
  BFP8_ETIMEOUT = 5,     /* a device-side bounded wait expired; reported by bfp8_sync_status */
  BFP8_EWORKSPACE = 6    /* workspace pointer null or smaller than the matching *_workspace_bytes() */
} bfp8_status;

/* The three GEMMs of a linear layer Y = X . W^T with X [tokens, in], W [out, in]. */
typedef enum {
  BFP8_FPROP = 0, /* Y  = X  . W^T : reduction over in-features  */
  BFP8_DGRAD = 1, /* dX = dY . W   : reduction over out-features */
  BFP8_WGRAD = 2  /* dW = dY^T . X : reduction over tokens       */
} bfp8_layout;

/* How a group's scale s is chosen from its amax (the largest |x|). */
typedef enum {
  BFP8_SCALE_AMAX448 = 0,   /* s = fp32(amax / 448): the default, used by every entry point without _ex */
  BFP8_SCALE_POW2 = 1,      /* s = smallest power of two >= amax / 448 (the paper's SM120 power-of-two scales) */
  BFP8_SCALE_MUL_RECIP = 2  /* s = fp32(amax / 448); codes from x * fp32(448 / amax) instead of x / s */
} bfp8_scale_mode;

/*
 * Activation / activation-gradient quantiser, 1x128 groups (section 3.2:
 * groups of 128 consecutive values along the GEMM reduction dimension).
 *
 *   x   bf16 [M, K], read only.
 *   q   E4M3 [M, K] or NULL: groups of 128 along K (the fprop operand for an
 *       activation, the dgrad operand for an output gradient).
 *   s   fp32 [K/128, M]: scales of q; required when q is given, else ignored.
 *   qT  E4M3 [K, M] or NULL: groups of 128 consecutive rows (tokens) of x per
 *       column, stored transposed so each group is contiguous (the wgrad
 *       operand, where the reduction runs over tokens).
 *   sT  fp32 [M/128, K]: scales of qT; required when qT is given.
 * At least one of q / qT must be given.  Both outputs come from a single
 * read of x.  Errors: EINVAL, EALIGN, ECUDA.
 */
bfp8_status bfp8_quantize_act_1x128(const void* x, int64_t M, int64_t K,
                                    uint8_t* q, float* s,
                                    uint8_t* qT, float* sT,
                                    bfp8_stream_t stream);

/*
 * Weight quantiser, 128x128 blocks (section 3.2: weights use 2-D 128x128
 * blocks).  A block is the same set of values in W and W^T, so one scale
 * array serves fprop (W) and dgrad (W^T).
 *
 *   w   bf16 [N, K], read only.
 *   q   E4M3 [N, K] or NULL (fprop operand).
 *   qT  E4M3 [K, N] or NULL (dgrad operand, = q transposed).
 *   s   fp32 [N/128, K/128], required.
 * At least one of q / qT must be given.  Errors: EINVAL, EALIGN, ECUDA.
 */
bfp8_status bfp8_quantize_w_128x128(const void* w, int64_t N, int64_t K,
                                    uint8_t* q, uint8_t* qT, float* s,
                                    bfp8_stream_t stream);

/*
 * The two quantisers above with an explicit scale rule ("Puro-2B ...",
 * section 3.2: the same 1x128 / 128x128 grouping runs on SM120 with
 * power-of-two scales).  Arguments, layouts, ownership and errors are those of
 * bfp8_quantize_act_1x128 and bfp8_quantize_w_128x128; scale_mode selects s:
 *   BFP8_SCALE_AMAX448  s = fp32(amax / 448) (identical to the calls above);
 *   BFP8_SCALE_POW2     s = 2^k, the smallest power of two with s >= amax/448
 *                       (so nothing saturates and the group's largest |x|/s
 *                       lies in (224, 448]); 1 for an all-zero group.
 *   BFP8_SCALE_MUL_RECIP  s = fp32(amax / 448) as in the default mode, but the
 *                       codes multiply by the group's reciprocal instead of
 *                       dividing by s (the pages do not fix which; this is the
 *                       other reading): q = E4M3_rn_satfinite(fp32(x * m)),
 *                       m = fp32(448 / amax), saturated at the largest finite
 *                       fp32 (amax below about 2^-119); m = 1 for an all-zero
 *                       group.  One division per group instead of per value;
 *                       a few codes near E4M3 rounding midpoints differ from
 *                       the default mode's by one step.
 * In the first two modes q = E4M3_rn_satfinite(fp32(x / s)); with a
 * power-of-two s the division is an exact scaling.  The scales are fp32 in
 * every mode, so the GEMM and linear entry points consume any of them.  An
 * unknown scale_mode returns BFP8_EINVAL.
 */
bfp8_status bfp8_quantize_act_1x128_ex(const void* x, int64_t M, int64_t K,
                                       uint8_t* q, float* s, uint8_t* qT, float* sT,
                                       bfp8_scale_mode scale_mode, bfp8_stream_t stream);
bfp8_status bfp8_quantize_w_128x128_ex(const void* w, int64_t N, int64_t K,
                                       uint8_t* q, uint8_t* qT, float* s,
                                       bfp8_scale_mode scale_mode, bfp8_stream_t stream);

/*
 * Several weights quantised by one launch (the rule of
 * bfp8_quantize_w_128x128_ex applied to each; "Puro-2B ...", section 3.2:
 * 128x128 weight blocks).  A Transformer layer quantises four weights of
 * 8-50 MB each, and one launch per weight spends much of its time filling and
 * draining the GPU; this call walks the blocks of all of them in one launch
 * (up to four weights per launch, several launches for more) and writes
 * exactly what count calls of bfp8_quantize_w_128x128_ex would write.
 *
 *   jobs   host array of count descriptors, read during the call only; each
 *          names a weight w bf16 [n, k] and its outputs q [n, k], qT [k, n],
 *          s [n/128, k/128] (device pointers, 16-byte aligned), with the same
 *          meaning and the same rules as bfp8_quantize_w_128x128.
 *   count  number of jobs, >= 1.
 * Every job must ask for the same outputs: all give q or all leave it NULL,
 * and the same for qT.  Errors: EINVAL (a bad job, count < 1, mixed
 * outputs, unknown scale_mode) and EALIGN are found before anything is
 * launched; ECUDA (a tensor-map encode or launch failure) can come after the
 * launches of earlier groups of four jobs, whose outputs are then written.
 */
typedef struct {
  const void* w;
  int64_t n, k;
  uint8_t* q;
  uint8_t* qT;
  float* s;
} bfp8_w_job;
bfp8_status bfp8_quantize_w_128x128_batch(const bfp8_w_job* jobs, int count, bfp8_scale_mode scale_mode,
                                          bfp8_stream_t stream);

/*
 * SiLU-gated FFN activation fused into the activation quantiser: the input of
 * the FFN's down projection, h = bf16_rn(SiLU(g) * u) with
 * SiLU(g) = g / (1 + e^-g), is formed from the fused gate+up output and
 * quantised in 1x128 groups without a round trip through HBM ("Puro-2B ...",
 * section 3.2: the activation stays BF16 and FP8 is the linear layers' operand
 * format; the tutorial's model-architecture paragraph: FFN width 6144).
 *
 *   gu  bf16 [M, 2F], read only: gate g in columns 0..F-1, up u in F..2F-1.
 *   h   bf16 [M, F] or NULL: a copy of h (not needed by the down projection).
 *   q, s, qT, sT  as bfp8_quantize_act_1x128 for x = h [M, F] (K = F).
 * M and F positive multiples of 128, F at most 2^26.  h is computed in fp32
 * with the hardware 2^x and 1/x approximations (relative error about 2^-22)
 * and rounded to bf16 once, so it can differ from the exactly rounded value by
 * one bf16 unit where the product lies that close to a rounding midpoint;
 * the codes are the scale_mode quantisation of this h, bit for bit.  At least
 * one of q / qT must be given.  Errors: EINVAL, EALIGN, ECUDA.
 */
bfp8_status bfp8_swiglu_quantize_1x128(const void* gu, int64_t M, int64_t F, void* h,
                                       uint8_t* q, float* s, uint8_t* qT, float* sT,
                                       bfp8_scale_mode scale_mode, bfp8_stream_t stream);

/*
 * MXFP8 1x32 recipe, the finer-grained scaling that the blockwise recipe is
 * compared with (bloombook.cn tutorial, FP8 paragraph and MXFP concept figure:
 * every 32 consecutive values share one scale X, and a code decodes as
 * V_i = Q_i * X; section 3.2 of the paper runs its own recipe through that
 * hardware path on SM120 with power-of-two scales).
 *
 * bfp8_quantize_mx_1x32: groups of 32 instead of 128, for activations,
 * gradients and weights alike (the recipe has no 2-D blocks).
 *   x   bf16 [M, K], read only.
 *   q   E4M3 [M, K] or NULL: groups of 32 along K;  s fp32 [K/32, M].
 *   qT  E4M3 [K, M] or NULL: groups of 32 consecutive rows per column,
 *       stored transposed;  sT fp32 [M/32, K].
 * Scale of a group: s = 2^k, the smallest power of two >= amax/448, with k
 * clamped to the E8M0 range [-127, 127] (only the lower end is ever reached);
 * 1 for an all-zero group.  Codes: q = E4M3_rn_satfinite(x / s), an exact
 * scaling.  At least one of q / qT.  Errors: EINVAL, EALIGN, ECUDA.
 *
 * bfp8_mx_gemm: C bf16 [M, N] = bf16( sum over 32-deep slices t of
 *   P_t[i, j] * sa(i, t) * sb(j, t) ), P_t the tensor-core fp32 sum of the
 *   slice's products, promoted in fp32 slice by slice.
 *   A E4M3 [M, K], sa fp32 [K/32, M];  B E4M3 [N, K], sb fp32 [K/32, N]:
 *   both as bfp8_quantize_mx_1x32 returns them in either direction.  For a
 *   linear layer Y = X . W^T: FPROP A = q(X), B = q(W); DGRAD A = q(dY),
 *   B = qT(W) (W^T quantised along the output features); WGRAD A = qT(dY),
 *   B = qT(X).  M, N, K positive multiples of 128.  Errors: EINVAL, EALIGN,
 *   EUNSUPPORTED, ECUDA.
 */
bfp8_status bfp8_quantize_mx_1x32(const void* x, int64_t M, int64_t K,
                                  uint8_t* q, float* s, uint8_t* qT, float* sT,
                                  bfp8_stream_t stream);
bfp8_status bfp8_mx_gemm(const uint8_t* A, const float* sa,
                         const uint8_t* B, const float* sb,
                         int64_t M, int64_t N, int64_t K,
                         void* C, bfp8_stream_t stream);

/*
 * Block-scaled FP8 GEMM with fp32 promotion per 128-deep slice (section 3.2:
 * E4M3 operands, fp32 training state; scales per 1x128 group / 128x128 block).
 *
 *   C[i, j] = bf16( sum over slices kb of  P_kb[i, j] * sa(i, kb) * sb(j, kb) )
 *   P_kb[i, j] = sum_{k in slice kb} A[i, k] * B[j, k]   (tensor-core fp32 accumulation)
 *
 * M, N: output rows and columns; K: reduction length.  A E4M3 [M, K] and
 * B E4M3 [N, K] are both K-contiguous.  sa is fp32 [K/128, M] for every
 * layout.  sb depends on the layout:
 *   FPROP: A = Xq,   B = Wq  [N, K]: sb = sW  [N/128, K/128] (weight blocks)
 *   DGRAD: A = dYq,  B = WqT [N, K]: sb = sW  [K/128, N/128] (the same weight
 *          scales, whose block rows now run along the reduction)
 *   WGRAD: A = dYqT, B = XqT [N, K]: sb = sXT [K/128, N]     (token groups)
 *   C    bf16 [M, N], written.
 *   Cq / sCq  optional fused quantised epilogue: E4M3 [M, N] codes of the
 *        bf16 C in 1x128 groups along N, with fp32 scales [N/128, M], exactly
 *        as bfp8_quantize_act_1x128 (the default amax/448 rule; there is no
 *        scale-mode variant) would produce from C.  Both or neither.
 *   workspace / ws_bytes  scratch of at least bfp8_gemm_workspace_bytes()
 *        bytes (may be 0 bytes, then workspace may be NULL).
 * Errors: EINVAL, EALIGN, EWORKSPACE, EUNSUPPORTED, ECUDA.
 */
bfp8_status bfp8_fp8_block_gemm(bfp8_layout layout,
                                const uint8_t* A, const float* sa,
                                const uint8_t* B, const float* sb,
                                int64_t M, int64_t N, int64_t K,
                                void* C, uint8_t* Cq, float* sCq,
                                void* workspace, size_t ws_bytes,
                                bfp8_stream_t stream);

/* Scratch bytes bfp8_fp8_block_gemm needs for these arguments (0 when none). */
size_t bfp8_gemm_workspace_bytes(bfp8_layout layout, int64_t M, int64_t N, int64_t K);

/*
 * fp32 accumulate-into GEMM: C_f32 [M, N] += the block-scaled product, with
 * the operands, scales and layouts of bfp8_fp8_block_gemm.  Each element
 * receives one fp32 addition of the fp32 promotion accumulator (no bf16
 * rounding), as an fp32 main gradient needs: section 3.2 keeps the training
 * state on the BF16/FP32 path.  C_f32 is caller-owned, read and written;
 * calls on the same C_f32 must not overlap.  The workspace is the one
 * bfp8_gemm_workspace_bytes() reports for the same layout and sizes.
 * Errors: as bfp8_fp8_block_gemm; C_f32 null returns BFP8_EINVAL.
 */
bfp8_status bfp8_fp8_block_gemm_accumulate(bfp8_layout layout,
                                           const uint8_t* A, const float* sa,
                                           const uint8_t* B, const float* sb,
                                           int64_t M, int64_t N, int64_t K,
                                           float* C_f32,
                                           void* workspace, size_t ws_bytes,
                                           bfp8_stream_t stream);

/*
 * The same GEMM as bfp8_fp8_block_gemm, for callers that cannot allocate
 * device memory for its split-K workspace and have none to hand over: a
 * process whose device memory is all reserved by another framework's memory
 * pool, where a cudaMalloc would fail; a latency-bound loop where cudaMalloc
 * and cudaFree, which may synchronise the device, must not run; code bound to
 * an interface that has no workspace argument.  The paper has no counterpart;
 * this is a convenience of the library.  Call it from ordinary host code, as
 * every other entry point: it makes CUDA runtime calls (device queries,
 * kernel launches).
 *
 * Arguments, layouts and results are those of bfp8_fp8_block_gemm without
 * the workspace: the caller still passes every input and output.  The
 * split-K partial sums go to one static device array of
 * BFP8_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  This entry point calls
 * no cudaMalloc, cudaFree or other allocating routine.  Its results equal
 * bfp8_fp8_block_gemm's bit for bit (the same plan runs the same kernels).
 *
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it; make that
 *     first call before any stream capture on the device.  The kept address
 *     does not survive cudaDeviceReset() (see the conventions above).
 *   - Every call shares the one array.  Calls that run at the same time on
 *     the GPU (different streams or threads) race on it and corrupt each
 *     other's results: serialise them.  Each call overwrites every partial
 *     it reads, so nothing has to be cleared between calls.
 *   - Sizes whose split-K partials (splits x M x N x 4 bytes, with the split
 *     count bfp8_fp8_block_gemm would use) exceed the array are rejected
 *     with BFP8_EWORKSPACE before anything is launched.
 * Errors: EINVAL, EALIGN, EWORKSPACE, EUNSUPPORTED, ECUDA.
 */
#define BFP8_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
bfp8_status bfp8_fp8_block_gemm_noalloc(bfp8_layout layout,
                                        const uint8_t* A, const float* sa,
                                        const uint8_t* B, const float* sb,
                                        int64_t M, int64_t N, int64_t K,
                                        void* C, uint8_t* Cq, float* sCq,
                                        bfp8_stream_t stream);

/*
 * Fused forward of one linear layer, Y [M, N] = X [M, K] . W [N, K]^T
 * (section 3.2: W stays bf16/fp32 and is re-quantised on every use; FP8 is
 * the online compute and activation-storage format).  Runs the weight
 * quantiser, the dual activation quantiser and the FPROP GEMM.
 *
 *   X bf16 [M, K], W bf16 [N, K]: inputs.   Y bf16 [M, N]: output.
 *   Saved for the backward pass, caller-owned outputs:
 *     WqT E4M3 [K, N], sW fp32 [N/128, K/128], XqT E4M3 [K, M], sXT fp32 [M/128, K].
 *   ws / ws_bytes: scratch of at least bfp8_linear_fwd_workspace_bytes().
 * Errors: as the calls it makes.
 */
bfp8_status bfp8_linear_fwd(const void* X, const void* W,
                            int64_t M, int64_t N, int64_t K,
                            void* Y,
                            uint8_t* WqT, float* sW, uint8_t* XqT, float* sXT,
                            void* ws, size_t ws_bytes,
                            bfp8_stream_t stream);
size_t bfp8_linear_fwd_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Fused backward of the same layer: quantises dY [M, N] along N (dgrad) and
 * along tokens (wgrad) in one pass, then runs DGRAD (dX [M, K]) and WGRAD
 * (dW [N, K]) with the tensors saved by bfp8_linear_fwd.
 *   dX, dW: bf16 outputs.  ws / ws_bytes: scratch of at least
 *   bfp8_linear_bwd_workspace_bytes().
 */
bfp8_status bfp8_linear_bwd(const void* dY,
                            const uint8_t* WqT, const float* sW,
                            const uint8_t* XqT, const float* sXT,
                            int64_t M, int64_t N, int64_t K,
                            void* dX, void* dW,
                            void* ws, size_t ws_bytes,
                            bfp8_stream_t stream);
size_t bfp8_linear_bwd_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Forward of one linear layer whose weight is already quantised: the
 * weight quantisation cached across micro-steps (W changes only at an
 * optimizer step, while section 3.2 re-quantises it on every use).  Wq E4M3
 * [N, K] and sW fp32 [N/128, K/128] are what bfp8_quantize_w_128x128 (or
 * _ex) returned for the current W; its WqT serves bfp8_linear_bwd.  Runs the
 * dual activation quantiser (scale_mode) and the FPROP GEMM.  X, Y, XqT,
 * sXT, the workspace (bfp8_linear_fwd_workspace_bytes) and errors are those
 * of bfp8_linear_fwd; Y equals bfp8_linear_fwd's output bit for bit when Wq
 * and sW come from the same W.
 */
bfp8_status bfp8_linear_fwd_prequantised(const void* X, const uint8_t* Wq, const float* sW,
                                         int64_t M, int64_t N, int64_t K,
                                         void* Y, uint8_t* XqT, float* sXT,
                                         void* ws, size_t ws_bytes,
                                         bfp8_scale_mode scale_mode, bfp8_stream_t stream);

/*
 * bfp8_linear_fwd / bfp8_linear_bwd with an explicit scale rule for every
 * quantisation they run (see bfp8_quantize_act_1x128_ex).  The saved tensors
 * carry fp32 scales in every mode; bfp8_linear_bwd_ex takes the mode for
 * the output-gradient quantisation only (the mode need not match the
 * forward's).  Arguments, workspaces and errors
 * are otherwise those of the calls without _ex; an unknown scale_mode
 * returns BFP8_EINVAL.
 */
bfp8_status bfp8_linear_fwd_ex(const void* X, const void* W,
                               int64_t M, int64_t N, int64_t K,
                               void* Y,
                               uint8_t* WqT, float* sW, uint8_t* XqT, float* sXT,
                               void* ws, size_t ws_bytes,
                               bfp8_scale_mode scale_mode, bfp8_stream_t stream);
bfp8_status bfp8_linear_bwd_ex(const void* dY,
                               const uint8_t* WqT, const float* sW,
                               const uint8_t* XqT, const float* sXT,
                               int64_t M, int64_t N, int64_t K,
                               void* dX, void* dW,
                               void* ws, size_t ws_bytes,
                               bfp8_scale_mode scale_mode, bfp8_stream_t stream);

/*
 * bfp8_linear_bwd_ex with the weight gradient added into an fp32 main
 * gradient instead of written as bf16: dW_main [N, K] fp32 (caller-owned,
 * read and written) += dY^T . X by bfp8_fp8_block_gemm_accumulate.  dX is
 * bf16 as before; workspace and errors as bfp8_linear_bwd.
 */
bfp8_status bfp8_linear_bwd_main_grad(const void* dY,
                                      const uint8_t* WqT, const float* sW,
                                      const uint8_t* XqT, const float* sXT,
                                      int64_t M, int64_t N, int64_t K,
                                      void* dX, float* dW_main,
                                      void* ws, size_t ws_bytes,
                                      bfp8_scale_mode scale_mode, bfp8_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns BFP8_ETIMEOUT if a kernel's bounded wait expired since the
 * last call (that kernel's outputs are then undefined), BFP8_ECUDA if the
 * synchronisation failed, else BFP8_OK.
 */
bfp8_status bfp8_sync_status(bfp8_stream_t stream);

/*
 * Sets the limit, in nanoseconds, of the device-side waits the kernels make
 * on the current device from now on (default 2e9); 0 restores the default.
 * Not affected: the waits a kernel makes on its way out for its own TMA
 * copies and MMAs still in flight, which have a fixed 5 s limit, so that a
 * kernel that gave up never leaves a copy into its shared memory or an MMA
 * into tensor memory it frees.  The tests shorten the limit and make a wait
 * expire on purpose (bfp8_test_stall_next_launch), then check that
 * bfp8_sync_status reports BFP8_ETIMEOUT and that the next call with the
 * default limit is exact.
 */
bfp8_status bfp8_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook of the timeout path (there is no counterpart in the paper).  The
 * next quantiser or GEMM kernel this library launches, on any device, first
 * makes one device-side wait on a barrier that nothing completes.  The wait
 * gives up after the current wait limit (bfp8_set_wait_limit_ns), the kernel
 * leaves early without starting any copy or MMA, and bfp8_sync_status reports
 * BFP8_ETIMEOUT; that call's outputs are undefined.  Later launches are
 * unaffected.  The hook only ever delays a kernel by the wait limit: it never
 * faults, traps or hangs the GPU.  Always returns BFP8_OK.
 */
bfp8_status bfp8_test_stall_next_launch(void);

/*
 * Selects the GEMM tiling for every later call in the process: 0 (default)
 * uses 256 x 256 output tiles computed by pairs of CTAs (tensor-core pair
 * MMAs) for FPROP and DGRAD whenever both output dimensions are multiples of
 * 256, and 128 x 256 (or 128 x 128) single-CTA tiles otherwise (always for
 * WGRAD); 1 always uses single-CTA tiles; 2 uses CTA pairs for WGRAD as well.
 * All give results within the same tolerance of the oracle.
 * Errors: EINVAL for any other value.
 */
bfp8_status bfp8_set_gemm_kernel(int kind);

/*
 * Overrides the split-K factor the GEMM picks (0 restores the automatic
 * choice, which splits the reduction only when that fills idle SMs at a
 * lower cost than the extra fp32 partial traffic).  Applies to every later
 * bfp8_fp8_block_gemm / linear call in the process and to the matching
 * *_workspace_bytes() results; the factor is capped at K/128.
 */
bfp8_status bfp8_set_gemm_splits(int splits);

/*
 * Number of kernels this library has launched in this process (all devices),
 * counted on the host at each launch.  A diagnostic for benchmarks that
 * report how many of the library's kernels ran in a timed region.
 */
uint64_t bfp8_launch_count(void);

/* Static description of a status code. */
const char* bfp8_status_string(bfp8_status status);

#ifdef __cplusplus
}
#endif

#endif /* BFP8_H */
