"""Blockwise E4M3 quantisers (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090"
(papers.lianghsun.dev translation), section 3.2 "FP8 mixed-precision
training": activations and activation gradients use 1-D groups of 128
consecutive values along the GEMM reduction dimension, weights use 2-D
128x128 blocks, and each group's scale is computed online from that group.
The decoded value of a stored code is code * scale (the MXFP concept figure on
the bloombook.cn tutorial page, "V_i = Q_i x X"), so the scale stored here is a
dequantisation multiplier.

One group G (128 values, or 128x128 values for a weight block) is quantised as

1. amax = max |x| over G, in float32, ignoring NaN (fmaxf semantics);
2. s = 1.0 if amax == 0 else float32(amax / 448)          (one IEEE division);
3. q = E4M3_rn_satfinite(float32(x / s)) for every x in G (one IEEE division,
   then one rounding to E4M3).

Readings where the pages are silent: the scale is an arbitrary fp32 value
amax/448 (not the power of two used on SM120); quantisation divides by s
rather than multiplying by 448/amax; an all-zero group gets s = 1.

Power-of-two mode (scale_mode="pow2").  Section 3.2 of the paper runs the
same grouping on SM120 through the hardware MXFP8 path, whose scales are
powers of two.  In this mode s is the smallest power of two with
s >= amax/448, i.e. s = 2^ceil(log2(amax/448)), so no value of the group
saturates and the largest lands in (224, 448]; an all-zero group keeps
s = 1.  Step 3 is unchanged: x/s with s a power of two is an exact scaling
(rounded once only where it leaves the fp32 range).

Reciprocal-multiply mode (scale_mode="mul_recip").  The pages do not say
whether a code comes from dividing by the scale or from multiplying by its
reciprocal; this mode takes the second reading.  The stored scale is the
default mode's s = float32(amax / 448), so the GEMMs consume it unchanged,
and each group's codes are q = E4M3_rn_satfinite(float32(x * m)) with one
multiplier per group, m = float32(448 / amax) (one IEEE division per group,
none per element).  m saturates at the largest finite float32, which only a
group with amax below 448 / FLT_MAX (about 2^-119.2) reaches; an all-zero
group gets m = 1.  The two roundings (of m, then of x * m) make some codes
one E4M3 step away from the default mode's, near the E4M3 rounding midpoints.

Scale layouts (shared with the C ABI, which states the same contract):

* quantize_act_1x128(X [R, C]) groups along C:  q [R, C],  s [C/128, R]
  (s[g, r] is the scale of row r's g-th group: group-major, so the 128 row
  scales of one group index are contiguous);
* quantize_act_tokens_1x128(X [M, K]) groups along M (tokens) and stores the
  transpose:  qT [K, M],  sT [M/128, K];
* quantize_w_128x128(W [N, K]):  q [N, K],  qT [K, N] (= q transposed),
  s [N/128, K/128].
"""

import numpy as np

from .formats import e4m3_encode

GROUP = 128
E4M3_MAX = np.float32(448.0)


def _check_bf16_grid(x, name):
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError(f"{name} must be 2-D")
    if x.shape[0] % GROUP or x.shape[1] % GROUP:
        raise ValueError(f"{name} dims must be multiples of {GROUP}, got {x.shape}")
    return x


def group_scale(amax):
    """Scale of a group from its amax: amax/448 in fp32, or 1 when amax == 0."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / E4M3_MAX  # float32 / float32 -> float32, IEEE round to nearest
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def group_scale_pow2(amax):
    """Power-of-two scale of a group: the smallest 2^k >= amax/448 (1 when
    amax == 0), as float32.

    t = amax/448 is formed in float64.  For a float32 amax that quotient is
    either exactly a power of two (amax = 7 * 2^j) or further than 2^-26 in
    relative terms from every power of two (amax has at most 24 significant
    bits, so amax/7 cannot come closer), far more than the 2^-53 rounding of
    the float64 division; ceil(log2(t)) is therefore read off frexp exactly:
    t = f * 2^e with f in [0.5, 1) gives k = e - 1 when f == 0.5, else e.
    """
    amax = np.asarray(amax, dtype=np.float32)
    t = amax.astype(np.float64) / 448.0
    f, e = np.frexp(t)
    k = np.where(f == 0.5, e - 1, e)
    s = np.ldexp(np.float64(1.0), k).astype(np.float32)  # 2^k for k in [-141, 120]: exact in float32
    return np.where(amax == 0, np.float32(1.0), s).astype(np.float32)


def group_multiplier(amax):
    """Code multiplier of the reciprocal-multiply mode: float32(448 / amax) by
    one IEEE float32 division, saturated at the largest finite float32; 1 when
    amax == 0."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        m = E4M3_MAX / amax  # float32 / float32 -> float32, IEEE round to nearest
    m = np.minimum(m, np.finfo(np.float32).max)
    return np.where(amax == 0, np.float32(1.0), m).astype(np.float32)


# the stored (dequantisation) scale of each mode
SCALE_MODES = {"amax448": group_scale, "pow2": group_scale_pow2, "mul_recip": group_scale}


def _scale_fn(scale_mode):
    try:
        return SCALE_MODES[scale_mode]
    except KeyError:
        raise ValueError(f"unknown scale_mode {scale_mode!r}") from None


def quantize_values(x, s):
    """q = E4M3(float32(x / s)), elementwise with broadcasting."""
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        y = x / s  # float32 division
    return e4m3_encode(y)


def quantize_values_mul(x, m):
    """q = E4M3(float32(x * m)), elementwise with broadcasting."""
    x = np.asarray(x, dtype=np.float32)
    m = np.asarray(m, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        y = x * m  # float32 product, IEEE round to nearest
    return e4m3_encode(y)


def _group_codes(x, amax, s, scale_mode):
    """Codes of the values x (broadcast against their group's amax and s)
    under the mode's rule: x / s, or x * m in the reciprocal-multiply mode."""
    if scale_mode == "mul_recip":
        return quantize_values_mul(x, group_multiplier(amax))
    return quantize_values(x, s)


def quantize_act_1x128(x, scale_mode="amax448"):
    """Quantise X [R, C] in 1x128 groups along C.

    Returns (q uint8 [R, C], s float32 [C/128, R]).
    """
    x = _check_bf16_grid(x, "x")
    R, C = x.shape
    xg = x.reshape(R, C // GROUP, GROUP)
    amax = np.nanmax(np.abs(xg), axis=2) if xg.size else np.zeros((R, C // GROUP), np.float32)
    s = _scale_fn(scale_mode)(amax)  # [R, C/128]
    q = _group_codes(xg, amax[:, :, None], s[:, :, None], scale_mode).reshape(R, C)
    return q, np.ascontiguousarray(s.T)


def quantize_act_tokens_1x128(x, scale_mode="amax448"):
    """Quantise X [M, K] in groups of 128 consecutive rows (tokens) per column.

    This is the grouping that the weight-gradient GEMM needs, where the
    reduction runs over tokens.  The codes are stored transposed.
    Returns (qT uint8 [K, M], sT float32 [M/128, K]).
    """
    x = _check_bf16_grid(x, "x")
    return quantize_act_1x128(np.ascontiguousarray(x.T), scale_mode)


def quantize_w_128x128(w, scale_mode="amax448"):
    """Quantise W [N, K] in 128x128 blocks.

    Returns (q uint8 [N, K], qT uint8 [K, N], s float32 [N/128, K/128]).
    """
    w = _check_bf16_grid(w, "w")
    N, K = w.shape
    wb = w.reshape(N // GROUP, GROUP, K // GROUP, GROUP)
    amax = np.nanmax(np.abs(wb), axis=(1, 3)) if wb.size else np.zeros((N // GROUP, K // GROUP), np.float32)
    s = _scale_fn(scale_mode)(amax)  # [N/128, K/128]
    q = _group_codes(wb, amax[:, None, :, None], s[:, None, :, None], scale_mode).reshape(N, K)
    return q, np.ascontiguousarray(q.T), s


def quantize_per_tensor(x):
    """Comparator: one scale for the whole tensor (the scheme the paper moves
    away from because a few outliers widen every value's quantisation step).

    Returns (q uint8 same shape, s float32 scalar).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.nanmax(np.abs(x))) if x.size else np.float32(0)
    s = group_scale(amax)
    return quantize_values(x, s), np.float32(s)
