"""MXFP8 1x32 recipe (oracle side): the finer-grained scaling workload that
the blockwise 1x128 / 128x128 recipe is compared against.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the bloombook.cn tutorial's FP8 paragraph and its MXFP concept figure.
MXFP8 gives every 32 consecutive elements their own shared scale X, and a
stored code decodes as V_i = Q_i * X.  Section 3.2 of "Puro-2B: Poor Lab's
Qwen2-1.5B Trained on RTX 5090 within $5090" runs its own 1x128 / 128x128
recipe on SM120 through that hardware path, with power-of-two block scales.

Readings where the pages are silent:

* the scale of a group is the power-of-two rule of ``quant.group_scale_pow2``
  (the smallest 2^k >= amax/448, so nothing saturates), with k clamped to the
  E8M0 exponent range [-127, 127];
* groups run along the GEMM reduction dimension for every operand, weights
  included (MX has no 2-D blocks).  The dgrad operand W^T is therefore
  quantised on its own, along the layer's output features;
* the GEMM promotes each 32-deep slice in fp32, in ascending order, as the
  1x128 GEMM promotes its 128-deep slices:
      acc = f32(acc + f32(f32(P_kb) * f32(sa(i, kb) * sb(j, kb)))),
  with P_kb the exact fp64 sum of 32 decoded products.

Scale layouts follow the 1x128 ones with 32 in place of 128:
quantize_mx_1x32(X [R, C]) -> q [R, C], s [C/32, R];
quantize_mx_tokens_1x32(X [M, K]) -> qT [K, M], sT [M/32, K].
"""

import numpy as np

from .formats import bf16_round, e4m3_decode
from . import quant

MX_GROUP = 32
E8M0_KMIN, E8M0_KMAX = -127, 127


def mx_scale(amax):
    """Power-of-two scale of a 32-group, clamped to the E8M0 range."""
    s = quant.group_scale_pow2(amax).astype(np.float64)
    return np.clip(s, 2.0 ** E8M0_KMIN, 2.0 ** E8M0_KMAX).astype(np.float32)


def quantize_mx_1x32(x):
    """Quantise X [R, C] in 1x32 groups along C.  Returns (q uint8 [R, C],
    s float32 [C/32, R])."""
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % MX_GROUP:
        raise ValueError(f"x must be 2-D with columns a multiple of {MX_GROUP}")
    R, C = x.shape
    xg = x.reshape(R, C // MX_GROUP, MX_GROUP)
    amax = np.nanmax(np.abs(xg), axis=2) if xg.size else np.zeros((R, C // MX_GROUP), np.float32)
    s = mx_scale(amax)
    q = quant.quantize_values(xg, s[:, :, None]).reshape(R, C)
    return q, np.ascontiguousarray(s.T)


def quantize_mx_tokens_1x32(x):
    """Quantise X [M, K] in groups of 32 tokens per column, stored transposed.
    Returns (qT uint8 [K, M], sT float32 [M/32, K])."""
    x = np.asarray(x, dtype=np.float32)
    return quantize_mx_1x32(np.ascontiguousarray(x.T))


def mx_gemm(A_q, sA, B_q, sB, rows=None, cols=None):
    """C = A . B^T from 1x32-quantised operands, A_q [M, K] with sA [K/32, M]
    and B_q [N, K] with sB [K/32, N], promoted per 32-deep slice.
    Returns (acc float32, out float32 bf16-valued)."""
    A_q = np.asarray(A_q, dtype=np.uint8)
    B_q = np.asarray(B_q, dtype=np.uint8)
    sA = np.asarray(sA, dtype=np.float32)
    sB = np.asarray(sB, dtype=np.float32)
    K = A_q.shape[1]
    if B_q.shape[1] != K or K % MX_GROUP:
        raise ValueError("reduction lengths differ or are not multiples of 32")
    ri = np.arange(A_q.shape[0]) if rows is None else np.asarray(rows)
    ci = np.arange(B_q.shape[0]) if cols is None else np.asarray(cols)
    A = e4m3_decode(A_q[ri])
    B = e4m3_decode(B_q[ci])
    acc = np.zeros((len(ri), len(ci)), dtype=np.float32)
    for kb in range(K // MX_GROUP):
        ks = slice(kb * MX_GROUP, (kb + 1) * MX_GROUP)
        P = A[:, ks] @ B[:, ks].T  # exact in fp64 (32 products of E4M3 values)
        scale = sA[kb, ri][:, None] * sB[kb, ci][None, :]  # float32 product
        acc = acc + P.astype(np.float32) * scale
    return acc, bf16_round(acc)


def mx_linear_fwd(X, W):
    """Y = X . W^T with both operands 1x32-quantised along the in-features."""
    Xq, sX = quantize_mx_1x32(X)
    Wq, sW = quantize_mx_1x32(W)
    return mx_gemm(Xq, sX, Wq, sW)[1]


def mx_linear_bwd(dY, X, W):
    """(dX, dW) for Y = X . W^T: dgrad reduces over out-features (dY and W^T
    quantised along them), wgrad over tokens (dY^T and X^T along tokens)."""
    dYq, sdY = quantize_mx_1x32(dY)
    WTq, sWT = quantize_mx_1x32(np.ascontiguousarray(np.asarray(W, np.float32).T))
    dX = mx_gemm(dYq, sdY, WTq, sWT)[1]
    dYqT, sdYT = quantize_mx_tokens_1x32(dY)
    XqT, sXT = quantize_mx_tokens_1x32(X)
    dW = mx_gemm(dYqT, sdYT, XqT, sXT)[1]
    return dX, dW
