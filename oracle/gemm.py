"""Block-scaled FP8 GEMM with fp32 promotion per 128-deep slice (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090"
(papers.lianghsun.dev translation), section 3.2: the Transformer linear-layer
GEMMs take E4M3 operands whose scales belong to 1x128 groups (activations and
activation gradients, along the reduction dimension) and 128x128 blocks
(weights), with training state kept in BF16/FP32 (section 2 overview and 3.2).

Definition used (reduction split into slices kb of 128 consecutive indices,
each slice lying inside exactly one scale group of both operands):

    P_kb[i, j] = sum_{k in kb} dec(A[i, k]) * dec(B[j, k])      (exact, fp64)
    acc[i, j]  = 0;  for kb ascending:
    acc[i, j]  = f32( acc + f32( f32(P_kb) * f32(sa(i, kb) * sb(j, kb)) ) )
    C[i, j]    = bf16_rn(acc[i, j])

The fp64 sum is exact: every E4M3 value is an integer <= 15 times 2^k with
-9 <= k <= 5, so every product and every partial sum of 128 products is an
integer multiple of 2^-18 below 2^25, which binary64 holds exactly whatever
the summation order.  That is why a library fp64 matmul may serve as the
per-slice step.

Layouts (M, N, K are the output rows, output columns and reduction length of
the GEMM being run; X [M_tok, K_in], W [N_out, K_in], dY [M_tok, N_out]):

* fprop  Y  = X  . W^T :  A = Xq   [M_tok, K_in],  sa = sX   [K_in/128, M_tok]
                          B = Wq   [N_out, K_in],  sb(j, kb) = sW[j/128, kb]
* dgrad  dX = dY . W   :  A = dYq  [M_tok, N_out], sa = sdY  [N_out/128, M_tok]
                          B = WqT  [K_in, N_out],  sb(j, kb) = sW[kb, j/128]
* wgrad  dW = dY^T . X :  A = dYqT [N_out, M_tok], sa = sdYT [M_tok/128, N_out]
                          B = XqT  [K_in, M_tok],  sb(j, kb) = sXT[kb, j]
"""

import numpy as np

from .formats import e4m3_decode, bf16_round
from . import quant

GROUP = 128


def _slices(K):
    if K % GROUP:
        raise ValueError(f"reduction length {K} is not a multiple of {GROUP}")
    return K // GROUP


def block_scaled_gemm(A_q, B_q, sa_of, sb_of, rows=None, cols=None):
    """Core promotion loop.

    A_q uint8 [M, K], B_q uint8 [N, K] (both K contiguous).
    sa_of(kb) -> float32 [M] (scale of each A row for slice kb);
    sb_of(kb) -> float32 [N] (scale of each B row for slice kb).
    rows / cols optionally restrict the computed outputs to a subset (the
    value of C[i, j] depends only on row i of A and row j of B).
    Returns (acc float32 [m, n], out float32 bf16-valued [m, n]).
    """
    A_q = np.asarray(A_q, dtype=np.uint8)
    B_q = np.asarray(B_q, dtype=np.uint8)
    if A_q.shape[1] != B_q.shape[1]:
        raise ValueError("A and B reduction lengths differ")
    ri = np.arange(A_q.shape[0]) if rows is None else np.asarray(rows)
    ci = np.arange(B_q.shape[0]) if cols is None else np.asarray(cols)
    A = e4m3_decode(A_q[ri])  # float64
    B = e4m3_decode(B_q[ci])
    acc = np.zeros((len(ri), len(ci)), dtype=np.float32)
    for kb in range(_slices(A_q.shape[1])):
        ks = slice(kb * GROUP, (kb + 1) * GROUP)
        P = A[:, ks] @ B[:, ks].T  # exact in fp64
        sa = np.asarray(sa_of(kb), dtype=np.float32)[ri]
        sb = np.asarray(sb_of(kb), dtype=np.float32)[ci]
        scale = sa[:, None] * sb[None, :]  # float32 * float32 -> float32
        term = P.astype(np.float32) * scale  # f32(P) * f32(scale), rounded to f32
        acc = acc + term  # float32 + float32 -> float32
    return acc, bf16_round(acc)


def fprop(Xq, sX, Wq, sW, rows=None, cols=None):
    """Y[m, n] for Y = X . W^T.  Returns (acc fp32, Y bf16-valued fp32)."""
    sX = np.asarray(sX, dtype=np.float32)
    sW = np.asarray(sW, dtype=np.float32)
    N = np.asarray(Wq).shape[0]
    return block_scaled_gemm(
        Xq, Wq,
        lambda kb: sX[kb, :],
        lambda kb: sW[np.arange(N) // GROUP, kb],
        rows, cols)


def dgrad(dYq, sdY, WqT, sW, rows=None, cols=None):
    """dX[m, k] for dX = dY . W (reduction over the layer's output features)."""
    sdY = np.asarray(sdY, dtype=np.float32)
    sW = np.asarray(sW, dtype=np.float32)
    K_in = np.asarray(WqT).shape[0]
    return block_scaled_gemm(
        dYq, WqT,
        lambda kb: sdY[kb, :],
        lambda kb: sW[kb, np.arange(K_in) // GROUP],
        rows, cols)


def wgrad(dYqT, sdYT, XqT, sXT, rows=None, cols=None):
    """dW[n, k] for dW = dY^T . X (reduction over tokens)."""
    sdYT = np.asarray(sdYT, dtype=np.float32)
    sXT = np.asarray(sXT, dtype=np.float32)
    return block_scaled_gemm(
        dYqT, XqT,
        lambda kb: sdYT[kb, :],
        lambda kb: sXT[kb, :],
        rows, cols)


def accumulate_into(main, acc):
    """fp32 accumulate-into: main_new = f32(main + acc), one IEEE addition per
    element.

    acc is the GEMM's fp32 promotion accumulator (before the bf16 rounding of
    the plain output).  This is how a weight gradient lands in an fp32 main
    gradient: section 3.2 keeps the training state on the BF16/FP32 path and
    uses FP8 only as the online compute format of the linear layers.
    """
    return (np.asarray(main, dtype=np.float32) + np.asarray(acc, dtype=np.float32)).astype(np.float32)


def linear_fwd(X, W, scale_mode="amax448"):
    """Quantise W (128x128) and X (1x128 along features, and along tokens for
    the later wgrad) under the quantisers' scale_mode, then run fprop.

    Returns (Y bf16-valued float32 [M, N], saved dict).  ``saved`` holds what
    the backward pass reuses: FP8 is the storage format of the saved
    activation (section 3.2), and W is re-quantised on every use.
    """
    Wq, WqT, sW = quant.quantize_w_128x128(W, scale_mode)
    Xq, sX = quant.quantize_act_1x128(X, scale_mode)
    XqT, sXT = quant.quantize_act_tokens_1x128(X, scale_mode)
    _, Y = fprop(Xq, sX, Wq, sW)
    saved = dict(Wq=Wq, WqT=WqT, sW=sW, Xq=Xq, sX=sX, XqT=XqT, sXT=sXT)
    return Y, saved


def linear_bwd(dY, saved, main_grad=None, scale_mode="amax448"):
    """Quantise dY along features (for dgrad) and along tokens (for wgrad)
    under scale_mode, then run dgrad and wgrad.  Returns (dX, dW) as
    bf16-valued float32; with main_grad (fp32 [N, K]) dW is instead
    main_grad + the wgrad accumulator (accumulate_into), returned as a new
    float32 array."""
    dYq, sdY = quant.quantize_act_1x128(dY, scale_mode)
    dYqT, sdYT = quant.quantize_act_tokens_1x128(dY, scale_mode)
    _, dX = dgrad(dYq, sdY, saved["WqT"], saved["sW"])
    acc, dW = wgrad(dYqT, sdYT, saved["XqT"], saved["sXT"])
    if main_grad is not None:
        dW = accumulate_into(main_grad, acc)
    return dX, dW
