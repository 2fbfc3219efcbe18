"""SiLU-gated FFN activation followed by the 1x128 activation quantiser (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the down projection of Puro-2B's FFN takes h = SiLU(g) * u, where
[g || u] is the output of the fused gate+up projection.  The bloombook.cn
tutorial's model-architecture paragraph gives a Qwen3-1.7B-compatible
configuration with FFN width 6144; a SiLU-gated FFN is the reading taken for
that configuration.  Section 3.2 of "Puro-2B: Poor Lab's Qwen2-1.5B Trained
on RTX 5090 within $5090" keeps everything outside the linear layers' operands
on the BF16/FP32 path, so h is a bf16 tensor; the down projection then
quantises it like any activation (1x128 groups along its features for fprop,
and along tokens, stored transposed, for wgrad).

Definition used here, per element:

    h = bf16_rn( g * u / (1 + exp(-g)) )

evaluated in float64 and rounded once to bf16 (round to nearest, ties to
even).  The float64 evaluation is off by a few units of 2^-53 relative, so it
can only round differently from the exact value when the product lies within
that distance of a bf16 rounding midpoint.
"""

import numpy as np

from . import quant


def bf16_round_f64(v):
    """Round float64 values directly to bfloat16 (one rounding, ties to even,
    gradual underflow, overflow to inf).  Returns float32 arrays holding
    bf16-representable values (NaN stays NaN)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(v)                       # |v| = f 2^e, f in [0.5, 1)
        qexp = np.maximum(e - 8, -133)           # bf16 quantum: 8 significant bits, 2^-133 below 2^-126
        r = np.round(np.ldexp(v, -qexp))         # exact scaling, then round half to even
        out = np.ldexp(r, qexp)
        out = np.where(np.isfinite(v), out, v)
        return out.astype(np.float32)            # exact (bf16 values), or inf past the largest finite


def swiglu(gu):
    """h [M, F] from the gate+up output gu [M, 2F] (gate in columns 0..F-1,
    up in F..2F-1), bf16 values held in float32."""
    gu = np.asarray(gu, dtype=np.float32)
    if gu.ndim != 2 or gu.shape[1] % 2:
        raise ValueError("gu must be [M, 2F]")
    F = gu.shape[1] // 2
    g = gu[:, :F].astype(np.float64)
    u = gu[:, F:].astype(np.float64)
    with np.errstate(over="ignore"):
        h = g * u / (1.0 + np.exp(-g))
    return bf16_round_f64(h)


def quantize_swiglu_1x128(gu, scale_mode="amax448"):
    """h = swiglu(gu), then both 1x128 quantisations of h that the down
    projection needs.  Returns (h, q [M, F], s [F/128, M], qT [F, M],
    sT [M/128, F])."""
    h = swiglu(gu)
    q, s = quant.quantize_act_1x128(h, scale_mode)
    qT, sT = quant.quantize_act_tokens_1x128(h, scale_mode)
    return h, q, s, qT, sT
