"""The SiLU-gated prologue (bfp8_swiglu_quantize_1x128) against the oracle.

h = bf16(SiLU(g) * u) is formed on the GPU with hardware 2^x and 1/x
approximations, so it is compared within one bf16 unit of the oracle's
exactly rounded h (and equal almost everywhere); the E4M3 codes and scales are
then required bit for bit against the oracle's quantisation of the GPU's own
h, in every scale mode, for both groupings.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import assert_codes_equal, assert_scales_equal, dev, np32, u8
from oracle import quant, swiglu
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu

MAX_DIFF_FRAC = 2e-3  # h values one bf16 unit from the oracle's, at most


def _ordered(bits):
    """bf16 bit patterns as integers ordered like their values (+-0 equal)."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def check_swiglu(gu_bf16, scale_mode):
    gu = gu_bf16.to(dev())
    h, q, s, qT, sT = ops.swiglu_quantize_1x128(gu, want_h=True, scale_mode=scale_mode)
    assert ops.sync_status() == 0
    # h within one bf16 unit of the oracle's exactly rounded value
    oh = swiglu.swiglu(np32(gu_bf16))
    gb = (np32(h).view(np.uint32) >> 16).astype(np.uint16)
    ob = (oh.view(np.uint32) >> 16).astype(np.uint16)
    d = np.abs(_ordered(gb) - _ordered(ob))
    assert d.max() <= 1, f"h differs by {d.max()} bf16 units"
    assert np.count_nonzero(d) <= MAX_DIFF_FRAC * d.size + 2, f"{np.count_nonzero(d)} of {d.size} h values differ"
    # the codes are the mode's quantisation of this h, bit for bit
    hn = np32(h)
    oq, os_ = quant.quantize_act_1x128(hn, scale_mode)
    oqT, osT = quant.quantize_act_tokens_1x128(hn, scale_mode)
    assert_codes_equal(u8(q), oq, "q")
    assert_scales_equal(s.cpu().numpy(), os_, "s")
    assert_codes_equal(u8(qT), oqT, "qT")
    assert_scales_equal(sT.cpu().numpy(), osT, "sT")
    # without the h copy, and with one grouping at a time, the same bytes
    _, q2, s2, qT2, sT2 = ops.swiglu_quantize_1x128(gu, scale_mode=scale_mode)
    _, q3, s3, _, _ = ops.swiglu_quantize_1x128(gu, rows=True, tokens=False, scale_mode=scale_mode)
    _, _, _, qT4, sT4 = ops.swiglu_quantize_1x128(gu, rows=False, tokens=True, scale_mode=scale_mode)
    assert ops.sync_status() == 0
    for a, b in ((q2, q), (s2, s), (qT2, qT), (sT2, sT), (q3, q), (s3, s), (qT4, qT), (sT4, sT)):
        assert torch.equal(a, b)
    return d


def _gated_input(M, F, seed, extremes=False):
    rng = np.random.default_rng(seed)
    gu = (rng.standard_t(4, (M, 2 * F)) * 0.5).astype(np.float32)
    if extremes:
        # the wide exponent path (|g| > 64), signed zeros, huge u and values
        # whose h falls below the fp32 normal range
        g = gu[:, :F]
        u = gu[:, F:]
        sel = rng.random((M, F))
        g[sel < 0.002] = -70.0
        g[(sel >= 0.002) & (sel < 0.004)] = -100.0
        g[(sel >= 0.004) & (sel < 0.006)] = 90.0
        g[(sel >= 0.006) & (sel < 0.007)] = -0.0
        u[(sel >= 0.007) & (sel < 0.009)] = 3.0e4
        g[(sel >= 0.009) & (sel < 0.010)] = -88.5
        u[(sel >= 0.009) & (sel < 0.010)] = 1.0e6
        g[(sel >= 0.010) & (sel < 0.011)] = -300.0
    return workloads.to_bf16(gu)


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
@pytest.mark.parametrize("M,F", [(128, 128), (384, 640), (1152, 256)])
def test_small_shapes(M, F, scale_mode):
    check_swiglu(_gated_input(M, F, M + F), scale_mode)


@pytest.mark.parametrize("scale_mode", ["amax448", "mul_recip"])
def test_extreme_gates_take_the_wide_path(scale_mode):
    check_swiglu(_gated_input(512, 384, 9, extremes=True), scale_mode)


def test_full_size_down_projection_input():
    """The mlp_down recipe's gate+up output [8192, 12288] (G, U ~ 0.5 t(4))."""
    wl = workloads.make("mlp_down")
    d = check_swiglu(workloads.tensor(wl, "gu"), "amax448")
    assert np.count_nonzero(d) <= 1e-3 * d.size


def test_rejects_a_gate_up_with_odd_width():
    gu = torch.zeros((128, 129), dtype=torch.bfloat16, device=dev())
    with pytest.raises(ValueError):
        ops.swiglu_quantize_1x128(gu)
