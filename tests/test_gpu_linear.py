"""Fused linear forward/backward through the C ABI vs the oracle's composed
linear: saved FP8 tensors bit-exact, outputs within relative Frobenius 1e-3."""

import numpy as np
import pytest
import torch

from gpu_helpers import (REL_FRO_TOL, assert_codes_equal, assert_scales_equal, dev, np32, rel_fro, sample_index, u8)
from oracle import gemm as ogemm
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def check_linear(X, W, dY, rows=None):
    Xg, Wg, dYg = X.to(dev()), W.to(dev()), dY.to(dev())
    Y, saved = ops.linear_fwd(Xg, Wg)
    dX, dW = ops.linear_bwd(dYg, saved)
    assert ops.sync_status() == 0
    Xn, Wn, dYn = np32(X), np32(W), np32(dY)
    oY, osaved = ogemm.linear_fwd(Xn, Wn)
    for k in ("WqT", "XqT"):
        assert_codes_equal(u8(saved[k]), osaved[k], k)
    for k in ("sW", "sXT"):
        assert_scales_equal(saved[k].cpu().numpy(), osaved[k], k)
    assert rel_fro(np32(Y), oY) <= REL_FRO_TOL
    odX, odW = ogemm.linear_bwd(dYn, osaved)
    assert rel_fro(np32(dX), odX) <= REL_FRO_TOL
    assert rel_fro(np32(dW), odW) <= REL_FRO_TOL


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (384, 640, 512), (1024, 768, 1280)])
def test_linear_small(M, N, K):
    rng = np.random.default_rng(M * N + K)
    X = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = workloads.to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    dY = workloads.to_bf16((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    check_linear(X, W, dY)


def test_linear_repeat_is_deterministic():
    rng = np.random.default_rng(0)
    X = workloads.to_bf16(rng.standard_normal((512, 768)).astype(np.float32)).to(dev())
    W = workloads.to_bf16((rng.standard_normal((640, 768)) * 0.02).astype(np.float32)).to(dev())
    dY = workloads.to_bf16((rng.standard_normal((512, 640)) * 1e-3).astype(np.float32)).to(dev())
    outs = []
    for _ in range(2):
        Y, saved = ops.linear_fwd(X, W)
        dX, dW = ops.linear_bwd(dY, saved)
        outs.append((Y.clone(), dX.clone(), dW.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
def test_prequantised_weights_give_the_same_forward(scale_mode):
    """Weights quantised once (cached across micro-steps) and passed to the
    prequantised forward give linear_fwd's output and saved tensors bit for
    bit; the backward runs from them unchanged."""
    rng = np.random.default_rng(31)
    X = workloads.to_bf16(rng.standard_normal((512, 384)).astype(np.float32)).to(dev())
    W = workloads.to_bf16((rng.standard_normal((640, 384)) * 0.02).astype(np.float32)).to(dev())
    dY = workloads.to_bf16((rng.standard_normal((512, 640)) * 1e-3).astype(np.float32)).to(dev())
    Y, saved = ops.linear_fwd(X, W, scale_mode=scale_mode)
    Wq, WqT, sW = ops.quantize_w_128x128(W, scale_mode=scale_mode)
    for _ in range(2):  # the cached weight serves several micro-steps
        Y2, saved2 = ops.linear_fwd_prequantised(X, Wq, sW, WqT=WqT, scale_mode=scale_mode)
        assert ops.sync_status() == 0
        assert torch.equal(Y2, Y)
        for k in ("WqT", "sW", "XqT", "sXT"):
            assert torch.equal(saved2[k], saved[k]), k
    dX, dW = ops.linear_bwd(dY, saved, scale_mode=scale_mode)
    dX2, dW2 = ops.linear_bwd(dY, saved2, scale_mode=scale_mode)
    assert torch.equal(dX, dX2) and torch.equal(dW, dW2)
