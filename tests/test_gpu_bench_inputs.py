"""The stack28 benchmark's own inputs through the GPU path, against the oracle.

bench.py draws the stack28 tensors on the device (workloads.tensor_cuda: the
same distributions as the CPU recipe, different values) to keep start-up
short.  These tests draw them the same way, run the quantisers and GEMMs the
bench runs, and compare with the oracle on the very same values: codes and
scales bit for bit, GEMM outputs within the relative Frobenius tolerance on
sampled 128 x 128 tiles."""

import numpy as np
import pytest
import torch

from gpu_helpers import REL_FRO_TOL, assert_codes_equal, assert_scales_equal, dev, np32, rel_fro, u8
from oracle import gemm as ogemm
from oracle import quant
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def bench_input(wl, tag, layer=None):
    """One stack28 input exactly as bench.py draws it."""
    return workloads.tensor_cuda(wl, tag, layer, device=dev()).contiguous()


def tiles(n, count, rng):
    """Indices of `count` whole 128-blocks of [0, n), seeded."""
    blocks = np.sort(rng.choice(n // 128, count, replace=False))
    return (blocks[:, None] * 128 + np.arange(128)).ravel()


def check_act(x):
    q, s, qT, sT = ops.quantize_act_1x128(x, rows=True, tokens=True)
    assert ops.sync_status() == 0
    xn = np32(x)
    oq, os_ = quant.quantize_act_1x128(xn)
    oqT, osT = quant.quantize_act_tokens_1x128(xn)
    assert_codes_equal(u8(q), oq, "q")
    assert_scales_equal(s.cpu().numpy(), os_, "s")
    assert_codes_equal(u8(qT), oqT, "qT")
    assert_scales_equal(sT.cpu().numpy(), osT, "sT")
    return (q, s, qT, sT), (oq, os_, oqT, osT)


def test_layer0_quantisers_and_gemms_on_the_bench_inputs():
    """Layer 0's O projection as the bench step runs it: the batched weight
    quantiser over the layer's four weights, the dual activation quantiser on
    x_h and dy_o, then FPROP, DGRAD and WGRAD."""
    wl = workloads.make("stack28")
    rng = np.random.default_rng(2026)
    ws = [bench_input(wl, t, 0) for t in ("w_qkv", "w_o", "w_gu", "w_down")]
    got_w = ops.quantize_w_batch(ws)
    assert ops.sync_status() == 0
    ow = []
    for w, (q, qT, s) in zip(ws, got_w):
        oq, oqT, os_ = quant.quantize_w_128x128(np32(w))
        assert_codes_equal(u8(q), oq, "Wq")
        assert_codes_equal(u8(qT), oqT, "WqT")
        assert_scales_equal(s.cpu().numpy(), os_, "sW")
        ow.append((oq, oqT, os_))
    Wq, WqT, sW = got_w[1]
    oWq, oWqT, osW = ow[1]

    (Xq, sX, XqT, sXT), (oXq, osX, oXqT, osXT) = check_act(bench_input(wl, "x_h"))
    (dYq, sdY, dYqT, sdYT), (odYq, osdY, odYqT, osdYT) = check_act(bench_input(wl, "dy_o"))

    M, K = Xq.shape
    N = Wq.shape[0]
    cases = [("fprop", ops.FPROP, (Xq, sX, Wq, sW), (oXq, osX, oWq, osW), M, N),
             ("dgrad", ops.DGRAD, (dYq, sdY, WqT, sW), (odYq, osdY, oWqT, osW), M, K),
             ("wgrad", ops.WGRAD, (dYqT, sdYT, XqT, sXT), (odYqT, osdYT, oXqT, osXT), N, K)]
    for name, lay, gargs, oargs, R, C in cases:
        out = ops.fp8_block_gemm(lay, *gargs)
        assert ops.sync_status() == 0
        rows, cols = tiles(R, 3, rng), tiles(C, 3, rng)
        want = getattr(ogemm, name)(*oargs, rows=rows, cols=cols)[1]
        got = np32(out)[np.ix_(rows, cols)]
        err = rel_fro(got, want)
        assert err <= REL_FRO_TOL, (name, err)


@pytest.mark.parametrize("tag", ["x_f", "dy_qkv", "dy_down"])
def test_activation_quantiser_on_the_bench_inputs(tag):
    check_act(bench_input(workloads.make("stack28"), tag))
