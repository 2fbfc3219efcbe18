"""The bounded-wait timeout path, exercised on the GPU without a fault.

Every device-side wait of the kernels gives up after a limit, raises the
device error word and lets the kernel leave early; bfp8_sync_status then
reports BFP8_ETIMEOUT and the context stays usable.  A wait is made to expire
on purpose with the library's test hook (the next launch first waits on a
barrier that nothing completes) under a short limit.  On its way out the
kernel waits for its own copies and MMAs with a fixed long limit, so nothing
is left in flight: the next call, with the default limit, must again match
the oracle exactly (codes and scales) or within the GEMM tolerance.
"""

import numpy as np
import pytest

from gpu_helpers import REL_FRO_TOL, assert_codes_equal, assert_scales_equal, np32, rel_fro, to_gpu, u8
from oracle import gemm as ogemm, quant
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu

ETIMEOUT = 5
LIMIT_NS = 2_000_000  # 2 ms: the stalled launch gives up quickly


def stalled(call):
    """Runs call() with its first launch stalled under a short wait limit;
    returns the device status reported afterwards."""
    assert ops.sync_status() == 0
    ops.set_wait_limit_ns(LIMIT_NS)
    try:
        ops.test_stall_next_launch()
        call()
        return ops.sync_status()
    finally:
        ops.set_wait_limit_ns(0)


def operands(M, K, seed):
    rng = np.random.default_rng(seed)
    return workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32))


@pytest.mark.parametrize("weight", [False, True], ids=["activation", "weight"])
def test_quantiser_timeout_then_exact(weight):
    x = operands(256, 384, 1)
    xg = x.to("cuda")
    if weight:
        assert stalled(lambda: ops.quantize_w_128x128(xg)) == ETIMEOUT
        q, qT, s = ops.quantize_w_128x128(xg)
        assert ops.sync_status() == 0
        oq, oqT, os_ = quant.quantize_w_128x128(np32(x))
        assert_codes_equal(u8(q), oq, "Wq")
        assert_codes_equal(u8(qT), oqT, "WqT")
        assert_scales_equal(s.cpu().numpy(), os_, "sW")
    else:
        assert stalled(lambda: ops.quantize_act_1x128(xg, rows=True, tokens=True)) == ETIMEOUT
        q, s, qT, sT = ops.quantize_act_1x128(xg, rows=True, tokens=True)
        assert ops.sync_status() == 0
        oq, os_ = quant.quantize_act_1x128(np32(x))
        oqT, osT = quant.quantize_act_tokens_1x128(np32(x))
        assert_codes_equal(u8(q), oq, "q")
        assert_scales_equal(s.cpu().numpy(), os_, "s")
        assert_codes_equal(u8(qT), oqT, "qT")
        assert_scales_equal(sT.cpu().numpy(), osT, "sT")


@pytest.mark.parametrize("kind", [0, 1, 2], ids=["pair-tiles", "single-cta-tiles", "pair-tiles-wgrad"])
@pytest.mark.parametrize("layout", ["fprop", "wgrad"])
def test_gemm_timeout_then_within_tolerance(layout, kind):
    M, N, K = 512, 512, 768
    X, W = np32(operands(M, K, 2)), np32(operands(N, K, 3)) * np.float32(0.02)
    if layout == "fprop":
        Aq, sa = quant.quantize_act_1x128(X)
        Bq, _, sb = quant.quantize_w_128x128(W)
        lay = ops.FPROP
        want = ogemm.fprop(Aq, sa, Bq, sb)[1]
    else:
        # dW [N, K] = dY^T X with M tokens; here dY = W-shaped [M, N] values
        dY = np32(operands(M, N, 4)) * np.float32(1e-3)
        Aq, sa = quant.quantize_act_tokens_1x128(dY)
        Bq, sb = quant.quantize_act_tokens_1x128(X)
        lay = ops.WGRAD
        want = ogemm.wgrad(Aq, sa, Bq, sb)[1]
    args = [to_gpu(a) for a in (Aq, sa, Bq, sb)]
    try:
        ops.set_gemm_kernel(kind)
        assert stalled(lambda: ops.fp8_block_gemm(lay, *args)) == ETIMEOUT
        C = ops.fp8_block_gemm(lay, *args)
        assert ops.sync_status() == 0
    finally:
        ops.set_gemm_kernel(0)
    assert rel_fro(np32(C), want) <= REL_FRO_TOL


def test_weight_batch_timeout_then_exact():
    ws = [operands(256, 384, 5), operands(128, 256, 6)]
    wg = [w.to("cuda") for w in ws]
    assert stalled(lambda: ops.quantize_w_batch(wg)) == ETIMEOUT
    got = ops.quantize_w_batch(wg)
    assert ops.sync_status() == 0
    for w, (q, qT, s) in zip(ws, got):
        oq, oqT, os_ = quant.quantize_w_128x128(np32(w))
        assert_codes_equal(u8(q), oq, "Wq")
        assert_codes_equal(u8(qT), oqT, "WqT")
        assert_scales_equal(s.cpu().numpy(), os_, "sW")


def test_stall_hook_affects_one_launch_only():
    x = operands(128, 128, 5).to("cuda")
    assert stalled(lambda: (ops.quantize_act_1x128(x), ops.quantize_act_1x128(x))) == ETIMEOUT
    ops.quantize_act_1x128(x)
    assert ops.sync_status() == 0
