"""GPU block-scaled GEMM (fprop, dgrad, wgrad) vs the CPU oracle.

The GPU GEMM is fed the oracle's own quantised operands, so these tests see
only the GEMM; bf16 outputs must agree with the oracle's bf16 outputs within
relative Frobenius error 1e-3.  Small shapes are compared in full; the
full-size workloads are compared on outputs sampled from every 128-row and
128-column block, in the launch configuration the benchmark uses.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import (REL_FRO_TOL, assert_codes_equal, assert_scales_equal, bf16_input, dev, np32, rel_fro,
                         sample_index, to_gpu, u8)
from oracle import gemm as ogemm, quant
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def quantised_layer(X, W, dY):
    """Oracle-quantised operands of one layer (numpy)."""
    o = {}
    o["Wq"], o["WqT"], o["sW"] = quant.quantize_w_128x128(X if W is None else W)
    if X is not None:
        o["Xq"], o["sX"] = quant.quantize_act_1x128(X)
        o["XqT"], o["sXT"] = quant.quantize_act_tokens_1x128(X)
    if dY is not None:
        o["dYq"], o["sdY"] = quant.quantize_act_1x128(dY)
        o["dYqT"], o["sdYT"] = quant.quantize_act_tokens_1x128(dY)
    return o


def gpu(o, k):
    return to_gpu(o[k])


def run_layouts(o, layouts, rows=None, cols=None, fused=False):
    """Run the requested GPU GEMMs and compare with the oracle."""
    results = {}
    for lay in layouts:
        if lay == "fprop":
            C = ops.fp8_block_gemm(ops.FPROP, gpu(o, "Xq"), gpu(o, "sX"), gpu(o, "Wq"), gpu(o, "sW"),
                                   fused_quant=fused)
            want = ogemm.fprop(o["Xq"], o["sX"], o["Wq"], o["sW"], rows=rows, cols=cols)[1]
        elif lay == "dgrad":
            C = ops.fp8_block_gemm(ops.DGRAD, gpu(o, "dYq"), gpu(o, "sdY"), gpu(o, "WqT"), gpu(o, "sW"),
                                   fused_quant=fused)
            want = ogemm.dgrad(o["dYq"], o["sdY"], o["WqT"], o["sW"], rows=rows, cols=cols)[1]
        else:
            C = ops.fp8_block_gemm(ops.WGRAD, gpu(o, "dYqT"), gpu(o, "sdYT"), gpu(o, "XqT"), gpu(o, "sXT"),
                                   fused_quant=fused)
            want = ogemm.wgrad(o["dYqT"], o["sdYT"], o["XqT"], o["sXT"], rows=rows, cols=cols)[1]
        assert ops.sync_status() == 0
        Cg = C[0] if fused else C
        got = np32(Cg)
        if rows is not None:
            got = got[np.ix_(rows, cols)]
        err = rel_fro(got, want)
        assert err <= REL_FRO_TOL, (lay, err)
        results[lay] = (C, want, err)
    return results


def rand_layer(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = workloads.to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    dY = workloads.to_bf16((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    return np32(X), np32(W), np32(dY)


@pytest.fixture(params=[0, 1, 2], ids=["pair-tiles", "single-cta-tiles", "pair-tiles-wgrad"])
def gemm_kind(request):
    """Run a test with the CTA-pair GEMM (where the shape allows), with
    single-CTA tiles only, and with CTA pairs for WGRAD as well."""
    ops.set_gemm_kernel(request.param)
    yield request.param
    ops.set_gemm_kernel(0)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (384, 640, 512), (512, 768, 384), (1024, 1280, 1536),
                                   (128, 128, 128), (2304, 512, 640), (768, 1024, 2048)])
def test_small_shapes_all_layouts(M, N, K, gemm_kind):
    X, W, dY = rand_layer(M, N, K, M + N + K)
    o = quantised_layer(X, W, dY)
    run_layouts(o, ["fprop", "dgrad", "wgrad"])


def test_pair_and_single_tiles_agree():
    """Both tilings accumulate the same slices in the same order, so their
    bf16 outputs agree to rounding of the tensor-core partial sums."""
    X, W, dY = rand_layer(1024, 1536, 2048, 11)
    o = quantised_layer(X, W, dY)
    outs = []
    for kind in (0, 1):
        try:
            ops.set_gemm_kernel(kind)
            outs.append(np32(ops.fp8_block_gemm(ops.FPROP, gpu(o, "Xq"), gpu(o, "sX"), gpu(o, "Wq"), gpu(o, "sW"))))
        finally:
            ops.set_gemm_kernel(0)
    assert ops.sync_status() == 0
    assert rel_fro(outs[0], outs[1]) <= 1e-4


def test_tiny_config():
    wl = workloads.make("tiny")
    X, W = np32(workloads.tensor(wl, "x")), np32(workloads.tensor(wl, "w"))
    o = quantised_layer(X, W, None)
    r = run_layouts(o, ["fprop"])
    C, want, err = r["fprop"]
    # also report how many bf16 outputs differ at all (diagnostic bound)
    diff = np.count_nonzero(np32(C) != want)
    assert diff <= want.size // 20


@pytest.mark.parametrize("splits", [1, 2, 3, 5])
def test_forced_split_k(splits, gemm_kind):
    X, W, dY = rand_layer(640, 512, 768, 99)
    o = quantised_layer(X, W, dY)
    try:
        ops.set_gemm_splits(splits)
        run_layouts(o, ["fprop", "dgrad", "wgrad"])
    finally:
        ops.set_gemm_splits(0)


@pytest.mark.parametrize("splits", [1, 3])
def test_fused_quantised_epilogue(splits, gemm_kind):
    X, W, dY = rand_layer(512, 768, 640, 5)
    o = quantised_layer(X, W, dY)
    try:
        ops.set_gemm_splits(splits)
        r = run_layouts(o, ["fprop", "wgrad"], fused=True)
    finally:
        ops.set_gemm_splits(0)
    for lay, ((C, Cq, sCq), want, _) in r.items():
        # the fused codes are the activation quantiser's codes of the bf16 output
        q, s, _, _ = ops.quantize_act_1x128(C, rows=True, tokens=False)
        assert torch.equal(Cq, q), lay
        assert torch.equal(sCq.view(torch.int32), s.view(torch.int32)), lay
        # ... and the oracle's codes of that same bf16 output, bit for bit
        oq, os_ = quant.quantize_act_1x128(np32(C))
        assert_codes_equal(u8(Cq), oq, lay + " Cq")
        assert_scales_equal(sCq.cpu().numpy(), os_, lay + " sCq")
        # and they decode close to the oracle's output
        deq = (Cq.view(torch.float8_e4m3fn).float() * sCq.t().repeat_interleave(128, dim=1)).cpu().numpy()
        assert rel_fro(deq, want) < 0.05


def test_bad_workspace_is_rejected():
    X, W, dY = rand_layer(256, 256, 1024, 3)
    o = quantised_layer(X, W, dY)
    try:
        ops.set_gemm_splits(4)
        with pytest.raises(ops.BFP8Error):
            ops.fp8_block_gemm(ops.FPROP, gpu(o, "Xq"), gpu(o, "sX"), gpu(o, "Wq"), gpu(o, "sW"),
                               workspace=torch.empty(16, dtype=torch.uint8, device=dev()))
    finally:
        ops.set_gemm_splits(0)


def sampled(M, N, seed):
    rng = np.random.default_rng(seed)
    return sample_index(M, 512, rng), sample_index(N, 512, rng)


def test_full_mlp_gateup_fprop():
    wl = workloads.make("mlp_gateup")
    X, W = np32(workloads.tensor(wl, "x")), np32(workloads.tensor(wl, "w"))
    o = quantised_layer(X, W, None)
    rows, cols = sampled(X.shape[0], W.shape[0], 1)
    run_layouts(o, ["fprop"], rows, cols)


def test_full_mlp_down_fwd_bwd():
    wl = workloads.make("mlp_down")
    X, W, dY = (np32(workloads.tensor(wl, t)) for t in ("x", "w", "dy"))
    o = quantised_layer(X, W, dY)
    M, K = X.shape
    N = W.shape[0]
    r, c = sampled(M, N, 2)
    run_layouts(o, ["fprop"], r, c)
    r, c = sampled(M, K, 3)
    run_layouts(o, ["dgrad"], r, c)
    r, c = sampled(N, K, 4)
    run_layouts(o, ["wgrad"], r, c)


@pytest.mark.parametrize("w_tag,dy_tag", [("w_qkv", "dy_qkv"), ("w_o", "dy_o")])
def test_full_attn_proj(w_tag, dy_tag):
    wl = workloads.make("attn_proj")
    X, W, dY = np32(workloads.tensor(wl, "x")), np32(workloads.tensor(wl, w_tag)), np32(workloads.tensor(wl, dy_tag))
    o = quantised_layer(X, W, dY)
    M, K = X.shape
    N = W.shape[0]
    r, c = sampled(M, N, 5)
    run_layouts(o, ["fprop"], r, c)
    r, c = sampled(M, K, 6)
    run_layouts(o, ["dgrad"], r, c)
    r, c = sampled(N, K, 7)
    run_layouts(o, ["wgrad"], r, c)


def test_full_stack_gate_up_layer():
    wl = workloads.make("stack28")
    X = np32(workloads.tensor(wl, "x_h"))
    W = np32(workloads.tensor(wl, "w_gu", layer=13))
    dY = np32(workloads.tensor(wl, "dy_gu"))
    o = quantised_layer(X, W, dY)
    M, K = X.shape
    N = W.shape[0]
    r, c = sampled(M, N, 8)
    run_layouts(o, ["fprop"], r, c)
    r, c = sampled(M, K, 9)
    run_layouts(o, ["dgrad"], r, c)
    r, c = sampled(N, K, 10)
    run_layouts(o, ["wgrad"], r, c)


# ------------------------------------------------------- fp32 accumulate-into


def _accumulate(o, lay, C):
    if lay == "fprop":
        ops.fp8_block_gemm_accumulate(ops.FPROP, gpu(o, "Xq"), gpu(o, "sX"), gpu(o, "Wq"), gpu(o, "sW"), C)
        return ogemm.fprop(o["Xq"], o["sX"], o["Wq"], o["sW"])[0]
    if lay == "dgrad":
        ops.fp8_block_gemm_accumulate(ops.DGRAD, gpu(o, "dYq"), gpu(o, "sdY"), gpu(o, "WqT"), gpu(o, "sW"), C)
        return ogemm.dgrad(o["dYq"], o["sdY"], o["WqT"], o["sW"])[0]
    ops.fp8_block_gemm_accumulate(ops.WGRAD, gpu(o, "dYqT"), gpu(o, "sdYT"), gpu(o, "XqT"), gpu(o, "sXT"), C)
    return ogemm.wgrad(o["dYqT"], o["sdYT"], o["XqT"], o["sXT"])[0]


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("M,N,K", [(512, 768, 640), (256, 384, 1280)])
def test_accumulate_into_fp32_all_layouts(M, N, K, splits, gemm_kind):
    """C_f32 += product, twice: each increment is the oracle's fp32
    accumulator (before bf16 rounding) within the GEMM tolerance."""
    X, W, dY = rand_layer(M, N, K, M + 3 * N + K)
    o = quantised_layer(X, W, dY)
    rng = np.random.default_rng(11)
    try:
        ops.set_gemm_splits(splits)
        for lay in ("fprop", "dgrad", "wgrad"):
            shape = {"fprop": (M, N), "dgrad": (M, K), "wgrad": (N, K)}[lay]
            C0 = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dev())
            C = C0.clone()
            acc = _accumulate(o, lay, C)
            assert ops.sync_status() == 0
            scale = np.abs(acc).max()
            C0s = C0 * float(scale)  # start values of the accumulator's size
            C = C0s.clone()
            _accumulate(o, lay, C)
            assert ops.sync_status() == 0
            inc1 = (C.double() - C0s.double()).cpu().numpy()
            assert rel_fro(inc1, acc) <= REL_FRO_TOL, (lay, rel_fro(inc1, acc))
            _accumulate(o, lay, C)
            assert ops.sync_status() == 0
            inc2 = (C.double() - C0s.double()).cpu().numpy()
            assert rel_fro(inc2, 2.0 * acc) <= REL_FRO_TOL, lay
            # the plain GEMM's bf16 output rounds the same accumulator
            Cb = run_layouts(o, [lay])[lay][0]
            assert rel_fro(np32(Cb), inc1) <= 1e-2
    finally:
        ops.set_gemm_splits(0)


def test_linear_bwd_main_grad_matches_oracle():
    X, W, dY = rand_layer(384, 512, 640, 21)
    Xg, Wg, dYg = (workloads.to_bf16(a).to(dev()) for a in (X, W, dY))
    _, saved = ops.linear_fwd(Xg, Wg)
    dX_ref, dW_ref = ops.linear_bwd(dYg, saved)
    main0 = np.random.default_rng(5).standard_normal((512, 640)).astype(np.float32) * 1e-3
    main = torch.from_numpy(main0).to(dev())
    dX, main1 = ops.linear_bwd(dYg, saved, dW_main=main)
    assert ops.sync_status() == 0
    assert main1.data_ptr() == main.data_ptr()
    assert torch.equal(dX, dX_ref)
    _, o_saved = ogemm.linear_fwd(X, W)
    _, want = ogemm.linear_bwd(dY, o_saved, main_grad=main0)
    got_inc = (main1.double().cpu().numpy() - main0)
    want_inc = want.astype(np.float64) - main0
    assert rel_fro(got_inc, want_inc) <= REL_FRO_TOL
    assert rel_fro(np32(dW_ref), got_inc) <= 1e-2


def test_accumulate_rejects_a_missing_target():
    from blockwise_fp8_linear_quantise_b300 import _lib
    st = torch.cuda.current_stream().cuda_stream
    fake = 1 << 20
    assert _lib.load().bfp8_fp8_block_gemm_accumulate(ops.FPROP, fake, fake, fake, fake, 256, 256, 256, None,
                                                      None, 0, st) == 1


def test_full_stack_gate_up_wgrad_accumulate():
    """fp32 main-gradient accumulation at the stack's largest WGRAD
    (12288 x 2048 over 16384 tokens), checked on sampled outputs."""
    wl = workloads.make("stack28")
    X = np32(workloads.tensor(wl, "x_h"))
    dY = np32(workloads.tensor(wl, "dy_gu"))
    o = quantised_layer(X, None, dY)
    N, K = dY.shape[1], X.shape[1]
    r, c = sampled(N, K, 12)
    want = ogemm.wgrad(o["dYqT"], o["sdYT"], o["XqT"], o["sXT"], rows=r, cols=c)[0]
    rng = np.random.default_rng(13)
    C0 = torch.from_numpy((rng.standard_normal((N, K)) * float(np.abs(want).max())).astype(np.float32)).to(dev())
    C = C0.clone()
    ops.fp8_block_gemm_accumulate(ops.WGRAD, gpu(o, "dYqT"), gpu(o, "sdYT"), gpu(o, "XqT"), gpu(o, "sXT"), C)
    assert ops.sync_status() == 0
    inc = (C.double() - C0.double()).cpu().numpy()[np.ix_(r, c)]
    assert rel_fro(inc, want) <= REL_FRO_TOL
