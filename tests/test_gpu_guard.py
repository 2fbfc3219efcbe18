"""Guard bands around every GPU output, in place of a memory checker.

Every output a kernel writes (codes, scales, bf16 and fp32 results, the
split-K workspace, the fused calls' scratch) is placed inside a larger buffer
whose 4 KB on either side hold a known byte.  After the call the bands must be
untouched, and the result must equal that of a call on ordinary buffers, on
small shapes and on shapes whose tiles are ragged (dimensions that are not
multiples of 256, so 128-wide tiles and partial CTA-pair coverage occur).
A write past the edge of a tile into a neighbouring allocation shows up here
even where the output itself is right.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import dev
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` with GUARD bytes of PATTERN on each side."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=dev())
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self, what):
        raw = self.raw.cpu()
        lo = torch.nonzero(raw[:GUARD] != PATTERN)
        hi = torch.nonzero(raw[-GUARD:] != PATTERN)
        assert lo.numel() == 0, f"{what}: {lo.numel()} bytes written before the buffer"
        assert hi.numel() == 0, f"{what}: {hi.numel()} bytes written after the buffer"


def guarded(**spec):
    return {k: Guarded(shape, dtype) for k, (shape, dtype) in spec.items()}


def bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return workloads.to_bf16((rng.standard_normal(shape) * scale).astype(np.float32)).to(dev())


def check_all(g):
    assert ops.sync_status() == 0
    for k, v in g.items():
        v.check(k)


@pytest.mark.parametrize("M,K", [(128, 128), (384, 640), (1152, 256)])
def test_quantisers_stay_inside_their_outputs(M, K):
    x = bf16((M, K), M + K)
    g = guarded(q=((M, K), torch.uint8), s=((K // 128, M), torch.float32), qT=((K, M), torch.uint8),
                sT=((M // 128, K), torch.float32))
    ops.quantize_act_1x128(x, rows=True, tokens=True, q=g["q"].t, s=g["s"].t, qT=g["qT"].t, sT=g["sT"].t)
    check_all(g)
    want = ops.quantize_act_1x128(x, rows=True, tokens=True)
    for k, w in zip(("q", "s", "qT", "sT"), want):
        assert torch.equal(g[k].t, w), k
    gw = guarded(Wq=((M, K), torch.uint8), WqT=((K, M), torch.uint8), sW=((M // 128, K // 128), torch.float32))
    ops.quantize_w_128x128(x, q=gw["Wq"].t, qT=gw["WqT"].t, s=gw["sW"].t)
    check_all(gw)
    for k, w in zip(("Wq", "WqT", "sW"), ops.quantize_w_128x128(x)):
        assert torch.equal(gw[k].t, w), k


def test_weight_batch_stays_inside_its_outputs():
    shapes = [(384, 640), (128, 128), (1152, 256)]
    xs = [bf16(sh, sum(sh)) for sh in shapes]
    gs = [guarded(Wq=((M, K), torch.uint8), WqT=((K, M), torch.uint8), sW=((M // 128, K // 128), torch.float32))
          for M, K in shapes]
    ops.quantize_w_batch(xs, outs=[(g["Wq"].t, g["WqT"].t, g["sW"].t) for g in gs])
    for g, x in zip(gs, xs):
        check_all(g)
        for k, w in zip(("Wq", "WqT", "sW"), ops.quantize_w_128x128(x)):
            assert torch.equal(g[k].t, w), k


def test_swiglu_prologue_stays_inside_its_outputs():
    M, F = 384, 256
    gu = bf16((M, 2 * F), 7, 0.5)
    g = guarded(h=((M, F), torch.bfloat16), q=((M, F), torch.uint8), s=((F // 128, M), torch.float32),
                qT=((F, M), torch.uint8), sT=((M // 128, F), torch.float32))
    ops.swiglu_quantize_1x128(gu, h=g["h"].t, q=g["q"].t, s=g["s"].t, qT=g["qT"].t, sT=g["sT"].t)
    check_all(g)
    want = ops.swiglu_quantize_1x128(gu, want_h=True)
    for k, w in zip(("h", "q", "s", "qT", "sT"), want):
        assert torch.equal(g[k].t, w), k


def gemm_operands(layout, M, N, K, seed):
    a = bf16((M, K), seed)
    b = bf16((N, K), seed + 1, 0.02)
    A, sa, _, _ = ops.quantize_act_1x128(a)
    if layout == ops.WGRAD:
        B, sb, _, _ = ops.quantize_act_1x128(b)
    elif layout == ops.FPROP:
        B, _, sb = ops.quantize_w_128x128(b)
    else:
        _, B, sb = ops.quantize_w_128x128(b.t().contiguous())
    return A, sa, B, sb


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("M,N,K", [(384, 640, 512), (512, 256, 1280), (256, 384, 384)])
def test_gemms_stay_inside_their_outputs(M, N, K, splits, kind):
    try:
        ops.set_gemm_kernel(kind)
        ops.set_gemm_splits(splits)
        for layout in (ops.FPROP, ops.DGRAD, ops.WGRAD):
            A, sa, B, sb = gemm_operands(layout, M, N, K, M + N + K + layout)
            need = ops.gemm_workspace_bytes(layout, M, N, K)
            spec = dict(C=((M, N), torch.bfloat16), Cq=((M, N), torch.uint8), sCq=((N // 128, M), torch.float32))
            if need:
                spec["ws"] = ((need,), torch.uint8)
            g = guarded(**spec)
            ws = g["ws"].t if need else None
            ops.fp8_block_gemm(layout, A, sa, B, sb, C=g["C"].t, fused_quant=True, Cq=g["Cq"].t, sCq=g["sCq"].t,
                               workspace=ws)
            check_all(g)
            wC, wq, ws_ = ops.fp8_block_gemm(layout, A, sa, B, sb, fused_quant=True)
            assert torch.equal(g["C"].t, wC) and torch.equal(g["Cq"].t, wq) and torch.equal(g["sCq"].t, ws_)
            # plain bf16 output, and the fp32 accumulate-into target
            gp = guarded(C=((M, N), torch.bfloat16), **({"ws": ((need,), torch.uint8)} if need else {}))
            ops.fp8_block_gemm(layout, A, sa, B, sb, C=gp["C"].t, workspace=gp["ws"].t if need else None)
            check_all(gp)
            assert torch.equal(gp["C"].t, ops.fp8_block_gemm(layout, A, sa, B, sb))
            ga = guarded(acc=((M, N), torch.float32), **({"ws": ((need,), torch.uint8)} if need else {}))
            ga["acc"].t.fill_(0.5)
            ops.fp8_block_gemm_accumulate(layout, A, sa, B, sb, ga["acc"].t, workspace=ga["ws"].t if need else None)
            check_all(ga)
            ref = torch.full((M, N), 0.5, dtype=torch.float32, device=dev())
            ops.fp8_block_gemm_accumulate(layout, A, sa, B, sb, ref)
            assert torch.equal(ga["acc"].t, ref)
    finally:
        ops.set_gemm_kernel(0)
        ops.set_gemm_splits(0)


def test_fused_linear_calls_stay_inside_their_outputs():
    M, N, K = 384, 640, 256
    X, W, dY = bf16((M, K), 1), bf16((N, K), 2, 0.02), bf16((M, N), 3, 1e-3)
    gf = guarded(Y=((M, N), torch.bfloat16), WqT=((K, N), torch.uint8), sW=((N // 128, K // 128), torch.float32),
                 XqT=((K, M), torch.uint8), sXT=((M // 128, K), torch.float32),
                 ws=((ops.linear_fwd_workspace_bytes(M, N, K),), torch.uint8))
    saved = {k: gf[k].t for k in ("WqT", "sW", "XqT", "sXT")}
    ops.linear_fwd(X, W, Y=gf["Y"].t, saved=saved, workspace=gf["ws"].t)
    check_all(gf)
    Y, want_saved = ops.linear_fwd(X, W)
    assert torch.equal(gf["Y"].t, Y)
    for k in saved:
        assert torch.equal(saved[k], want_saved[k]), k
    gb = guarded(dX=((M, K), torch.bfloat16), dW=((N, K), torch.bfloat16),
                 ws=((ops.linear_bwd_workspace_bytes(M, N, K),), torch.uint8))
    ops.linear_bwd(dY, saved, dX=gb["dX"].t, dW=gb["dW"].t, workspace=gb["ws"].t)
    check_all(gb)
    dX, dW = ops.linear_bwd(dY, want_saved)
    assert torch.equal(gb["dX"].t, dX) and torch.equal(gb["dW"].t, dW)
