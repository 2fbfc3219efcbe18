"""The GEMM entry point that allocates nothing (bfp8_fp8_block_gemm_noalloc).

Some callers cannot allocate device memory for a workspace: code running in
a CUDA host callback (which may not call the CUDA API), an allocator that
would recurse into itself, or a latency-bound loop that must not let
cudaMalloc synchronise the device.  They call this variant, whose split-K
scratch is a static array inside the library.  Its results must equal those
of the ordinary entry point that takes a caller-allocated workspace, call
after call (the shared array keeps the previous call's contents).

This file sorts last so that a run stopping at its first failure has run
every other test before it.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import REL_FRO_TOL, dev, np32, rel_fro
from blockwise_fp8_linear_quantise_b300 import _lib, ops, workloads

pytestmark = pytest.mark.gpu

EWORKSPACE = 6


def operands(M, N, K, layout, seed):
    """Quantised GEMM operands made by the library's own quantisers."""
    rng = np.random.default_rng(seed)
    a = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32)).to(dev())
    b = workloads.to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(dev())
    A, sa, _, _ = ops.quantize_act_1x128(a, rows=True, tokens=False)
    if layout == ops.WGRAD:
        # one scale per row of B and 128-slice of the reduction: [K/128, N],
        # which is what the 1x128 quantiser returns for b [N, K]
        B, sb = ops.quantize_act_1x128(b, rows=True, tokens=False)[:2]
        return A, sa, B, sb
    Bq, BqT, sW = ops.quantize_w_128x128(b)
    if layout == ops.FPROP:
        return A, sa, Bq, sW
    # DGRAD: B [N, K] holds the transposed weight of a [K, N] layer, so its
    # block scales are indexed [K/128, N/128]
    Bw, BwT, sWt = ops.quantize_w_128x128(b.t().contiguous())
    return A, sa, BwT, sWt


def noalloc(layout, A, sa, B, sb, C, Cq=None, sCq=None):
    lib = _lib.load()
    M, K = A.shape
    N = B.shape[0]
    p = lambda t: None if t is None else t.data_ptr()
    return lib.bfp8_fp8_block_gemm_noalloc(layout, p(A), p(sa), p(B), p(sb), M, N, K, p(C), p(Cq), p(sCq),
                                           torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("layout", [ops.FPROP, ops.DGRAD, ops.WGRAD])
@pytest.mark.parametrize("splits", [0, 3])
def test_noalloc_matches_workspace_gemm_on_consecutive_calls(layout, splits):
    M, N, K = 512, 768, 1280
    A, sa, B, sb = operands(M, N, K, layout, seed=17 + layout)
    try:
        ops.set_gemm_splits(splits)
        if splits:
            assert ops.gemm_workspace_bytes(layout, M, N, K) > 0  # the static scratch is really used
        want = ops.fp8_block_gemm(layout, A, sa, B, sb)
        assert ops.sync_status() == 0
        for _ in range(2):
            C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev())
            assert noalloc(layout, A, sa, B, sb, C) == 0
            assert ops.sync_status() == 0
            assert rel_fro(np32(C), np32(want)) <= REL_FRO_TOL
    finally:
        ops.set_gemm_splits(0)


def test_noalloc_fused_epilogue_matches_on_consecutive_calls():
    M, N, K = 384, 512, 1024
    A, sa, B, sb = operands(M, N, K, ops.FPROP, seed=5)
    try:
        ops.set_gemm_splits(2)
        want, wq, ws = ops.fp8_block_gemm(ops.FPROP, A, sa, B, sb, fused_quant=True)
        for _ in range(2):
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
            Cq = torch.empty((M, N), dtype=torch.uint8, device=dev())
            sCq = torch.empty((N // 128, M), dtype=torch.float32, device=dev())
            assert noalloc(ops.FPROP, A, sa, B, sb, C, Cq, sCq) == 0
            assert ops.sync_status() == 0
            assert rel_fro(np32(C), np32(want)) <= REL_FRO_TOL
            # codes are those of the library's quantiser applied to this call's own output
            q, s, _, _ = ops.quantize_act_1x128(C, rows=True, tokens=False)
            assert torch.equal(Cq, q) and torch.equal(sCq.view(torch.int32), s.view(torch.int32))
    finally:
        ops.set_gemm_splits(0)


def test_noalloc_rejects_partials_beyond_its_scratch():
    lib = _lib.load()
    M, N, K = 2048, 2048, 2048
    try:
        ops.set_gemm_splits(4)  # 4 x 2048 x 2048 x 4 bytes = 64 MiB of partials
        need = ops.gemm_workspace_bytes(ops.FPROP, M, N, K)
        assert need > (32 << 20)
        fake = 1 << 20  # 16-byte aligned, never dereferenced: rejected before any launch
        before = ops.launch_count()
        st = lib.bfp8_fp8_block_gemm_noalloc(ops.FPROP, fake, fake, fake, fake, M, N, K, fake, None, None,
                                             torch.cuda.current_stream().cuda_stream)
        assert st == EWORKSPACE
        assert ops.launch_count() == before
    finally:
        ops.set_gemm_splits(0)
