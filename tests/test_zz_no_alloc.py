"""The GEMM entry point that allocates nothing (bfp8_fp8_block_gemm_noalloc).

Some callers cannot allocate device memory for a workspace and have none to
pass: a process whose device memory is all reserved by another framework's
memory pool, a latency-bound loop where cudaMalloc or cudaFree (which may
synchronise the device) must not run, or code bound to an interface without
a workspace argument.  They call this variant from ordinary host code; its
split-K scratch is a static array inside the library.  Its results must equal
those of the ordinary entry point, which takes a caller-allocated workspace
and runs the same plan, bit for bit, call after call, although the shared
array keeps what the previous call left in it.

This file sorts last so that a run stopping at its first failure has run
every other test before it.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import dev
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


def noalloc_out(layout, ops_, M, N):
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev())
    assert noalloc(layout, *ops_, C) == 0
    assert ops.sync_status() == 0
    return C


@pytest.mark.parametrize("layout", [ops.FPROP, ops.DGRAD, ops.WGRAD])
@pytest.mark.parametrize("splits", [0, 3])
def test_noalloc_equals_workspace_gemm_on_consecutive_calls(layout, splits):
    M, N, K = 512, 768, 1280
    first = operands(M, N, K, layout, seed=17 + layout)
    other = operands(M, N, K, layout, seed=91 + layout)  # different values: different partials in the array
    try:
        ops.set_gemm_splits(splits)
        if splits:
            assert ops.gemm_workspace_bytes(layout, M, N, K) > 0  # the static scratch is really used
        want = ops.fp8_block_gemm(layout, *first)
        want_other = ops.fp8_block_gemm(layout, *other)
        assert ops.sync_status() == 0
        # first operands, other operands, first again: a split that failed to
        # overwrite its slice of the array would leave the other call's
        # partials in the third result
        assert torch.equal(noalloc_out(layout, first, M, N), want)
        assert torch.equal(noalloc_out(layout, other, M, N), want_other)
        assert not torch.equal(want, want_other)
        assert torch.equal(noalloc_out(layout, first, M, N), want)
    finally:
        ops.set_gemm_splits(0)


def test_noalloc_fused_epilogue_equals_on_consecutive_calls():
    M, N, K = 384, 512, 1024
    first = operands(M, N, K, ops.FPROP, seed=5)
    other = operands(M, N, K, ops.FPROP, seed=6)
    try:
        ops.set_gemm_splits(2)
        want = ops.fp8_block_gemm(ops.FPROP, *first, fused_quant=True)
        want_other = ops.fp8_block_gemm(ops.FPROP, *other, fused_quant=True)
        for opnds, (wC, wq, ws) in ((first, want), (other, want_other), (first, want)):
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
            Cq = torch.empty((M, N), dtype=torch.uint8, device=dev())
            sCq = torch.empty((N // 128, M), dtype=torch.float32, device=dev())
            assert noalloc(ops.FPROP, *opnds, C, Cq, sCq) == 0
            assert ops.sync_status() == 0
            assert torch.equal(C, wC)
            assert torch.equal(Cq, wq) and torch.equal(sCq.view(torch.int32), ws.view(torch.int32))
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
