"""The library's calls replay from a CUDA graph.

The library allocates nothing, never synchronises inside a call and launches
only on the caller's stream, so a whole training step of its calls can be
captured once and replayed.  Replays must give the eager results bit for
bit, including after new input data is copied into the captured buffers.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import dev
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def _inputs(seed, M=512, N=640, K=384):
    rng = np.random.default_rng(seed)
    X = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32)).to(dev())
    W = workloads.to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32)).to(dev())
    dY = workloads.to_bf16((rng.standard_normal((M, N)) * 1e-3).astype(np.float32)).to(dev())
    return X, W, dY


def _eager(X, W, dY, scale_mode):
    Y, saved = ops.linear_fwd(X, W, scale_mode=scale_mode)
    dX, dW = ops.linear_bwd(dY, saved, scale_mode=scale_mode)
    q, s, qT, sT = ops.quantize_act_1x128(Y, rows=True, tokens=True, scale_mode=scale_mode)
    assert ops.sync_status() == 0
    return dict(Y=Y, dX=dX, dW=dW, q=q, s=s, qT=qT, sT=sT, **{"saved_" + k: v for k, v in saved.items()})


@pytest.mark.parametrize("scale_mode", ["amax448", "pow2", "mul_recip"])
def test_linear_step_replays_from_a_cuda_graph(scale_mode):
    M, N, K = 512, 640, 384
    X, W, dY = _inputs(1)
    # static buffers the graph reads and writes
    X_s, W_s, dY_s = X.clone(), W.clone(), dY.clone()
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
    saved = dict(WqT=torch.empty((K, N), dtype=torch.uint8, device=dev()),
                 sW=torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev()),
                 XqT=torch.empty((K, M), dtype=torch.uint8, device=dev()),
                 sXT=torch.empty((M // 128, K), dtype=torch.float32, device=dev()))
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev())
    dW = torch.empty((N, K), dtype=torch.bfloat16, device=dev())
    q = torch.empty((M, N), dtype=torch.uint8, device=dev())
    s = torch.empty((N // 128, M), dtype=torch.float32, device=dev())
    qT = torch.empty((N, M), dtype=torch.uint8, device=dev())
    sT = torch.empty((M // 128, N), dtype=torch.float32, device=dev())
    ws_f = torch.empty(ops.linear_fwd_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev())
    ws_b = torch.empty(ops.linear_bwd_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev())

    def step():
        ops.linear_fwd(X_s, W_s, Y=Y, saved=saved, workspace=ws_f, scale_mode=scale_mode)
        ops.linear_bwd(dY_s, saved, dX=dX, dW=dW, workspace=ws_b, scale_mode=scale_mode)
        ops.quantize_act_1x128(Y, rows=True, tokens=True, q=q, s=s, qT=qT, sT=sT, scale_mode=scale_mode)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (first-call set-up happens here)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    outs = dict(Y=Y, dX=dX, dW=dW, q=q, s=s, qT=qT, sT=sT, **{"saved_" + k: v for k, v in saved.items()})
    for seed in (1, 1, 2):  # twice on the captured data, then on new data in the same buffers
        Xn, Wn, dYn = _inputs(seed)
        X_s.copy_(Xn), W_s.copy_(Wn), dY_s.copy_(dYn)
        for t in outs.values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert ops.sync_status() == 0
        want = _eager(Xn, Wn, dYn, scale_mode)
        for k, t in outs.items():
            assert torch.equal(t.view(torch.uint8) if t.dtype != torch.uint8 else t,
                               want[k].view(torch.uint8) if want[k].dtype != torch.uint8 else want[k]), (seed, k)
