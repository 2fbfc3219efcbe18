"""Blockwise-FP8 Transformer linear layer for NVIDIA B300 (sm_103a).

E4M3 quantisation of activations in 1x128 groups and of weights in 128x128
blocks, each with an fp32 scale, and the block-scaled GEMM with fp32
promotion for fprop, dgrad and wgrad -- the linear-layer numerics of
"Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090",
section 3.2.  All compute runs in the hand-written CUDA kernels of
``libbfp8.so`` behind the C ABI declared in ``include/bfp8.h``; the Python
layer (``ops``) only marshals torch tensors to that ABI.  There is no CPU
fallback: the ops raise if the library is missing or the device is not an
sm_103 GPU.

Submodules are loaded on first use so that ``workloads`` (seeded input
generation) imports without the CUDA library.
"""

import importlib

__all__ = ["ops", "workloads", "build"]

_OPS = ("quantize_act_1x128", "quantize_w_128x128", "fp8_block_gemm", "linear_fwd", "linear_bwd",
        "gemm_workspace_bytes", "linear_fwd_workspace_bytes", "linear_bwd_workspace_bytes",
        "sync_status", "set_wait_limit_ns", "set_gemm_splits", "set_gemm_kernel", "launch_count", "FPROP", "DGRAD", "WGRAD")


def __getattr__(name):
    if name in ("ops", "workloads", "build", "_lib"):
        return importlib.import_module(f"{__name__}.{name}")
    if name in _OPS:
        return getattr(importlib.import_module(f"{__name__}.ops"), name)
    raise AttributeError(name)
