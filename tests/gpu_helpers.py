"""Shared helpers for the GPU parity tests (no method arithmetic here)."""

import numpy as np
import torch

from blockwise_fp8_linear_quantise_b300 import workloads

REL_FRO_TOL = 1e-3  # GEMM bf16 outputs vs the oracle's bf16 outputs


def dev():
    return torch.device("cuda:0")


def np32(t):
    """bf16/float tensor -> float32 numpy (exact for bf16)."""
    return t.detach().float().cpu().numpy()


def u8(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def f32_bits(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def to_gpu(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(dev())


def rel_fro(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    den = np.linalg.norm(want)
    return np.linalg.norm(got - want) / (den if den > 0 else 1.0)


def assert_codes_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
                          f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def assert_scales_equal(got, want, what):
    assert_codes_equal(f32_bits(got), f32_bits(want), what)


def bf16_input(name, tag, layer=None):
    wl = workloads.make(name)
    return workloads.tensor(wl, tag, layer)


def sample_index(n, count, rng, block=128):
    """Indices spread over every 128-block of [0, n), including both ends."""
    nb = n // block
    idx = {0, n - 1}
    for b in range(nb):
        idx.add(b * block + int(rng.integers(0, block)))
    while len(idx) < min(count, n):
        idx.add(int(rng.integers(0, n)))
    return np.array(sorted(idx))
