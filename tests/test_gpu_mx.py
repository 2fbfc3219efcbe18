"""The MXFP8 1x32 recipe on the GPU against its oracle (oracle/mx.py).

Quantiser codes and power-of-two scales bit-exact, in both groupings (32
values along a row; 32 rows per column, stored transposed), including
subnormal-scale groups that reach the E8M0 clamp at 2^-127 and every bf16 bit
pattern; the GEMM that promotes every 32-deep slice within relative Frobenius
error 1e-3 of the oracle's bf16 output, for the FPROP, DGRAD and WGRAD uses of
a linear layer, on small shapes in full and on a full-size layer sampled from
every 128-block.
"""

import numpy as np
import pytest
import torch

from gpu_helpers import (REL_FRO_TOL, assert_codes_equal, assert_scales_equal, bf16_input, dev, np32, rel_fro,
                         sample_index, to_gpu, u8)
from oracle import mx
from blockwise_fp8_linear_quantise_b300 import ops, workloads

pytestmark = pytest.mark.gpu


def check_mx(x_bf16):
    x = x_bf16.to(dev())
    q, s, qT, sT = ops.quantize_mx_1x32(x, rows=True, tokens=True)
    assert ops.sync_status() == 0
    xn = np32(x_bf16)
    oq, os_ = mx.quantize_mx_1x32(xn)
    oqT, osT = mx.quantize_mx_tokens_1x32(xn)
    assert_codes_equal(u8(q), oq, "q")
    assert_scales_equal(s.cpu().numpy(), os_, "s")
    assert_codes_equal(u8(qT), oqT, "qT")
    assert_scales_equal(sT.cpu().numpy(), osT, "sT")
    q2, s2, _, _ = ops.quantize_mx_1x32(x, rows=True, tokens=False)
    _, _, qT2, sT2 = ops.quantize_mx_1x32(x, rows=False, tokens=True)
    assert torch.equal(q2, q) and torch.equal(s2, s) and torch.equal(qT2, qT) and torch.equal(sT2, sT)
    return q, s, qT, sT


@pytest.mark.parametrize("M,K", [(128, 128), (384, 640), (1152, 256)])
def test_mx_quantiser_multi_tile(M, K):
    rng = np.random.default_rng(M + K)
    x = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32) * np.exp2(rng.integers(-20, 20, (M, 1))))
    check_mx(x)


def test_mx_quantiser_edge_values():
    M, K = 256, 384
    x = np.zeros((M, K), np.float32)
    x[1, :] = -0.0
    x[2, 5] = 1e-38                  # amax / 448 below 2^-127: the scale clamps to 2^-127
    x[2, 40] = -3e-39
    x[3, :] = 3.0e38
    x[3, 7] = -1.0
    x[4, 64:96] = np.float32(0.5)
    x[5:, :] = np.random.default_rng(0).standard_normal((M - 5, K)).astype(np.float32)
    x[200:232, 128:160] = 0.0        # a zero token group
    x[100, 0:32] = np.float32(2.0 ** -130)   # bf16 subnormal amax
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    fin = bits[np.isfinite(bits)]
    x[128:256, 256:384].flat[: min(fin.size, 128 * 128)] = fin[: 128 * 128]
    check_mx(workloads.to_bf16(x))


def test_mx_quantiser_every_bf16_bit_pattern():
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    fin = bits[np.isfinite(bits)]
    x = np.zeros((512, 256), np.float32)
    x.flat[: fin.size] = fin
    check_mx(workloads.to_bf16(x))


@pytest.mark.parametrize("name,tag", [("mlp_gateup", "x"), ("mlp_down", "x"), ("attn_proj", "dy_qkv")])
def test_mx_quantiser_full_size(name, tag):
    check_mx(bf16_input(name, tag))


def layer(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = workloads.to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = workloads.to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    dY = workloads.to_bf16((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    return X, W, dY


def mx_layer_gemms(X, W, dY):
    """The three GEMMs of a linear layer in the 1x32 recipe: (name, A, sa, B, sb)."""
    Xq, sX, XqT, sXT = ops.quantize_mx_1x32(X.to(dev()), rows=True, tokens=True)
    Wq, sW, WqT, sWT = ops.quantize_mx_1x32(W.to(dev()), rows=True, tokens=True)
    dYq, sdY, dYqT, sdYT = ops.quantize_mx_1x32(dY.to(dev()), rows=True, tokens=True)
    return [("fprop", Xq, sX, Wq, sW), ("dgrad", dYq, sdY, WqT, sWT), ("wgrad", dYqT, sdYT, XqT, sXT)]


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (384, 640, 512), (1024, 768, 1280), (128, 128, 128)])
def test_mx_gemm_small_shapes_all_layouts(M, N, K):
    X, W, dY = layer(M, N, K, M + N + K)
    for name, A, sa, B, sb in mx_layer_gemms(X, W, dY):
        C = ops.mx_gemm(A, sa, B, sb)
        assert ops.sync_status() == 0
        want = mx.mx_gemm(u8(A), sa.cpu().numpy(), u8(B), sb.cpu().numpy())[1]
        err = rel_fro(np32(C), want)
        assert err <= REL_FRO_TOL, (name, err)


def test_mx_layer_matches_oracle_linear_layer():
    """The oracle's own linear functions (quantisation and GEMMs together)."""
    X, W, dY = layer(256, 384, 512, 3)
    g = {name: np32(ops.mx_gemm(A, sa, B, sb)) for name, A, sa, B, sb in mx_layer_gemms(X, W, dY)}
    oY = mx.mx_linear_fwd(np32(X), np32(W))
    odX, odW = mx.mx_linear_bwd(np32(dY), np32(X), np32(W))
    assert rel_fro(g["fprop"], oY) <= REL_FRO_TOL
    assert rel_fro(g["dgrad"], odX) <= REL_FRO_TOL
    assert rel_fro(g["wgrad"], odW) <= REL_FRO_TOL


def test_mx_gemm_full_size_sampled():
    """mlp_gateup fprop (8192 x 12288 x 2048), sampled from every 128-block."""
    X = bf16_input("mlp_gateup", "x")
    W = bf16_input("mlp_gateup", "w")
    Xq, sX, _, _ = ops.quantize_mx_1x32(X.to(dev()))
    Wq, sW, _, _ = ops.quantize_mx_1x32(W.to(dev()))
    C = ops.mx_gemm(Xq, sX, Wq, sW)
    assert ops.sync_status() == 0
    rng = np.random.default_rng(1)
    rows = sample_index(C.shape[0], 200, rng)
    cols = sample_index(C.shape[1], 300, rng)
    want = mx.mx_gemm(u8(Xq), sX.cpu().numpy(), u8(Wq), sW.cpu().numpy(), rows=rows, cols=cols)[1]
    got = np32(C)[np.ix_(rows, cols)]
    assert rel_fro(got, want) <= REL_FRO_TOL
