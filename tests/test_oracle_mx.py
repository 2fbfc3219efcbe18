"""Pins for the oracle's MXFP8 1x32 recipe.

Checked against: the hand-worked power-of-two group (golden fixture) placed in
one 32-group; powers of two within the E8M0 range for every bf16 amax; the
nesting of power-of-two E4M3 grids (a 32-group's scale never exceeds its
128-group's, so every element rounds at least as close as under 1x128
power-of-two scaling, exactly, element by element); group locality at 32;
the GEMM against an exact integer matmul where fp32 is exact and against a
dequantised fp64 matmul elsewhere; and the recipe's purpose, shown where it
applies: a value far beyond E4M3's range relative to its neighbours coarsens
only its own 32-group.  (On the workloads' x30-x50 outliers the two recipes
lose about the same: E4M3 spans about 17 binades, so such a group's other
values stay in the normal range either way.)
"""

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats, mx, quant
from blockwise_fp8_linear_quantise_b300 import workloads

T_DEC = formats.e4m3_decode(np.arange(256, dtype=np.uint8))


def test_worked_group_in_a_32_group():
    rows = read_golden("pow2_quant_worked_example.txt")
    want_s = float(rows[0][1])
    x = np.zeros((1, 128), np.float32)
    want = np.zeros(128, np.uint8)
    for pos, xv, _xs, code in rows[1:]:
        x[0, int(pos)] = np.float32(float(xv))
        want[int(pos)] = int(code, 16)
    q, s = mx.quantize_mx_1x32(np.tile(x, (4, 1)))
    assert s.shape == (4, 4)
    assert np.all(s[0] == want_s)  # the fixture's values all sit in the first 32-group
    assert np.all(s[1:] == 1.0)   # all-zero groups
    assert np.array_equal(q[0], want) and np.array_equal(q[3], want)


def test_scales_are_powers_of_two_in_the_e8m0_range():
    amax = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    s = mx.mx_scale(amax).astype(np.float64)
    f, _ = np.frexp(s)
    assert np.all(f == 0.5)
    assert np.all((s >= 2.0 ** -127) & (s <= 2.0 ** 127))
    a = amax.astype(np.float64)
    covered = 448.0 * s >= a
    assert np.all(covered | (s == 2.0 ** -127))          # only the clamp can leave amax uncovered
    assert np.all((448.0 * s / 2 < a) | (s == 2.0 ** -127))  # and otherwise it is the smallest such power


@pytest.mark.parametrize("name,tag", [("tiny", "x"), ("mlp_down", "x"), ("attn_proj", "x")])
def test_finer_groups_never_round_worse(name, tag):
    x = workloads.tensor(workloads.make(name), tag).float().numpy()[:256, :512]
    q32, s32 = mx.quantize_mx_1x32(x)
    q128, s128 = quant.quantize_act_1x128(x, scale_mode="pow2")
    S32 = np.repeat(s32.T, 32, axis=1).astype(np.float64)
    S128 = np.repeat(s128.T, 128, axis=1).astype(np.float64)
    assert np.all(S32 <= S128)
    e32 = np.abs(x.astype(np.float64) - T_DEC[q32] * S32)
    e128 = np.abs(x.astype(np.float64) - T_DEC[q128] * S128)
    assert np.all(e32 <= e128)
    assert np.count_nonzero(e32 < e128) > 0


def test_group_locality():
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((128, 128)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    q0, s0 = mx.quantize_mx_1x32(x)
    y = x.copy()
    y[5, 70] = np.float32(1000.0)  # group 2 of row 5
    q1, s1 = mx.quantize_mx_1x32(y)
    changed = np.argwhere(q0 != q1)
    assert changed.size and np.all(changed[:, 0] == 5) and np.all(changed[:, 1] // 32 == 2)
    assert np.argwhere(s0 != s1).tolist() == [[2, 5]]


def test_gemm_is_exact_where_fp32_is():
    rng = np.random.default_rng(6)
    # codes of 0, +-1, +-2 (0x00, 0x38, 0xB8, 0x40, 0xC0) with unit scales: every
    # partial sum is a small integer, so the promotion is exact
    codes = np.array([0x00, 0x38, 0xB8, 0x40, 0xC0], np.uint8)
    A = codes[rng.integers(0, 5, (64, 256))]
    B = codes[rng.integers(0, 5, (96, 256))]
    ones_a = np.ones((8, 64), np.float32)
    ones_b = np.ones((8, 96), np.float32)
    acc, _ = mx.mx_gemm(A, ones_a, B, ones_b)
    want = T_DEC[A].astype(np.int64) @ T_DEC[B].astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), want)


def test_gemm_against_dequantised_fp64():
    rng = np.random.default_rng(8)
    X = torch.from_numpy(rng.standard_normal((128, 512)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    W = torch.from_numpy((rng.standard_normal((192, 512)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    W = W.float().numpy()
    Xq, sX = mx.quantize_mx_1x32(X)
    Wq, sW = mx.quantize_mx_1x32(W)
    acc, _ = mx.mx_gemm(Xq, sX, Wq, sW)
    Xd = T_DEC[Xq] * np.repeat(sX.T, 32, axis=1).astype(np.float64)
    Wd = T_DEC[Wq] * np.repeat(sW.T, 32, axis=1).astype(np.float64)
    ref = Xd @ Wd.T
    # 16 fp32 promotions of exact slice sums: well under 1e-6 relative
    assert np.linalg.norm(acc - ref) <= 1e-6 * np.linalg.norm(ref)
    # the linear helpers use the same pieces
    Y = mx.mx_linear_fwd(X, W)
    assert np.array_equal(Y, formats.bf16_round(acc))


def test_backward_layouts_quantise_along_each_reduction():
    rng = np.random.default_rng(9)
    X = torch.from_numpy(rng.standard_normal((128, 256)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    W = torch.from_numpy((rng.standard_normal((192, 256)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    W = W.float().numpy()
    dY = torch.from_numpy((rng.standard_normal((128, 192)) * 1e-3).astype(np.float32)).to(torch.bfloat16)
    dY = dY.float().numpy()
    dX, dW = mx.mx_linear_bwd(dY, X, W)
    ref_dX = dY.astype(np.float64) @ W.astype(np.float64)
    ref_dW = dY.astype(np.float64).T @ X.astype(np.float64)
    # FP8 operands: a few percent of quantisation error, far from a wrong layout
    assert np.linalg.norm(dX - ref_dX) <= 0.06 * np.linalg.norm(ref_dX)
    assert np.linalg.norm(dW - ref_dW) <= 0.06 * np.linalg.norm(ref_dW)


def test_an_extreme_value_only_coarsens_its_own_32_group():
    """The pages' argument for fine groups: an extreme value should only
    coarsen its own small block.  With one value 2^16 times the others at the
    start of every 128-group, 1x128 scales push the rest of the group towards
    the E4M3 subnormals, while 1x32 scales keep the other three 32-groups at
    full precision."""
    rng = np.random.default_rng(12)
    x = torch.from_numpy(rng.standard_normal((128, 256)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    x[:, ::128] = np.float32(65536.0)
    others = np.ones(x.shape, bool)
    others[:, 0:32] = others[:, 128:160] = False  # the outliers' own 32-groups
    q32, s32 = mx.quantize_mx_1x32(x)
    d32 = T_DEC[q32] * np.repeat(s32.T, 32, axis=1)
    e32 = np.linalg.norm((x - d32)[others]) / np.linalg.norm(x[others])
    for mode in ("amax448", "pow2"):
        q128, s128 = quant.quantize_act_1x128(x, scale_mode=mode)
        d128 = T_DEC[q128] * np.repeat(s128.T, 128, axis=1)
        e128 = np.linalg.norm((x - d128)[others]) / np.linalg.norm(x[others])
        assert e32 < 0.04 and e128 > 2 * e32, (mode, e32, e128)
