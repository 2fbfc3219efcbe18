"""Pins for the oracle's block-scaled GEMM (fprop, dgrad, wgrad) and linear.

Checked against: hand-worked products (golden fixture); fp64 brute force in
plain Python loops with torch's float8 decode (independent of the oracle's
tables) on tiny inputs; the closed form for unit scales; full dequantise-then-
multiply references for every layout on non-square shapes, so a transposed
operand or a wrong scale index fails; and a sanity bound against the
unquantised product.
"""

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import gemm, quant
from blockwise_fp8_linear_quantise_b300 import workloads

T_DEC = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def parse_runs(spec):
    out = []
    for part in spec.split(","):
        code, count = part[:4], part[5:]  # "0xHHxCOUNT"
        out += [int(code, 16)] * int(count)
    return out


def test_worked_examples():
    for row in read_golden("gemm_worked_example.txt"):
        name, a0, a1, b0, b1 = row[:5]
        sa0, sa1, sb0, sb1, expect = map(float, row[5:])
        a = np.array([parse_runs(a0) + parse_runs(a1)], np.uint8)
        b = np.array([parse_runs(b0) + parse_runs(b1)], np.uint8)
        sa = np.array([[sa0], [sa1]], np.float32)
        sb = np.array([[sb0], [sb1]], np.float32)
        acc, out = gemm.block_scaled_gemm(a, b, lambda kb: sa[kb], lambda kb: sb[kb])
        assert acc[0, 0] == np.float32(expect), name
        assert out[0, 0] == np.float32(expect), name


def _random_operands(rng, M, N, K):
    a = rng.integers(0, 256, (M, K)).astype(np.uint8)
    b = rng.integers(0, 256, (N, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    b[(b & 0x7F) == 0x7F] = 0xC0
    return a, b


def test_brute_force_python_loops_tiny():
    rng = np.random.default_rng(11)
    M, N, K = 4, 3, 384
    a, b = _random_operands(rng, M, N, K)
    sa = rng.uniform(1e-3, 2.0, (K // 128, M)).astype(np.float32)
    sb = rng.uniform(1e-3, 2.0, (K // 128, N)).astype(np.float32)
    acc, out = gemm.block_scaled_gemm(a, b, lambda kb: sa[kb], lambda kb: sb[kb])
    for i in range(M):
        for j in range(N):
            exact = 0.0
            mag = 0.0
            for k in range(K):
                t = float(T_DEC[a[i, k]]) * float(sa[k // 128, i]) * float(T_DEC[b[j, k]]) * float(sb[k // 128, j])
                exact += t
                mag += abs(t)
            # per slice: f32(P), f32(scale), product and add each round once
            bound = 2.0 ** -23 * mag * (K // 128 * 3 + 1)
            assert abs(float(acc[i, j]) - exact) <= bound, (i, j)


def test_unit_scales_reduce_to_plain_matmul():
    rng = np.random.default_rng(5)
    a, b = _random_operands(rng, 64, 48, 128)
    one = np.ones(64, np.float32), np.ones(48, np.float32)
    acc, _ = gemm.block_scaled_gemm(a, b, lambda kb: one[0], lambda kb: one[1])
    ref = (torch.from_numpy(T_DEC[a]) @ torch.from_numpy(T_DEC[b]).T).to(torch.float32).numpy()
    assert np.array_equal(acc, ref)  # one slice: exactly f32(P)
    # two slices: f32(f32(P0) + f32(P1))
    a2, b2 = _random_operands(rng, 64, 48, 256)
    acc2, _ = gemm.block_scaled_gemm(a2, b2, lambda kb: one[0], lambda kb: one[1])
    p0 = (torch.from_numpy(T_DEC[a2[:, :128]]) @ torch.from_numpy(T_DEC[b2[:, :128]]).T).to(torch.float32)
    p1 = (torch.from_numpy(T_DEC[a2[:, 128:]]) @ torch.from_numpy(T_DEC[b2[:, 128:]]).T).to(torch.float32)
    assert np.array_equal(acc2, (p0 + p1).numpy())


def _deq_rows(q, s):
    """Dequantise [R, C] codes with group-major scales s [C/128, R]."""
    return T_DEC[q] * np.repeat(s.T.astype(np.float64), 128, axis=1)


def _bound_check(acc, exact, mag, nslices):
    assert np.all(np.abs(acc.astype(np.float64) - exact) <= 2.0 ** -23 * mag * (3 * nslices + 1) + 1e-30)


def test_layouts_against_dequantised_matmul():
    rng = np.random.default_rng(21)
    M, N, K = 384, 256, 640  # tokens, out features, in features (all distinct)
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    dY = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    X, W, dY = [torch.from_numpy(t).to(torch.bfloat16).float().numpy() for t in (X, W, dY)]

    Wq, WqT, sW = quant.quantize_w_128x128(W)
    Xq, sX = quant.quantize_act_1x128(X)
    XqT, sXT = quant.quantize_act_tokens_1x128(X)
    dYq, sdY = quant.quantize_act_1x128(dY)
    dYqT, sdYT = quant.quantize_act_tokens_1x128(dY)

    Wd = T_DEC[Wq] * np.repeat(np.repeat(sW.astype(np.float64), 128, 0), 128, 1)   # [N, K]
    Xd = _deq_rows(Xq, sX)            # [M, K]
    XdT = _deq_rows(XqT, sXT)         # [K, M]
    dYd = _deq_rows(dYq, sdY)         # [M, N]
    dYdT = _deq_rows(dYqT, sdYT)      # [N, M]

    acc, Y = gemm.fprop(Xq, sX, Wq, sW)
    assert acc.shape == (M, N)
    _bound_check(acc, Xd @ Wd.T, np.abs(Xd) @ np.abs(Wd).T, K // 128)

    acc, dX = gemm.dgrad(dYq, sdY, WqT, sW)
    assert acc.shape == (M, K)
    _bound_check(acc, dYd @ Wd, np.abs(dYd) @ np.abs(Wd), N // 128)

    acc, dW = gemm.wgrad(dYqT, sdYT, XqT, sXT)
    assert acc.shape == (N, K)
    _bound_check(acc, dYdT @ XdT.T, np.abs(dYdT) @ np.abs(XdT).T, M // 128)

    # composed linear equals the pieces
    Y2, saved = gemm.linear_fwd(X, W)
    dX2, dW2 = gemm.linear_bwd(dY, saved)
    assert np.array_equal(Y2, Y) and np.array_equal(dX2, dX) and np.array_equal(dW2, dW)

    # subset evaluation returns the same values
    rows, cols = np.array([5, 300]), np.array([0, 129, 255])
    acc_s, _ = gemm.fprop(Xq, sX, Wq, sW, rows=rows, cols=cols)
    acc_f, _ = gemm.fprop(Xq, sX, Wq, sW)
    assert np.array_equal(acc_s, acc_f[np.ix_(rows, cols)])


def test_bf16_output_is_rne_of_acc():
    rng = np.random.default_rng(2)
    a, b = _random_operands(rng, 32, 32, 256)
    sa = rng.uniform(0.1, 1, (2, 32)).astype(np.float32)
    acc, out = gemm.block_scaled_gemm(a, b, lambda kb: sa[kb], lambda kb: sa[kb])
    ref = torch.from_numpy(acc).to(torch.bfloat16).float().numpy()
    assert np.array_equal(out, ref)


def test_quantised_product_close_to_unquantised():
    wl = workloads.make("tiny")
    X = workloads.tensor(wl, "x").float().numpy()
    W = workloads.tensor(wl, "w").float().numpy()
    Y, _ = gemm.linear_fwd(X, W)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    rel = np.linalg.norm(Y - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 0.08


# ------------------------------------------------------- fp32 accumulate-into


def test_accumulate_into_hand_worked_sums():
    """One IEEE fp32 addition per element, checked on sums worked by hand:
    exact ones, a tie that rounds to even and one that rounds up."""
    main = np.array([1.0, -2.5, 1.0, 1.0, 3.0e38, 0.0], np.float32)
    acc = np.array([2.0, 0.75, 2.0 ** -24, 3 * 2.0 ** -24, 3.0e38, -0.0], np.float32)
    want = np.array([3.0, -1.75, 1.0, 1.0 + 2.0 ** -22, np.inf, 0.0], np.float32)
    # 1 + 2^-24: exactly halfway between 1 and 1 + 2^-23, ties to even -> 1
    # 1 + 3*2^-24: halfway between 1 + 2^-23 and 1 + 2^-22, ties to even -> 1 + 2^-22
    with np.errstate(over="ignore"):
        got = gemm.accumulate_into(main, acc)
    assert np.array_equal(got, want) and got.dtype == np.float32
    assert np.signbit(got[5]) == False  # +0 + -0 = +0


def test_linear_bwd_main_grad_adds_the_wgrad_accumulator():
    wl = workloads.make("tiny")
    x = workloads.tensor(wl, "x").float().numpy()
    w = workloads.tensor(wl, "w").float().numpy()
    dy = (np.random.default_rng(3).standard_normal((256, 256)) * 1e-3).astype(np.float32)
    dy = torch.from_numpy(dy).to(torch.bfloat16).float().numpy()
    _, saved = gemm.linear_fwd(x, w)
    dX, dW = gemm.linear_bwd(dy, saved)
    main0 = np.random.default_rng(4).standard_normal((256, 256)).astype(np.float32)
    dX2, main1 = gemm.linear_bwd(dy, saved, main_grad=main0)
    assert np.array_equal(dX, dX2)
    # the increment is the fp32 accumulator, whose bf16 rounding is dW
    dYqT, sdYT = quant.quantize_act_tokens_1x128(dy)
    acc, _ = gemm.wgrad(dYqT, sdYT, saved["XqT"], saved["sXT"])
    assert np.array_equal(main1, (main0.astype(np.float64) + acc).astype(np.float32))
    assert np.array_equal(torch.from_numpy(acc).to(torch.bfloat16).float().numpy(), dW)
    # zero main gradient: accumulate-into returns the accumulator itself
    _, main_z = gemm.linear_bwd(dy, saved, main_grad=np.zeros_like(main0))
    assert np.array_equal(main_z, acc)
