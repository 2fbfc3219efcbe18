"""Pins for the oracle's blockwise quantisers.

Checked against: a hand-worked group (golden fixture), torch's float8 cast of
a torch-computed x/s (library division and rounding), closed-form invariants
of the amax/448 rule, the E4M3 round-trip error bound, group locality under
single-element perturbations, and the paper's qualitative claim that local
scales beat one scale per tensor when outliers are present.  The power-of-two
mode is pinned by its own worked group, an exact-rational search for the
scale over every positive bf16 amax, and torch's float8 cast of the exactly
scaled values.  The reciprocal-multiply mode is pinned by its own worked
group (where it and the division give different codes), an exact-rational
evaluation of its rule with a hand-written float32 rounding, and closed-form
properties: every bf16 amax codes to 448, and codes stay within one E4M3
step of the division's.
"""

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats, quant
from blockwise_fp8_linear_quantise_b300 import workloads

T_DEC = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_exact(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def test_worked_example_group():
    rows = read_golden("quant_worked_example.txt")
    assert rows[0][0] == "scale"
    want_s = float(rows[0][1])
    x = np.zeros((1, 128), np.float32)
    want = np.zeros(128, np.uint8)
    for pos, xv, _xs, code in rows[1:]:
        x[0, int(pos)] = np.float32(float(xv))
        want[int(pos)] = int(code, 16)
    assert np.array_equal(bf16_exact(x).view(np.uint32), x.view(np.uint32))
    q, s = quant.quantize_act_1x128(np.tile(x, (128, 1)))
    assert s.shape == (1, 128) and np.all(s == want_s)
    assert np.array_equal(q[0], want) and np.array_equal(q[77], want)


def test_zero_group_gets_unit_scale():
    x = np.zeros((128, 256), np.float32)
    x[3, 130] = -0.0
    x[5, 200] = 1.0
    q, s = quant.quantize_act_1x128(x)
    assert s[0, 3] == 1.0 and s[1, 3] == 1.0 and s[0, 5] == 1.0
    assert q[3, 130] == 0x80 and np.count_nonzero(q[3]) == 1
    assert s[1, 5] == np.float32(1.0) / np.float32(448.0) and q[5, 200] == 0x7E


def test_quantised_codes_match_torch_cast_of_library_division():
    wl = workloads.make("tiny")
    x = workloads.tensor(wl, "x").float().numpy()
    q, s = quant.quantize_act_1x128(x)
    # independent: group amax and division via torch, cast via torch float8
    xt = torch.from_numpy(x).view(256, 2, 128)
    amax = xt.abs().amax(dim=2)
    st = amax / 448.0
    assert np.array_equal(st.numpy(), s.T)
    y = xt / st[:, :, None]
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(256, 256).numpy()
    assert np.array_equal(q, ref)


def test_every_bf16_pattern_in_groups():
    # all finite bf16 values, arranged in groups of 128 with a shared anchor
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    vals = bits[np.isfinite(bits)]
    n = vals.size - vals.size % 127
    g = vals[:n].reshape(-1, 127)
    for anchor in (1.0, 3.0e38, 2.0 ** -100):
        x = np.concatenate([np.full((g.shape[0], 1), anchor, np.float32), g], axis=1)
        x = x[: (x.shape[0] // 128) * 128]
        q, s = quant.quantize_act_1x128(x)
        amax = np.abs(x).max(axis=1)
        st = torch.from_numpy(amax) / 448.0
        assert np.array_equal(s[0], st.numpy())
        ref = (torch.from_numpy(x) / st[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        ok = np.isfinite(x / s[0][:, None]) & (np.abs(x / s[0][:, None]) <= 448)
        assert np.array_equal(q[ok], ref[ok])
        assert np.all(np.abs(T_DEC[q]) <= 448)


def _roundtrip_ok(x, q, s_full):
    dq = T_DEC[q] * s_full.astype(np.float64)
    err = np.abs(x.astype(np.float64) - dq)
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * s_full) * (1 + 2.0 ** -20) + 1e-45
    return np.all(err <= bound)


@pytest.mark.parametrize("name,tag", [("tiny", "x"), ("tiny", "w")])
def test_invariants_rows_tokens_weights(name, tag):
    wl = workloads.make(name)
    x = workloads.tensor(wl, tag).float().numpy()
    R, C = x.shape
    # rows
    q, s = quant.quantize_act_1x128(x)
    assert q.shape == (R, C) and s.shape == (C // 128, R)
    s_full = np.repeat(s.T, 128, axis=1)
    assert _roundtrip_ok(x, q, s_full)
    assert np.all(np.abs(T_DEC[q]) <= 448)
    for r in range(R):
        for g in range(C // 128):
            grp = q[r, g * 128:(g + 1) * 128]
            assert np.any((grp == 0x7E) | (grp == 0xFE))
            amax = np.abs(x[r, g * 128:(g + 1) * 128]).max()
            assert abs(float(s[g, r]) * 448.0 - amax) <= amax * 2.0 ** -23
    # tokens (transposed storage)
    qT, sT = quant.quantize_act_tokens_1x128(x)
    assert qT.shape == (C, R) and sT.shape == (R // 128, C)
    sT_full = np.repeat(sT, 128, axis=0)  # [R, C] scale of x[r, c]
    assert _roundtrip_ok(x, qT.T, sT_full)
    # weights
    wq, wqT, ws = quant.quantize_w_128x128(x)
    assert wq.shape == (R, C) and np.array_equal(wqT, wq.T) and ws.shape == (R // 128, C // 128)
    ws_full = np.repeat(np.repeat(ws, 128, axis=0), 128, axis=1)
    assert _roundtrip_ok(x, wq, ws_full)
    for b in range(R // 128):
        for c in range(C // 128):
            blk = wq[b * 128:(b + 1) * 128, c * 128:(c + 1) * 128]
            assert np.any((blk == 0x7E) | (blk == 0xFE))


def test_power_of_two_amax_gives_exact_scale():
    x = np.zeros((128, 128), np.float32)
    for r in range(128):
        x[r, r] = np.float32(448.0 * 2.0 ** (r - 64))
    _, s = quant.quantize_act_1x128(x)
    assert np.array_equal(s[0], np.float32(2.0) ** (np.arange(128) - 64).astype(np.float32))


def test_group_locality():
    rng = np.random.default_rng(3)
    x = bf16_exact(rng.standard_normal((256, 384)))
    q, s = quant.quantize_act_1x128(x)
    qT, sT = quant.quantize_act_tokens_1x128(x)
    wq, _, ws = quant.quantize_w_128x128(x)
    r0, c0 = 200, 260
    y = x.copy()
    y[r0, c0] = 100.0
    q2, s2 = quant.quantize_act_1x128(y)
    qT2, sT2 = quant.quantize_act_tokens_1x128(y)
    wq2, _, ws2 = quant.quantize_w_128x128(y)
    # rows: only group (r0, c0//128) changes
    ds = np.argwhere(s != s2)
    assert ds.tolist() == [[c0 // 128, r0]]
    dq = np.argwhere(q != q2)
    assert np.all(dq[:, 0] == r0) and np.all(dq[:, 1] // 128 == c0 // 128)
    # tokens: only group (r0//128, c0) changes
    assert np.argwhere(sT != sT2).tolist() == [[r0 // 128, c0]]
    dqT = np.argwhere(qT != qT2)
    assert np.all(dqT[:, 0] == c0) and np.all(dqT[:, 1] // 128 == r0 // 128)
    # weight block: only block (r0//128, c0//128) changes
    assert np.argwhere(ws != ws2).tolist() == [[r0 // 128, c0 // 128]]
    dw = np.argwhere(wq != wq2)
    assert np.all(dw[:, 0] // 128 == r0 // 128) and np.all(dw[:, 1] // 128 == c0 // 128)


def _rel_fro(x, dq):
    return np.linalg.norm(x - dq) / np.linalg.norm(x)


@pytest.mark.parametrize("name", ["tiny", "mlp_gateup"])
def test_blockwise_beats_per_tensor_on_outliers(name):
    wl = workloads.make(name)
    x = workloads.tensor(wl, "x").float().numpy()
    if x.shape[0] > 2048:
        x = x[:2048]
    x = x.astype(np.float64)
    q, s = quant.quantize_act_1x128(x)
    blk = _rel_fro(x, T_DEC[q] * np.repeat(s.T, 128, axis=1))
    qt, st = quant.quantize_per_tensor(x)
    per = _rel_fro(x, T_DEC[qt] * float(st))
    assert blk < per
    assert blk < 0.05


# ---------------------------------------------------------------- power of two


def test_pow2_worked_example_group():
    rows = read_golden("pow2_quant_worked_example.txt")
    assert rows[0][0] == "scale"
    want_s = float(rows[0][1])
    x = np.zeros((1, 128), np.float32)
    want = np.zeros(128, np.uint8)
    for pos, xv, _xs, code in rows[1:]:
        x[0, int(pos)] = np.float32(float(xv))
        want[int(pos)] = int(code, 16)
    assert np.array_equal(bf16_exact(x).view(np.uint32), x.view(np.uint32))
    q, s = quant.quantize_act_1x128(np.tile(x, (128, 1)), scale_mode="pow2")
    assert np.all(s == want_s)
    assert np.array_equal(q[0], want) and np.array_equal(q[127], want)


def _pow2_scale_by_search(amax):
    """Smallest k with 2^k * 448 >= amax, by exact rational comparison."""
    from fractions import Fraction
    a = Fraction(float(amax))
    k = 0
    while Fraction(2) ** k * 448 < a:
        k += 1
    while Fraction(2) ** (k - 1) * 448 >= a:
        k -= 1
    return k


def test_pow2_scale_of_every_bf16_amax():
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16  # every positive finite bf16 value
    amax = bits.view(np.float32)
    s = quant.group_scale_pow2(amax)
    f, e = np.frexp(s.astype(np.float64))
    assert np.all(f == 0.5)  # powers of two
    for a, sv in zip(amax[::7], s[::7]):  # exact search on a stride through all binades
        assert float(sv) == 2.0 ** _pow2_scale_by_search(a), a
    # closed-form bounds on all of them: s >= amax/448 > s/2, in exact float64 products
    a64, s64 = amax.astype(np.float64), s.astype(np.float64)
    assert np.all(448.0 * s64 >= a64) and np.all(448.0 * s64 / 2 < a64)
    assert quant.group_scale_pow2(np.float32(0.0)) == 1.0


@pytest.mark.parametrize("name,tag", [("mlp_gateup", "x"), ("mlp_down", "x"), ("attn_proj", "x")])
def test_pow2_codes_match_torch_cast_of_exact_scaling(name, tag):
    wl = workloads.make(name)
    x = workloads.tensor(wl, tag).float().numpy()[:256, :512]
    q, s = quant.quantize_act_1x128(x, scale_mode="pow2")
    xt = torch.from_numpy(x).view(256, 4, 128)
    amax = xt.abs().amax(dim=2)
    # independent scale: 2^ceil(log2(amax/448)) from torch's own frexp of the float64 quotient
    mant, ex = torch.frexp(amax.double() / 448.0)
    k = torch.where(mant == 0.5, ex - 1, ex)
    st = torch.ldexp(torch.ones_like(amax, dtype=torch.float64), k).float()
    assert np.array_equal(st.numpy(), s.T)
    y = xt * (1.0 / st)[:, :, None]  # multiplying by 2^-k is exact here
    ref = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(256, 512).numpy()
    assert np.array_equal(q, ref)
    # nothing saturates: each group's amax/s lies in (224, 448] exactly, so its
    # largest code decodes into [224, 448] (E4M3 rounding may reach 224)
    ratio = amax.double().numpy() / st.double().numpy()
    assert np.all((ratio > 224) & (ratio <= 448))
    dec = T_DEC[q].reshape(256, 4, 128)
    top = np.abs(dec).max(axis=2)
    assert np.all((top >= 224) & (top <= 448))


def test_pow2_weights_and_tokens_use_the_same_rule():
    wl = workloads.make("tiny")
    w = workloads.tensor(wl, "w").float().numpy()
    q, qT, s = quant.quantize_w_128x128(w, scale_mode="pow2")
    blk = np.abs(w.reshape(2, 128, 2, 128)).max(axis=(1, 3))
    assert np.array_equal(s, quant.group_scale_pow2(blk))
    assert np.array_equal(qT, q.T)
    x = workloads.tensor(wl, "x").float().numpy()
    qt, st = quant.quantize_act_tokens_1x128(x, scale_mode="pow2")
    q2, s2 = quant.quantize_act_1x128(np.ascontiguousarray(x.T), scale_mode="pow2")
    assert np.array_equal(qt, q2) and np.array_equal(st, s2)
    with pytest.raises(ValueError):
        quant.quantize_act_1x128(x, scale_mode="ue8m0")


# ------------------------------------------------------- reciprocal multiply


def test_mul_recip_worked_example_group():
    rows = read_golden("mul_recip_quant_worked_example.txt")
    assert rows[0][0] == "scale" and rows[1][0] == "multiplier"
    want_s, want_m = float.fromhex(rows[0][1]), float.fromhex(rows[1][1])
    x = np.zeros((1, 128), np.float32)
    want = np.zeros(128, np.uint8)
    want_div = np.zeros(128, np.uint8)
    for pos, xv, code, code_div in rows[2:]:
        x[0, int(pos)] = np.float32(float(xv))
        want[int(pos)] = int(code, 16)
        want_div[int(pos)] = int(code_div, 16)
    assert np.array_equal(bf16_exact(x).view(np.uint32), x.view(np.uint32))
    assert float(quant.group_multiplier(np.float32(13.0))) == want_m
    q, s = quant.quantize_act_1x128(np.tile(x, (128, 1)), scale_mode="mul_recip")
    assert np.all(s == want_s)
    assert np.array_equal(q[0], want) and np.array_equal(q[127], want)
    qd, sd = quant.quantize_act_1x128(np.tile(x, (128, 1)))
    assert np.array_equal(sd, s) and np.array_equal(qd[0], want_div)


def _rn_f32(v):
    """The float32 nearest to the Fraction v (ties to even, gradual underflow),
    +-inf where it rounds beyond the largest finite float32."""
    from fractions import Fraction
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = a // quantum
    r = a - n * quantum
    if 2 * r > quantum or (2 * r == quantum and n % 2 == 1):
        n += 1
    out = n * quantum
    mag = float("inf") if out >= Fraction(2) ** 128 else float(out)
    return -mag if v < 0 else mag


def test_mul_recip_codes_match_exact_rational_evaluation():
    from fractions import Fraction
    wl = workloads.make("mlp_down")
    x = workloads.tensor(wl, "x").float().numpy()[:64, :256].copy()
    # two groups with extreme amax: a tiny one whose multiplier saturates,
    # and one near the top of the bf16 range
    x[62, :128] *= np.float32(2.0 ** -126)
    x[63, 128:] *= np.float32(2.0 ** 100)
    x = bf16_exact(x)
    x = np.concatenate([x, -x], axis=0)  # 128 rows
    q, s = quant.quantize_act_1x128(x, scale_mode="mul_recip")
    fmax = float(np.finfo(np.float32).max)
    ys = np.zeros(x.shape, np.float32)
    for r in range(x.shape[0]):
        for g in range(2):
            xs = x[r, 128 * g:128 * (g + 1)]
            amax = Fraction(float(np.abs(xs).max()))
            assert float(s[g, r]) == _rn_f32(amax / 448)
            m = min(_rn_f32(Fraction(448) / amax), fmax)
            if r % 64 == 62 and g == 0:
                assert m == fmax  # the saturated multiplier is exercised
            for c, xv in enumerate(xs):
                # m > 0: the product has the sign of x, zeros included
                ys[r, 128 * g + c] = np.copysign(_rn_f32(Fraction(float(xv)) * Fraction(m)), xv)
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_mul_recip_properties_over_every_bf16_amax():
    from fractions import Fraction
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16  # every positive finite bf16 value
    amax = bits.view(np.float32)
    m = quant.group_multiplier(amax)
    fmax = float(np.finfo(np.float32).max)
    for a, mv in zip(amax[::11], m[::11]):
        assert float(mv) == min(_rn_f32(Fraction(448) / Fraction(float(a))), fmax), a
    # every group's amax codes to 448 unless its multiplier saturates
    n = amax.size - amax.size % 128
    x = amax[:n].reshape(-1, 128)  # rows of increasing bf16 values: amax is the last
    x = x[: (x.shape[0] // 128) * 128]
    q, s = quant.quantize_act_1x128(x, scale_mode="mul_recip")
    top = q[:, 127]
    unsat = quant.group_multiplier(x[:, 127]) < np.float32(fmax)
    assert np.all(top[unsat] == 0x7E) and np.all(top[~unsat] < 0x7E)
    # within one E4M3 step of the division, same sign, same scales
    qd, sd = quant.quantize_act_1x128(x)
    assert np.array_equal(s, sd)
    diff = np.abs((q & 0x7F).astype(int) - (qd & 0x7F).astype(int))
    assert np.all(diff[unsat] <= 1) and np.array_equal(q & 0x80, qd & 0x80)


@pytest.mark.parametrize("name,tag", [("tiny", "x"), ("tiny", "w")])
def test_mul_recip_invariants_rows_tokens_weights(name, tag):
    wl = workloads.make(name)
    x = workloads.tensor(wl, tag).float().numpy()
    R, C = x.shape
    q, s = quant.quantize_act_1x128(x, scale_mode="mul_recip")
    assert _roundtrip_ok(x, q, np.repeat(s.T, 128, axis=1))
    qd, sd = quant.quantize_act_1x128(x)
    assert np.array_equal(s, sd)
    assert np.all(np.abs((q & 0x7F).astype(int) - (qd & 0x7F).astype(int)) <= 1)
    qT, sT = quant.quantize_act_tokens_1x128(x, scale_mode="mul_recip")
    q2, s2 = quant.quantize_act_1x128(np.ascontiguousarray(x.T), scale_mode="mul_recip")
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)
    wq, wqT, ws = quant.quantize_w_128x128(x, scale_mode="mul_recip")
    assert np.array_equal(wqT, wq.T)
    assert _roundtrip_ok(x, wq, np.repeat(np.repeat(ws, 128, axis=0), 128, axis=1))
    blk = np.abs(x.reshape(R // 128, 128, C // 128, 128)).max(axis=(1, 3))
    mb = quant.group_multiplier(blk)
    ref = quant.quantize_values_mul(x.reshape(R // 128, 128, C // 128, 128), mb[:, None, :, None]).reshape(R, C)
    assert np.array_equal(wq, ref)


def golden_weight_block():
    """W [256, 256] of the hand-worked weight fixture, and its listed scales
    and codes."""
    i, j = np.meshgrid(np.arange(256), np.arange(256), indexing="ij")
    w = ((((7 * i + 3 * j) % 17) - 8) * 2.0 ** -8).astype(np.float32)
    w[5, 7], w[0, 128], w[255, 127], w[128, 255] = 448.0, -3.5, 0.875, 1.0
    scales, codes = {}, {}
    for row in read_golden("weight_block_worked_example.txt"):
        if row[0] == "scale":
            scales[(int(row[1]), int(row[2]))] = int(row[4], 16)
        else:
            codes[(int(row[1]), int(row[2]))] = (np.float32(float(row[3])), int(row[5], 16))
    return w, scales, codes


def test_weight_block_worked_example():
    w, scales, codes = golden_weight_block()
    assert np.array_equal(bf16_exact(w).view(np.uint32), w.view(np.uint32))
    q, qT, s = quant.quantize_w_128x128(w)
    assert s.shape == (2, 2)
    for (bi, bj), bits in scales.items():
        assert s[bi, bj].view(np.uint32) == bits, (bi, bj)
    for (ii, jj), (x, code) in codes.items():
        assert w[ii, jj] == x
        assert q[ii, jj] == code and qT[jj, ii] == code, (ii, jj)
