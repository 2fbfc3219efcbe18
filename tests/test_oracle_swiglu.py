"""Pins for the oracle's SiLU-gated activation and its quantisation.

Checked against: hand-worked values (golden fixture), a 200-bit evaluation
(mpmath) rounded to bf16 by hand on random and extreme inputs, torch's
float32 -> bf16 rounding for the direct float64 -> bf16 rounding, a
double-rounding case that a float32 intermediate would get wrong, and the
composition with the (separately pinned) 1x128 quantisers.
"""

import numpy as np
import torch

from conftest import read_golden
from oracle import quant, swiglu


def _gu(pairs):
    g = np.array([p[0] for p in pairs], np.float32)
    u = np.array([p[1] for p in pairs], np.float32)
    return np.concatenate([g, u])[None, :]


def test_worked_examples():
    rows = read_golden("swiglu_worked_example.txt")
    pairs = [(float(g), float(u)) for g, u, _ in rows]
    want = np.array([int(b, 16) for _, _, b in rows], np.uint32)
    h = swiglu.swiglu(_gu(pairs))[0]
    assert np.array_equal(h.view(np.uint32) >> 16, want)


def _bf16_exact(v):
    """bf16 bits of the mpmath value v by hand: quantum 2^(e-7) (2^-133 below
    2^-126), round half to even on the scaled value."""
    import mpmath
    if v == 0:
        return 0x8000 if mpmath.sign(v) < 0 else 0
    a = abs(v)
    e = int(mpmath.floor(mpmath.log(a, 2)))
    while mpmath.mpf(2) ** e > a:
        e -= 1
    while mpmath.mpf(2) ** (e + 1) <= a:
        e += 1
    qe = max(e - 7, -133)
    t = a / mpmath.mpf(2) ** qe
    n = int(mpmath.floor(t))
    frac = t - n
    if frac > 0.5 or (frac == 0.5 and n % 2 == 1):
        n += 1
    val = np.float32(float(mpmath.mpf(n) * mpmath.mpf(2) ** qe))
    bits = int(val.view(np.uint32)) >> 16
    return bits | (0x8000 if v < 0 else 0)


def test_against_200_bit_evaluation():
    import mpmath
    mpmath.mp.prec = 200
    rng = np.random.default_rng(11)
    g = torch.from_numpy((rng.standard_t(4, 3000) * 0.5).astype(np.float32)).to(torch.bfloat16).float().numpy()
    u = torch.from_numpy((rng.standard_t(4, 3000) * 0.5).astype(np.float32)).to(torch.bfloat16).float().numpy()
    extra = [(-700.0, 1.0), (-90.0, 3.0), (-88.0, 1.0), (-80.0, 2.0), (80.0, 1.5), (100.0, -2.0), (1e-30, 1e-10),
             (3e38, 1.0), (-3e38, 1.0), (0.0, -1.0), (-0.0, 1.0)]
    g = np.concatenate([g, np.array([p[0] for p in extra], np.float32)])
    u = np.concatenate([u, np.array([p[1] for p in extra], np.float32)])
    g = torch.from_numpy(g).to(torch.bfloat16).float().numpy()
    u = torch.from_numpy(u).to(torch.bfloat16).float().numpy()
    h = swiglu.swiglu(np.concatenate([g, u])[None, :])[0]
    for gv, uv, hv in zip(g, u, h):
        mg, mu = mpmath.mpf(float(gv)), mpmath.mpf(float(uv))
        exact = mg * mu / (1 + mpmath.exp(-mg))
        want = _bf16_exact(exact)
        if exact == 0:  # the sign of a zero product follows g * u
            want = 0x8000 if np.signbit(np.float32(gv)) != np.signbit(np.float32(uv)) else 0
        got = int(np.float32(hv).view(np.uint32)) >> 16
        if abs(exact) > mpmath.mpf("3.3e38"):  # beyond the largest finite bf16
            assert np.isinf(hv) and np.sign(hv) == mpmath.sign(exact)
            continue
        assert got == want, (gv, uv, float(exact), hex(got), hex(want))


def test_direct_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000).astype(np.float32)
         * np.exp2(rng.integers(-140, 120, 200000)).astype(np.float32))
    a = swiglu.bf16_round_f64(x.astype(np.float64))
    b = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_direct_rounding_avoids_double_rounding():
    # 1 + 2^-8 is the bf16 midpoint between 1 and 1 + 2^-7.  1 + 2^-8 + 2^-40
    # rounds to that midpoint in float32 (then to 1.0, ties to even), but
    # directly it is above the midpoint: 1 + 2^-7.
    v = np.array([1 + 2.0 ** -8 + 2.0 ** -40, -(1 + 2.0 ** -8 + 2.0 ** -40), 1 + 2.0 ** -8], np.float64)
    out = swiglu.bf16_round_f64(v)
    assert out[0] == np.float32(1 + 2.0 ** -7) and out[1] == -np.float32(1 + 2.0 ** -7) and out[2] == 1.0
    assert torch.tensor(v[0], dtype=torch.float32).to(torch.bfloat16).item() == 1.0  # the double rounding


def test_quantisation_is_the_1x128_quantisers_of_h():
    rng = np.random.default_rng(2)
    gu = torch.from_numpy((rng.standard_t(4, (256, 512)) * 0.5).astype(np.float32)).to(torch.bfloat16)
    gu = gu.float().numpy()
    for mode in ("amax448", "pow2", "mul_recip"):
        h, q, s, qT, sT = swiglu.quantize_swiglu_1x128(gu, mode)
        assert h.shape == (256, 256)
        q2, s2 = quant.quantize_act_1x128(h, mode)
        qT2, sT2 = quant.quantize_act_tokens_1x128(h, mode)
        assert np.array_equal(q, q2) and np.array_equal(s, s2)
        assert np.array_equal(qT, qT2) and np.array_equal(sT, sT2)
    # h is bf16-valued
    assert np.array_equal(h, torch.from_numpy(h).to(torch.bfloat16).float().numpy())
