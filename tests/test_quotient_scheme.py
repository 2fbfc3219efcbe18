"""The kernels' division-free quotient and scales, checked exhaustively on the CPU.

The GPU quantisers (amax/448 mode) form fp32_rn(x / s) without a division:
r = RN(1/s) once per group, y0 = RN(x r), then one FMA correction
Q = RN(y0 + r RN(x - s y0)).  For arbitrary x and s, Markstein's theorem asks
for a faithful y (one more refinement step).  Here the inputs are narrower:
x is bf16 and s = RN(amax / 448) with amax bf16.  Scaling x and amax by the
same power of two leaves y0 and Q unchanged while s stays in [2^-80, 2^100]
(the range the kernels send down this path; a remainder that rounds is then
a normal fp32), so one binade of amax, all 128 bf16 mantissas, with every bf16
x in (0, amax], covers every case.  This test evaluates the scheme there in
exact arithmetic (float64 where it is exact, plus an exact resolution of the
one float64 rounding that is not) and requires Q == fp32(x / s) bit for bit.

No oracle and no GPU code is used: the scheme is restated from the kernels'
header comment, and the reference quotient is numpy's IEEE float32 division.

Two per-group steps are checked the same way, over every positive bf16 amax:
the amax/448 scale (one FMA correction of RN(amax RN(1/448))) against the
IEEE quotient, and the power-of-two mode's exponent read off amax's bits
against an exact rational search.
"""

import numpy as np
import pytest


def _fma32_exact(a, b, c):
    """fp32 RN(a*b + c) for float32 arrays, via float64 with the one inexact
    float64 addition resolved exactly (TwoSum): a*b is exact in float64, and
    the float64 sum is rounded to float32 correctly unless it lands on a
    float32 rounding midpoint, where the TwoSum error decides."""
    p = a.astype(np.float64) * b.astype(np.float64)
    c64 = c.astype(np.float64)
    s = p + c64
    bb = s - p
    err = (p - (s - bb)) + (c64 - bb)  # exact: s + err == p + c64
    out = s.astype(np.float32)
    bits = s.view(np.uint64)
    on_mid = (bits & np.uint64((1 << 29) - 1)) == np.uint64(1 << 28)  # a float32 midpoint (normal range)
    fix = on_mid & (err != 0)
    if np.any(fix):
        lo = (s[fix] - np.ldexp(1.0, np.frexp(s[fix])[1] - 25)).astype(np.float32)  # neighbours of the midpoint
        hi = np.nextafter(lo, np.float32(np.inf))
        pos = s[fix] > 0
        up = np.where(pos, err[fix] > 0, err[fix] < 0)
        out[fix] = np.where(up == pos, np.maximum(lo, hi), np.minimum(lo, hi))
    return out


def _rn32_fraction(v):
    """The float32 nearest to the Fraction v (ties to even), normal range."""
    from fractions import Fraction as F
    if v == 0:
        return np.float32(0.0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while F(2) ** e > a:
        e -= 1
    while F(2) ** (e + 1) <= a:
        e += 1
    q = F(2) ** (e - 23)
    n = a // q
    r = a - n * q
    if 2 * r > q or (2 * r == q and n % 2 == 1):
        n += 1
    out = np.float32(float(n * q))
    return out if v > 0 else -out


def test_fma32_exact_against_fractions():
    from fractions import Fraction as F
    rng = np.random.default_rng(5)
    a = list(rng.standard_normal(600).astype(np.float32))
    b = list(rng.standard_normal(600).astype(np.float32))
    c = list((rng.standard_normal(600) * 2.0 ** rng.integers(-30, 30, 600)).astype(np.float32))
    # float64 sums that land exactly on a float32 midpoint with a nonzero
    # remainder, below (c odd) and above (c odd, negative product) it
    for j in range(1, 41):
        u = 2.0 ** -23
        for sg in (1.0, -1.0):
            a += [np.float32(sg * (1 + j * u)), np.float32(sg * (1 + j * u))]
            b += [np.float32(2.0 ** -24 * (1 - j * u)), np.float32(-(2.0 ** -24) * (1 - j * u))]
            c += [np.float32(sg * (1 + u)), np.float32(sg * (1 + 3 * u))]
    a, b, c = np.array(a, np.float32), np.array(b, np.float32), np.array(c, np.float32)
    got = _fma32_exact(a, b, c)
    want = np.array([_rn32_fraction(F(float(x)) * F(float(y)) + F(float(z))) for x, y, z in zip(a, b, c)],
                    np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    naive = (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)
    assert np.count_nonzero(naive != want) >= 80  # the midpoint branch decides these


def test_one_correction_gives_the_ieee_quotient_for_bf16_inputs():
    bf = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[(bf > 0) & (bf >= 2.0 ** -30)]
    wrong_q1 = 0
    wrong_y0_codes = 0
    n = 0
    for mant in range(128):
        amax = np.float32(1.0 + mant / 128.0)
        s = amax / np.float32(448.0)           # IEEE fp32 quotient
        r = np.float32(1.0) / s                # RN(1/s)
        x = bf[bf <= amax]
        y0 = x * r                             # RN(x r)
        e = _fma32_exact(-np.full_like(x, s), y0, x)       # RN(x - s y0)
        q1 = _fma32_exact(np.full_like(x, r), e, y0)       # RN(y0 + r e)
        want = x / s                           # RN(x / s)
        wrong_q1 += int(np.count_nonzero(q1.view(np.uint32) != want.view(np.uint32)))
        wrong_y0_codes += int(np.count_nonzero(_e4m3_index(y0) != _e4m3_index(want)))
        n += x.size
    assert n > 490_000
    assert wrong_q1 == 0
    assert wrong_y0_codes > 0  # the correction step is needed: y0 alone misses some codes


def _e4m3_index(v):
    """E4M3 code magnitude of positive float32 v (RNE, satfinite), by search
    over the 127 finite magnitudes: index of the nearest, ties to even."""
    mags = np.array([_e4m3_mag(c) for c in range(127)], np.float64)
    v64 = v.astype(np.float64)
    i = np.clip(np.searchsorted(mags, v64), 1, 126)
    lo, hi = mags[i - 1], mags[i]
    pick_hi = (v64 - lo > hi - v64) | ((v64 - lo == hi - v64) & ((i - 1) % 2 == 1))
    idx = np.where(pick_hi, i, i - 1)
    return np.where(v64 >= mags[126], 126, idx)


def _e4m3_mag(c):
    e, m = c >> 3, c & 7
    return m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)


def _positive_bf16():
    return (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)


def test_amax_scale_by_one_correction_is_the_ieee_quotient():
    """s = RN(amax / 448) as the kernels form it for a bf16 amax with a normal
    quotient: q0 = RN(amax c) with c = RN(1/448), then RN(q0 + c RN(amax - 448 q0))."""
    amax = _positive_bf16()
    amax = amax[(amax >= np.float32(448.0 * 2.0 ** -126)) & (amax <= np.float32(float.fromhex("0x1.FEp+127")))]
    c = np.float32(1.0) / np.float32(448.0)
    q0 = amax * c
    r = _fma32_exact(-q0, np.full_like(q0, 448.0), amax)
    s = _fma32_exact(r, np.full_like(r, c), q0)
    want = amax / np.float32(448.0)
    assert amax.size == 31392  # every positive bf16 amax whose quotient is a normal fp32
    assert np.array_equal(s.view(np.uint32), want.view(np.uint32))


def _pow2_k_from_bits(amax):
    """The kernels' exponent of the power-of-two scale, from amax's bits:
    amax = (1 + m) 2^e (fp32 subnormals normalised), k = e - 8 + (m > 0.75)."""
    b = amax.view(np.uint32).astype(np.int64)
    normal = b >= 0x00800000
    e = np.where(normal, (b >> 23) - 127, 0)
    m = np.where(normal, b & 0x007FFFFF, 0)
    sub = ~normal
    if np.any(sub):
        bs = b[sub]
        p = np.floor(np.log2(bs.astype(np.float64))).astype(np.int64)  # exact for integers below 2^23
        e[sub] = p - 149
        m[sub] = (bs << (23 - p)) & 0x007FFFFF
    return e - 8 + (m > 0x00600000)


def test_pow2_exponent_from_bits_is_the_smallest_covering_power():
    from fractions import Fraction as F
    amax = _positive_bf16()
    extra = (np.arange(1, 1 << 12, 7, dtype=np.uint32)).view(np.float32)  # fp32 subnormal amaxes
    amax = np.concatenate([amax, extra])
    k = _pow2_k_from_bits(amax)
    # 2^k >= amax/448 > 2^(k-1), in exact float64 products (448 * 2^k is exact)
    a64 = amax.astype(np.float64)
    assert np.all(448.0 * np.ldexp(1.0, k) >= a64) and np.all(448.0 * np.ldexp(1.0, k - 1) < a64)
    for a, kv in zip(amax[::97], k[::97]):  # exact rationals on a stride
        fa = F(float(a))
        assert F(2) ** int(kv) * 448 >= fa > F(2) ** (int(kv) - 1) * 448


def test_step_on_negated_x_keeps_every_quotient_and_the_sign_of_zero():
    """The quantisers run the step on nx = -x with nr = -RN(1/s):
    y0 = RN(nx nr), e = RN(s y0 + nx), Q = RN(e nr + y0).  Over the same
    exhaustive binade, both signs of x and both zeros, Q must be the IEEE
    quotient bit for bit, sign of zero included (-0 / s = -0)."""
    bf = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[(bf == 0) | (bf >= 2.0 ** -30)]
    n = 0
    for mant in range(0, 128, 3):
        amax = np.float32(1.0 + mant / 128.0)
        s = amax / np.float32(448.0)
        nr = -(np.float32(1.0) / s)
        xp = bf[bf <= amax]
        x = np.concatenate([xp, -xp])
        nx = -x
        y0 = nx * nr
        e = _fma32_exact(y0, np.full_like(x, s), nx)
        q = _fma32_exact(e, np.full_like(x, nr), y0)
        want = x / s
        assert np.array_equal(q.view(np.uint32), want.view(np.uint32)), mant
        n += x.size
    assert n > 300_000
    # the step on x itself loses the sign of -0 (the reason for the negated form)
    x0 = np.array([-0.0], np.float32)
    s = np.float32(1.0) / np.float32(448.0)
    r = np.float32(1.0) / s
    y0 = x0 * r
    q_plain = _fma32_exact(np.full_like(x0, r), _fma32_exact(-np.full_like(x0, s), y0, x0), y0)
    assert not np.signbit(q_plain[0])


def _scaled_quotient(x, s):
    """The quantisers' path for a group scale off the FMA range: p = 2^100
    for s < 1, 2^-64 otherwise, 0 for an infinite s (then s p := 1); two
    correction steps on nxp = -x p with nr = -RN(1 / (s p))."""
    if np.isinf(s):
        p, sp = np.float32(0.0), np.float32(1.0)
    else:
        p = np.float32(2.0 ** 100) if s < 1 else np.float32(2.0 ** -64)
        sp = s * p
    nr = -(np.float32(1.0) / sp)
    with np.errstate(invalid="ignore", under="ignore", over="ignore"):
        nxp = (-x) * p
        y0 = nxp * nr
        sv, nrv = np.full_like(x, sp), np.full_like(x, nr)
        y1 = _fma32_exact(_fma32_exact(y0, sv, nxp), nrv, y0)
        return _fma32_exact(_fma32_exact(y1, sv, nxp), nrv, y1)


@pytest.mark.parametrize("amax_bits", [0x00010000, 0x00800000, 0x02800000, 0x08C00000, 0x0F230000,
                                       0x76000000, 0x76A30000, 0x7A000000, 0x7F7F0000])
def test_prescaled_path_for_extreme_scales(amax_bits):
    """Groups with s = RN(amax/448) outside [2^-80, 2^100] (fp32-subnormal
    scales included): every bf16 x with |x| <= amax, both signs.  The code
    (E4M3 magnitude and sign) must be that of the IEEE quotient, and so must
    Q's bits wherever the quotient is a normal fp32."""
    amax = np.array([amax_bits], np.uint32).view(np.float32)[0]
    with np.errstate(under="ignore"):
        s = amax / np.float32(448.0)
    assert not (2.0 ** -80 <= s <= 2.0 ** 100)
    bf = (np.arange(0, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    xp = bf[bf <= amax]
    x = np.concatenate([xp, -xp])
    q = _scaled_quotient(x, s)
    with np.errstate(under="ignore"):
        want = x / s
    assert np.array_equal(np.signbit(q), np.signbit(want))
    assert np.array_equal(_e4m3_index(np.abs(q)), _e4m3_index(np.abs(want)))
    normal = np.abs(want) >= 2.0 ** -126
    assert np.array_equal(q[normal].view(np.uint32), want[normal].view(np.uint32))
    assert normal[x == amax].all()  # amax / s, near 448, is among them


def test_prescaled_path_for_an_infinite_scale():
    """amax = inf (an infinite input): x / inf is a signed zero for finite x
    and NaN for infinite x; the path with p = 0 gives the same."""
    x = np.array([0.0, -0.0, 1.0, -3.5, 3e38, -1e-40, np.inf, -np.inf], np.float32)
    q = _scaled_quotient(x, np.float32(np.inf))
    with np.errstate(invalid="ignore"):
        want = x / np.float32(np.inf)
    fin = np.isfinite(x)
    assert np.array_equal(q[fin].view(np.uint32), want[fin].view(np.uint32))
    assert np.all(np.isnan(q[~fin])) and np.all(np.isnan(want[~fin]))
