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
