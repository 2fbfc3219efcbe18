"""Pins for the oracle's E4M3 codec and bf16 rounding.

The oracle's tables are checked against things other than themselves: the
hand-written format values of the FP8 formats paper (golden fixture), torch's
own float8_e4m3fn / bfloat16 conversions (library routines), and closed-form
properties (midpoints, saturation, sign of zero).
"""

import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats


def torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_golden_format_values():
    table = formats.e4m3_decode_table()
    rows = read_golden("e4m3_format_values.txt")
    assert len(rows) >= 15
    for code_s, val_s in rows:
        code = int(code_s, 16)
        want = float(val_s)
        got = table[code]
        if math.isnan(want):
            assert math.isnan(got), code_s
        else:
            assert got == want, code_s
            assert math.copysign(1.0, got) == math.copysign(1.0, want), code_s


def test_decode_matches_torch_float8_for_all_codes():
    ours = formats.e4m3_decode_table()
    ref = torch_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_decode_closed_form_properties():
    t = formats.e4m3_decode_table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)          # strictly increasing codes
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6
    assert np.array_equal(t[0x80:0xFF], -pos)  # sign symmetry
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    # 8 values per binade above the subnormals, spaced by 2^(e-3)
    for e in range(-6, 9):
        b = pos[(pos >= 2.0 ** e) & (pos < 2.0 ** (e + 1))]
        assert len(b) == (7 if e == 8 else 8)  # 480 would be S.1111.111, which is NaN
        assert np.allclose(np.diff(b), 2.0 ** (e - 3))


def test_encode_round_trips_every_finite_code():
    t = formats.e4m3_decode_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = t[codes].astype(np.float32)
    vals[codes == 0x80] = -0.0
    assert np.array_equal(formats.e4m3_encode(vals), codes)


def test_encode_midpoints_tie_to_even_and_neighbours():
    t = formats.e4m3_decode_table()
    for c in range(0x7E):
        lo, hi = t[c], t[c + 1]
        mid = np.float32((lo + hi) / 2)  # exact in fp32
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert formats.e4m3_encode(mid)[()] == even
        assert formats.e4m3_encode(np.nextafter(mid, np.float32(0)))[()] == c
        assert formats.e4m3_encode(np.nextafter(mid, np.float32(1e9)))[()] == c + 1
        assert formats.e4m3_encode(-mid)[()] == (even | 0x80)


def test_encode_saturates_and_handles_specials():
    enc = lambda v: int(formats.e4m3_encode(np.float32(v))[()])
    assert enc(448.0) == 0x7E
    assert enc(463.99) == 0x7E
    assert enc(464.0) == 0x7E
    assert enc(480.0) == 0x7E
    assert enc(1e30) == 0x7E
    assert enc(-1e30) == 0xFE
    assert enc(np.inf) == 0x7E and enc(-np.inf) == 0xFE
    assert enc(np.nan) == 0x7F
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(1e-30) == 0x00 and enc(-1e-30) == 0x80
    assert enc(2.0 ** -10) == 0x00  # tie between 0 and 2^-9 -> even (0)
    assert enc(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01


def test_encode_matches_torch_float8_in_range():
    rng = np.random.default_rng(1234)
    # log-uniform magnitudes covering subnormals to the max, random signs
    mags = np.exp2(rng.uniform(-14, np.log2(448.0), 400000)).astype(np.float32)
    vals = mags * rng.choice([-1, 1], mags.size).astype(np.float32)
    # every bf16 bit pattern whose value is finite and within range
    bits = np.arange(65536, dtype=np.uint32) << 16
    bf = bits.view(np.float32)
    bf = bf[np.isfinite(bf) & (np.abs(bf) <= 448.0)]
    x = np.concatenate([vals, bf])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(formats.e4m3_encode(x), ref)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 30, 200000))).astype(np.float32)
    # exact ties: bf16 values plus half a bf16 ulp
    base = rng.standard_normal(1000).astype(np.float32)
    bu = (base.view(np.uint32) & 0xFFFF0000) | 0x8000
    x = np.concatenate([x, bu.view(np.float32), np.float32([0.0, -0.0, 3.0e38, -3.0e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    ours = formats.bf16_round(x)
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(formats.bf16_from_bits(formats.bf16_bits(ours)), ours)
