"""Number formats used by the blockwise-FP8 linear layer (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

E4M3 is the 8-bit floating-point format the Puro-2B paper selects for the
Transformer linear-layer operands ("Puro-2B: Poor Lab's Qwen2-1.5B Trained on
RTX 5090 within $5090", section 3.2), defined in Micikevicius et al. (2022),
"FP8 Formats for Deep Learning":

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0 encodes subnormals  m/8 * 2^(1-7) = m * 2^-9;
* exponent fields 1..15 encode normals (1 + m/8) * 2^(e-7);
* there are no infinities; S.1111.111 (0x7F / 0xFF) is NaN, so the largest
  finite magnitude is S.1111.110 = 1.75 * 2^8 = 448.

Encoding here is round-to-nearest with ties to the even code (the code whose
mantissa LSB is 0), followed by "satfinite" saturation: every finite or
infinite value whose magnitude exceeds 448 maps to +-448.  NaN maps to 0x7F.
The sign of zero is kept (-0.0 -> 0x80).

bf16 rounding is round-to-nearest-even of a binary32 value to its upper 16
bits, the usual bfloat16 definition.
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN_CODE = 0x7F


def e4m3_decode_table():
    """Return float64[256]: the value of every E4M3 code (NaN for 0x7F/0xFF).

    Written directly from the field definitions above.
    """
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if (code >> 7) & 1 else 1.0
        exp_field = (code >> 3) & 0xF
        mant_field = code & 0x7
        if exp_field == 0xF and mant_field == 0x7:
            table[code] = np.nan
        elif exp_field == 0:
            table[code] = sign * mant_field * 2.0 ** -9
        else:
            table[code] = sign * (1.0 + mant_field / 8.0) * 2.0 ** (exp_field - 7)
    return table


_DECODE = e4m3_decode_table()
# Non-negative finite magnitudes, indexed by code 0x00..0x7E; strictly increasing.
_POS = _DECODE[:0x7F].copy()


def e4m3_decode(codes):
    """Decode an array of uint8 E4M3 codes to float64."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """Encode float32 values to uint8 E4M3 codes (RNE, satfinite).

    ``x`` is converted to float32 first; the rounding is a single rounding of
    that exact binary32 value to the nearest E4M3 magnitude.
    """
    x32 = np.asarray(x, dtype=np.float32)
    ax = np.abs(x32).astype(np.float64)  # exact widening
    nan = np.isnan(ax)
    ax = np.where(nan, 0.0, ax)
    ax = np.minimum(ax, E4M3_MAX)  # satfinite: everything above 448 -> 448

    hi = np.searchsorted(_POS, ax, side="left")  # first magnitude >= ax
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = ax - _POS[lo]
    d_hi = _POS[hi] - ax
    exact = d_hi == 0.0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(exact | pick_hi, hi, lo).astype(np.uint8)

    code = code | (np.signbit(x32).astype(np.uint8) << 7)
    code = np.where(nan, np.uint8(E4M3_NAN_CODE), code)
    return code.astype(np.uint8)


def bf16_round(x):
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns float32 values that are exactly representable in bfloat16.  NaN
    stays NaN; values that round past the largest finite bf16 become inf.
    """
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x32), np.float32(np.nan), out)


def bf16_bits(x):
    """uint16 bit patterns of bf16-representable float32 values."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (x32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits):
    """float32 values of uint16 bf16 bit patterns (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
