"""Element encodings used by NVFP4 and MXFP4 (test infrastructure only).

E2M1 is the 4-bit element type of both formats.  The QUADS abstract calls it
"the coarse E2M1 grid" and the gist.science explainer (Technisches Resuemee
section 1) says it has only 8 non-negative levels per sign.  The levels
themselves come from the E2M1 definition (1 sign, 2 exponent, 1 mantissa
bit, exponent bias 1, subnormal at exponent 0, no inf/NaN):
    code 0..7  ->  0, 0.5, 1, 1.5, 2, 3, 4, 6      (bit 3 = sign)

E4M3 (the NVFP4 block scale) is FP8 E4M3FN: bias 7, 3 mantissa bits,
subnormals at exponent field 0, largest finite 448, byte 0x7F is NaN.  Only
the non-negative half is ever used for a scale.

E8M0 (the MXFP4 block scale) is a bare biased exponent: byte b means 2**(b-127).

Every encoder below is written as "pick the nearest representable value,
ties to the even code", with saturation to the largest finite value, which
is round-to-nearest-even with satfinite for these formats.
"""

import numpy as np
import torch

# ---------------------------------------------------------------- E2M1 ----

#: magnitudes of E2M1 codes 0..7 (code = index), from the E2M1 definition.
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nearest_even(table, v):
    """Index of the entry of ascending ``table`` nearest to each ``v`` (>= 0).

    Ties between two neighbours go to the even index.  Values above the last
    entry map to the last entry (saturation); the table's codes ascend with
    value, so "even index" is "even code".
    """
    v = np.asarray(v, dtype=np.float64)
    hi = np.searchsorted(table, v, side="left")  # first entry >= v
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = np.abs(v - table[lo])
    d_hi = np.abs(table[hi] - v)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    # at or beyond the top entry: saturate (the distances above lose all
    # precision for huge v and could otherwise tie)
    return np.where(v >= table[-1], len(table) - 1, idx)


def e2m1_encode(y):
    """Round float32 values ``y`` to E2M1 codes (uint8, low 4 bits).

    Magnitude: nearest of the 8 levels, ties to the even code, saturating
    at 6.  Sign bit (bit 3) = signbit(y), so a negative value that rounds to
    zero gives code 0x8 (negative zero), as an IEEE-style conversion does.
    Inputs are finite.
    """
    y = np.asarray(y, dtype=np.float32)
    mag_code = _nearest_even(E2M1_MAGNITUDES, np.abs(y).astype(np.float64))
    sign = np.signbit(y).astype(np.uint8) << 3
    return (mag_code.astype(np.uint8) | sign).astype(np.uint8)


def e2m1_value(code):
    """Decode E2M1 codes (low 4 bits of each uint8) to float64."""
    code = np.asarray(code, dtype=np.uint8) & 0xF
    mag = E2M1_MAGNITUDES[code & 0x7]
    return np.where(code & 0x8, -mag, mag)


# ---------------------------------------------------------------- E4M3 ----

def e4m3_decode(byte):
    """Decode non-negative FP8 E4M3FN bytes 0x00..0x7E to float64."""
    b = np.asarray(byte, dtype=np.int64)
    e = (b >> 3) & 0xF
    m = b & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    nrm = (1.0 + m / 8.0) * np.power(2.0, e - 7)
    return np.where(e == 0, sub, nrm)


#: all 127 finite non-negative E4M3 values, ascending, index == byte.
E4M3_VALUES = e4m3_decode(np.arange(0x7F))
E4M3_MAX = 448.0


def e4m3_encode(v):
    """Round non-negative values to E4M3 bytes: nearest, ties to even byte,
    saturating at 448 (byte 0x7E).  The byte's LSB is the mantissa LSB, so
    "even byte" is round-half-to-even."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0) or np.any(~np.isfinite(v)):
        raise ValueError("e4m3_encode: scale inputs must be finite and >= 0")
    return _nearest_even(E4M3_VALUES, v).astype(np.uint8)


def e4m3_encode_signed(v):
    """Round finite values to E4M3FN bytes with the sign in bit 7 (the
    element type of the FP8 compensation operands): the magnitude as
    :func:`e4m3_encode` (nearest, ties to even, saturating at 448), the sign
    bit = signbit(v), so a negative value that rounds to zero gives 0x80."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(~np.isfinite(v)):
        raise ValueError("e4m3_encode_signed: inputs must be finite")
    mag = _nearest_even(E4M3_VALUES, np.abs(v)).astype(np.uint8)
    return (mag | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def e4m3_value(byte):
    """Decode E4M3FN bytes with a sign bit (0x7F and 0xFF, the NaNs,
    excluded) to float64."""
    b = np.asarray(byte, dtype=np.uint8)
    mag = e4m3_decode(b & 0x7F)
    return np.where(b & 0x80, -mag, mag)


# ---------------------------------------------------------------- E8M0 ----

def e8m0_value(byte):
    """Decode E8M0 bytes to float64: 2**(byte - 127)."""
    return np.power(2.0, np.asarray(byte, dtype=np.float64) - 127.0)


# ---------------------------------------------------------------- BF16 ----

def bf16_round(x):
    """Round float32 values to bfloat16 (round-to-nearest-even), returned as
    float32.  Uses torch's CPU conversion, a library routine."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits(x):
    """bfloat16 bit patterns (uint16) of float32 values rounded RNE."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_from_bits(bits):
    """float32 values of bfloat16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
