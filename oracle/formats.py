"""E2M1 (FP4) and E4M3 (FP8) formats: decode tables and RNE encoders.

Test infrastructure only (see the package docstring).

The pages ("nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py",
runtime-gsa section) fix the two format maxima: 448 for the E4M3 block scale
and 6 for the E2M1 code, so that x/gsa tops out at 6 * 448 = 2688.  The rest is
the standard definition of the two formats, written out here:

* E2M1: 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.
  Magnitudes for codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  No inf, no NaN.
* E4M3 ("fn" variant): 1 sign bit (bit 7), 4 exponent bits (bias 7),
  3 mantissa bits.  Exponent field 0 is subnormal (m * 2**-9).  Only the
  all-ones pattern S.1111.111 is NaN, so the largest finite value is
  0x7E = 1.75 * 2**8 = 448.  No inf.

Encoding reading (the pages are silent on rounding): round to nearest, ties to
the code whose mantissa LSB is 0 ("ties to even"), saturate magnitudes above
the largest finite value to it ("satfinite"), keep the sign, so a negative
value that rounds to zero encodes as negative zero (E2M1 0x8).  NaN inputs are
outside the contract and raise.

Everything here works on float64 copies of float32 inputs, which is exact.
"""

import numpy as np

# ---------------------------------------------------------------- decoding

#: magnitude of E2M1 codes 0..7 (bit 3 is the sign)
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)

E2M1_MAX = 6.0
E4M3_MAX = 448.0
E4M3_MAX_CODE = 0x7E


def decode_e2m1(codes):
    """Value of each 4-bit E2M1 code (array of ints in 0..15) as float64."""
    c = np.asarray(codes, dtype=np.int64)
    if np.any((c < 0) | (c > 15)):
        raise ValueError("E2M1 codes are 4-bit")
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def _e4m3_value(code):
    """Value of one E4M3 byte from the bit-field definition (float64)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return np.nan
    if e == 0:
        return sign * m * 2.0 ** -9          # subnormal: (m/8) * 2**(1-7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


#: value of every E4M3 byte 0..255 (NaN for 0x7F and 0xFF)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes):
    """Value of each E4M3 byte as float64 (NaN for the two NaN patterns)."""
    c = np.asarray(codes, dtype=np.int64)
    if np.any((c < 0) | (c > 255)):
        raise ValueError("E4M3 codes are bytes")
    return E4M3_TABLE[c]


# ---------------------------------------------------------------- encoding

def _rne_encode(mag, grid, codes):
    """Round non-negative magnitudes onto an ascending grid, ties to even code.

    ``grid[i]`` is the value of ``codes[i]``; codes ascend with value and the
    code LSB is the mantissa LSB.  Magnitudes above the last grid point map to
    the last code (saturation); beyond the last midpoint everything rounds to
    the last point anyway.
    """
    mids = (grid[:-1] + grid[1:]) / 2.0          # exact: grid points are dyadic
    lo = np.searchsorted(mids, mag, side="left")   # midpoints strictly below
    hi = np.searchsorted(mids, mag, side="right")  # midpoints at or below
    tie = hi != lo                                  # mag sits exactly on mids[lo]
    # at a tie the candidates are codes[lo] and codes[lo + 1]: take the even one
    pick = np.where(tie & (codes[np.minimum(lo, len(codes) - 1)] & 1 == 1), hi, lo)
    return codes[pick]


_E2M1_CODES = np.arange(8, dtype=np.int64)
_E4M3_POS_CODES = np.arange(0x7F, dtype=np.int64)        # 0x00 .. 0x7E, finite, ascending
_E4M3_POS_VALUES = E4M3_TABLE[:0x7F]


def encode_e2m1(values):
    """E2M1 code (uint8 in 0..15) of each float32 value: RNE, satfinite, signed zero."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    if np.any(np.isnan(v)):
        raise ValueError("NaN is outside the quantizer contract")
    mag = np.abs(v)
    code = _rne_encode(mag, E2M1_MAGNITUDES, _E2M1_CODES)
    sign = np.signbit(v)
    return (code | np.where(sign, 8, 0)).astype(np.uint8)


def encode_e4m3(values):
    """E4M3 byte of each float32 value: RNE, satfinite at 448, signed zero."""
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    if np.any(np.isnan(v)):
        raise ValueError("NaN is outside the quantizer contract")
    mag = np.abs(v)
    code = _rne_encode(mag, _E4M3_POS_VALUES, _E4M3_POS_CODES)
    sign = np.signbit(v)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


# ------------------------------------------------------ rounding thresholds

def _thresholds(encoder, mask, n_codes):
    """For magnitude codes 1..n_codes-1: the smallest non-negative float32 (as
    its bit pattern) whose encoding has magnitude code >= that code.  Found
    by bisection over the bit patterns of [0, max finite float32], which
    order like the values; valid because the encoders are monotone in the
    magnitude (RNE onto an ascending grid, then saturation)."""
    lo = np.zeros(n_codes - 1, dtype=np.int64)                # encodes below the code
    hi = np.full(n_codes - 1, 0x7F7FFFFF, dtype=np.int64)    # encodes at or above it
    want = np.arange(1, n_codes, dtype=np.int64)
    top = encoder(np.array([np.float32(3.4028234663852886e38)])) & mask
    assert int(top[0]) == n_codes - 1, "the largest float32 saturates to the largest code"
    while np.any(hi - lo > 1):
        mid = (lo + hi) // 2
        codes = encoder(mid.astype(np.uint32).view(np.float32)).astype(np.int64) & mask
        up = codes >= want
        hi = np.where(up, mid, hi)
        lo = np.where(up, lo, mid)
    return hi.astype(np.uint32)


def e2m1_thresholds():
    """Bit patterns t_1..t_7: a float32 magnitude m encodes to the E2M1
    magnitude code #{i : bits(m) >= t_i} (the encoder as a step function)."""
    return _thresholds(encode_e2m1, 0x7, 8)


def e4m3_thresholds():
    """Bit patterns t_1..t_126 for the E4M3 magnitude codes 0x01..0x7E, as
    e2m1_thresholds (satfinite: everything above 448 is 0x7E)."""
    return _thresholds(encode_e4m3, 0x7F, 127)
