"""Pins for the oracle's E2M1 / E4M3 tables and encoders (CPU only).

The decode tables are checked against the printed format tables under
tests/golden and against ml_dtypes (an independent implementation, when it is
installed); the encoders against ml_dtypes over a broad sweep of float32 bit
patterns, against a brute-force nearest-value search, and on every midpoint and
its float32 neighbours.
"""

import os

import numpy as np
import pytest

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                a, b = line.split()
                rows.append((a, float(b)))
    return rows


def test_e2m1_decode_matches_printed_table():
    for code, val in _read_table("e2m1_table.txt"):
        got = formats.decode_e2m1(int(code))
        assert got == val and np.signbit(got) == np.signbit(val), code


def test_e4m3_decode_matches_printed_points():
    for code, val in _read_table("e4m3_points.txt"):
        got = formats.decode_e4m3(int(code, 16))
        assert got == val and np.signbit(got) == np.signbit(val), code


def test_e4m3_decode_structure():
    t = formats.E4M3_TABLE
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.count_nonzero(np.isnan(t)) == 2
    finite = t[:0x7F]
    assert np.all(np.diff(finite) > 0)               # codes ascend with value
    assert finite.max() == 448.0 == formats.E4M3_MAX
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])
    # subnormal spacing 2**-9, first normal 2**-6
    assert np.allclose(np.diff(finite[:9]), 2.0 ** -9)
    assert finite[8] == 2.0 ** -6


def test_decode_tables_against_ml_dtypes():
    mld = pytest.importorskip("ml_dtypes")
    c4 = np.arange(16, dtype=np.uint8)
    ref4 = c4.view(mld.float4_e2m1fn) if hasattr(mld, "float4_e2m1fn") else None
    if ref4 is not None:
        # float4 arrays are stored one code per byte
        ref = np.array([float(v) for v in ref4.astype(np.float32)])
        assert np.array_equal(ref, formats.decode_e2m1(c4))
    c8 = np.arange(256, dtype=np.uint8)
    ref8 = c8.view(mld.float8_e4m3fn).astype(np.float64)
    ours = formats.decode_e4m3(c8)
    assert np.array_equal(np.isnan(ref8), np.isnan(ours))
    m = ~np.isnan(ours)
    assert np.array_equal(ref8[m], ours[m])


def _brute_force(v, grid, codes):
    """Nearest grid value, ties to the even code; independent of searchsorted."""
    out = np.empty(v.shape, dtype=np.int64)
    for i, x in enumerate(np.abs(v.astype(np.float64))):
        x = min(x, grid[-1])            # saturation: beyond the top, the top value
        d = np.abs(grid - x)
        best = np.nonzero(d == d.min())[0]
        if best.size > 1:
            best = best[(codes[best] & 1) == 0]
        out[i] = codes[best[0]]
    return out


def _interesting_points(grid):
    mids = (grid[:-1] + grid[1:]) / 2
    pts = np.concatenate([grid, mids]).astype(np.float32)
    up = np.nextafter(pts, np.float32(np.inf))
    dn = np.nextafter(pts, np.float32(-np.inf))
    allp = np.concatenate([pts, up, dn, [grid[-1] * 1.5, 1e30, np.float32(1e-45)]]).astype(np.float32)
    allp = allp[allp >= 0]
    return np.concatenate([allp, -allp]).astype(np.float32)


def test_e2m1_encoder_brute_force_and_midpoints():
    grid = formats.E2M1_MAGNITUDES
    v = _interesting_points(grid)
    rng = np.random.default_rng(1)
    v = np.concatenate([v, rng.uniform(-8, 8, 4000).astype(np.float32)])
    codes = formats.encode_e2m1(v)
    ref = _brute_force(v, grid, np.arange(8))
    ref = ref | np.where(np.signbit(v), 8, 0)
    assert np.array_equal(codes, ref)
    # explicit tie rule: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    assert formats.decode_e2m1(formats.encode_e2m1(ties)).tolist() == [0, 1, 1, 2, 2, 4, 4]
    # saturation and signed zero
    assert formats.encode_e2m1(np.float32([7.0, 1e30, -1e30, -0.1, -0.0])).tolist() == [7, 7, 15, 8, 8]


def test_e4m3_encoder_brute_force_and_midpoints():
    grid = formats.E4M3_TABLE[:0x7F]
    v = _interesting_points(grid)
    codes = formats.encode_e4m3(v)
    ref = _brute_force(v, grid, np.arange(0x7F)) | np.where(np.signbit(v), 0x80, 0)
    assert np.array_equal(codes, ref)
    assert formats.encode_e4m3(np.float32([2.0 ** -10, 1.5 * 2.0 ** -10, 464.0, 1e9])).tolist() == \
        [0x00, 0x01, 0x7E, 0x7E]


def test_roundtrip_all_codes():
    c4 = np.arange(16)
    assert np.array_equal(formats.encode_e2m1(formats.decode_e2m1(c4).astype(np.float32)), c4)
    c8 = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(formats.encode_e4m3(formats.decode_e4m3(c8).astype(np.float32)), c8)


def _bit_sweep(stride, offset=0):
    bits = np.arange(offset, 2 ** 32, stride, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    return v[~np.isnan(v)]


def test_encoders_against_ml_dtypes_bit_sweep():
    """Every 4099th float32 bit pattern (about 1M values, all exponents)."""
    mld = pytest.importorskip("ml_dtypes")
    v = _bit_sweep(4099)
    if hasattr(mld, "float4_e2m1fn"):
        ref4 = v.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF
        assert np.array_equal(formats.encode_e2m1(v), ref4)
    small = v[np.abs(v) <= 464.0]          # beyond that ml_dtypes gives NaN, we saturate
    ref8 = small.astype(mld.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(formats.encode_e4m3(small), ref8)
    big = v[np.abs(v) > 464.0]
    assert np.all((formats.encode_e4m3(big) & 0x7F) == 0x7E)


def test_rounding_thresholds_are_the_ties_to_even_midpoints():
    """The encoders as step functions: threshold i (the smallest float32 with
    magnitude code >= i) is the midpoint of the values of codes i-1 and i
    when code i is even (a tie goes to it), else the next float32 above the
    midpoint -- from the decode tables, which are pinned to the printed
    format tables above.  Catches a tie sent the wrong way, a missing
    subnormal step or a wrong saturation point."""
    F = formats
    for thresholds, decode, n in ((F.e2m1_thresholds(), F.decode_e2m1, 8),
                                  (F.e4m3_thresholds(), F.decode_e4m3, 127)):
        vals = np.asarray(decode(np.arange(n)), dtype=np.float64)
        assert len(thresholds) == n - 1
        for i in range(1, n):
            mid = np.float32((vals[i - 1] + vals[i]) / 2)     # exact: midpoints are float32 values
            assert float(mid) == (vals[i - 1] + vals[i]) / 2
            exp = mid if i % 2 == 0 else np.nextafter(mid, np.float32(np.inf))
            assert thresholds[i - 1] == np.array([exp], dtype=np.float32).view(np.uint32)[0], (n, i)
