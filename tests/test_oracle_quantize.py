"""Pins for the oracle quantizer (CPU only).

* gsa: closed form on exact cases (amax = 2688 * 2**a gives gsa = 2**a) and the
  page's constants; amax = 0.
* invariants: x/gsa <= 2688 (the pages' bound), the block holding amax gets
  the 448 scale, byte 0 <=> sy <= 2**-10 with all codes 0, each code is within
  half an E2M1 step of the clipped ratio, signs follow the input.
* exact round trip: inputs built on the grid quantize without error.
* independent check of the scale bytes against ml_dtypes when installed.
* nibble packing and the 128x4 scale tile layout: bijection, hand-checked
  offsets, inverse.
"""

import os

import numpy as np
import pytest

from oracle import formats, quantize as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _page_constants():
    out = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def test_page_constants():
    c = _page_constants()
    assert c["e4m3_max"] == formats.E4M3_MAX == formats.decode_e4m3(formats.E4M3_MAX_CODE)
    assert c["e2m1_max"] == formats.E2M1_MAX == formats.decode_e2m1(7)
    assert c["gsa_divisor"] == c["e4m3_max"] * c["e2m1_max"] == float(Q.GSA_DIVISOR)


@pytest.mark.parametrize("a", [-20, -3, 0, 1, 7])
def test_gsa_closed_form(a):
    x = np.zeros((3, 64), dtype=np.float32)
    x[1, 17] = -np.float32(2688.0 * 2.0 ** a)
    x[2, 5] = np.float32(1000.0 * 2.0 ** a)
    assert Q.global_scale(x) == np.float32(2.0 ** a)


def test_gsa_is_one_ieee_division():
    rng = np.random.default_rng(3)
    for amax in rng.uniform(1e-3, 1e3, 200).astype(np.float32):
        x = np.array([[amax] + [0.0] * 15], dtype=np.float32)
        g = Q.global_scale(x)
        # correctly rounded quotient: the float32 nearest the exact amax/2688
        exact = np.float64(amax) / 2688.0
        lo, hi = np.nextafter(g, np.float32(0)), np.nextafter(g, np.float32(np.inf))
        assert abs(np.float64(g) - exact) <= min(abs(np.float64(lo) - exact), abs(np.float64(hi) - exact))


def test_zero_tensor():
    x = np.zeros((2, 32), dtype=np.float32)
    q, s, g = Q.quantize(x)
    assert g == 0 and not q.any() and not s.any()


def _random_x(seed=0, R=37, D=256):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, D)).astype(np.float32)
    x *= np.exp(rng.standard_normal((R, 1)) * 2).astype(np.float32)
    x[3, :16] = 0.0                              # an all-zero block
    x[5, 16:32] *= np.float32(1e-7)              # a block that underflows the scale
    x[7, 40] = np.float32(1e3)                   # a large outlier
    return x


def test_invariants_random():
    x = _random_x()
    q, sb, gsa = Q.quantize(x)
    y = (x / gsa).astype(np.float32)
    # the pages' bound: x / gsa <= 2688 (up to the rounding of gsa itself)
    assert np.max(np.abs(y)) <= np.nextafter(np.float32(2688.0), np.float32(np.inf))
    # the block holding amax has the largest scale byte
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sb[r, c // 16] == 0x7E
    s = formats.decode_e4m3(sb)
    yb = y.reshape(x.shape[0], -1, 16)
    sy = (np.max(np.abs(yb), axis=2) / np.float32(6.0)).astype(np.float32)
    zero = sb == 0
    assert np.all(sy[zero] <= 2.0 ** -10)
    assert np.all(sy[~zero] > 2.0 ** -10)
    qb = q.reshape(x.shape[0], -1, 16)
    assert not qb[zero].any()
    # every code lies within half a grid step of the clipped ratio
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (yb / s[:, :, None].astype(np.float32)).astype(np.float64)
    deq = formats.decode_e2m1(qb)
    clipped = np.clip(ratio, -6.0, 6.0)
    half_step = np.where(np.abs(clipped) <= 2.0, 0.25, np.where(np.abs(clipped) <= 4.0, 0.5, 1.0))
    nz = ~zero[:, :, None] & np.ones_like(qb, dtype=bool)
    assert np.all(np.abs(deq - clipped)[nz] <= half_step[nz])
    # sign of every nonzero code follows the input
    sign_bit = (qb & 8) != 0
    assert np.all(sign_bit[nz & (yb != 0)] == (yb < 0)[nz & (yb != 0)])


def test_scale_bytes_against_ml_dtypes():
    mld = pytest.importorskip("ml_dtypes")
    x = _random_x(seed=4)
    q, sb, gsa = Q.quantize(x)
    y = (x / gsa).astype(np.float32).reshape(x.shape[0], -1, 16)
    sy = (np.max(np.abs(y), axis=2) / np.float32(6.0)).astype(np.float32)
    ref = sy.astype(mld.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(ref, sb)
    s = sb.view(mld.float8_e4m3fn).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (y / s[:, :, None]).astype(np.float32)
    ref_q = ratio.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF
    ref_q = np.where((sb == 0)[:, :, None], 0, ref_q).reshape(q.shape)
    assert np.array_equal(ref_q, q)


def test_exact_grid_roundtrip():
    """Values e2m1 * 2**b * gsa with a 6 in every block quantize exactly."""
    rng = np.random.default_rng(7)
    R, D, a = 5, 128, -4
    gsa = 2.0 ** a
    vals = formats.decode_e2m1(rng.integers(0, 16, (R, D)))
    vals[:, ::16] = 6.0 * rng.choice([-1, 1], (R, D // 16))      # block max = 6 * scale
    b = rng.integers(-6, 6, (R, D // 16))                          # scale = 2**b, exact in E4M3
    b[0, 0] = 6                                                    # 6 * 2**6 * gsa... amax block
    x = (vals * np.repeat(2.0 ** b, 16, axis=1) * gsa).astype(np.float32)
    # amax = 6 * 64 * gsa; with gsa chosen as amax / 2688 this is not 2**a, so pass gsa in
    q, sb, g = Q.quantize(x, gsa=np.float32(gsa))
    assert np.array_equal(formats.decode_e4m3(sb), 2.0 ** b)
    assert np.array_equal(formats.decode_e2m1(q), vals)


def test_pack_unpack():
    rng = np.random.default_rng(2)
    c = rng.integers(0, 16, (3, 10)).astype(np.uint8)
    p = Q.pack_fp4(c)
    assert p.shape == (3, 5)
    assert p[0, 0] == (c[0, 0] | (c[0, 1] << 4))
    assert np.array_equal(Q.unpack_fp4(p), c)


def test_sf_tile_layout_hand_checked():
    KB = 8
    off = lambda r, c: int(Q.sf_tile_offset(r, c, KB))
    assert off(0, 0) == 0
    assert off(0, 1) == 1 and off(0, 3) == 3
    assert off(1, 0) == 16 and off(31, 0) == 496
    assert off(32, 0) == 4 and off(64, 2) == 10 and off(96, 3) == 15
    assert off(0, 4) == 512                       # next atom along K
    assert off(128, 0) == 1024                    # next row tile (KB/4 = 2 atoms per row tile)
    assert off(129, 5) == 1024 + 512 + 16 + 1


@pytest.mark.parametrize("R,KB", [(1, 4), (130, 8), (256, 4), (77, 12)])
def test_sf_tile_layout_bijection(R, KB):
    Rp = ((R + 127) // 128) * 128
    rr, cc = np.meshgrid(np.arange(Rp), np.arange(KB), indexing="ij")
    offs = Q.sf_tile_offset(rr, cc, KB).ravel()
    assert np.array_equal(np.sort(offs), np.arange(Rp * KB))
    rng = np.random.default_rng(R)
    s = rng.integers(0, 256, (R, KB)).astype(np.uint8)
    buf = Q.sf_to_tiles(s)
    assert buf.size == Q.sf_tile_bytes(R, KB * 16)
    assert np.array_equal(Q.sf_from_tiles(buf, R, KB), s)
    pad = np.ones(buf.size, dtype=bool)
    pad[Q.sf_tile_offset(rr[:R], cc[:R], KB).ravel()] = False
    assert not buf[pad].any()
