"""NVFP4 quantization of a whole tensor with a runtime global scale.

Test infrastructure only (see the package docstring).

Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py", runtime
gsa section, repeated on "commit df05289: dsv4/layers/grouped_linear.py":
the global activation scale is computed on every call from the activations
themselves, gsa = max(|x|) / (6.0 * 448.0), so that x/gsa never exceeds
2688 = 6 (largest E2M1 magnitude) * 448 (largest E4M3 block scale).  The
zero-sync section of the grouped_linear page flattens all rows of a call into
one (rows, D) tensor and computes one gsa for it.  The format (16-element
blocks along D, one E4M3 scale per block, E2M1 codes, fp32 global scale) is
the NVFP4 layout the same pages use for weights and activations.

Readings taken where the pages are silent (all arithmetic is IEEE float32
round-to-nearest-even, one rounding per operation, no fused multiply-add):

* scope: gsa is per tensor -- one scalar for every row passed in one call.
* gsa = fl32(amax / 2688.0): a single division (6 * 448 = 2688 is exact).
* y = fl32(x / gsa) for every element: the quantity the pages bound by 2688.
* block scale: sy = fl32(max|y over the 16-element block| / 6.0), stored as
  the E4M3 byte encode_e4m3(sy) (RNE, saturating at 448).
* code: q = encode_e2m1(fl32(y / dec(byte))) (RNE, saturating at 6, signed
  zero kept); when byte == 0 (all-zero or underflowing block) every code of
  the block is 0x0.
* amax == 0 gives gsa == 0 and all bytes and codes 0.
* packing: two codes per byte, element 2j in the low nibble, 2j+1 in the high.
* bf16 inputs are widened to float32 exactly (bits << 16) before anything.
"""

import numpy as np

from .formats import encode_e2m1, encode_e4m3, decode_e4m3

BLOCK = 16
#: 6 (largest E2M1 magnitude) * 448 (largest E4M3 scale)
GSA_DIVISOR = np.float32(6.0 * 448.0)


def bf16_bits_to_float32(bits):
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def global_scale(x32):
    """gsa = fl32(max|x| / 2688) over the whole tensor (float32 scalar)."""
    x32 = np.asarray(x32, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    return np.float32(amax / GSA_DIVISOR)


def quantize(x32, gsa=None):
    """Quantize rows of ``x32`` [R, D] (D % 16 == 0) to NVFP4.

    Returns ``(codes, scale_bytes, gsa)``: codes uint8 [R, D] (one 4-bit code
    per element, unpacked), scale_bytes uint8 [R, D/16], gsa float32.  ``gsa``
    may be passed in (used by the invariant tests); by default it is the
    runtime global scale of ``x32``.
    """
    x32 = np.asarray(x32, dtype=np.float32)
    if x32.ndim != 2 or x32.shape[1] % BLOCK:
        raise ValueError("x must be [rows, D] with D a multiple of 16")
    R, D = x32.shape
    if gsa is None:
        gsa = global_scale(x32)
    gsa = np.float32(gsa)
    codes = np.zeros((R, D), dtype=np.uint8)
    sbytes = np.zeros((R, D // BLOCK), dtype=np.uint8)
    if gsa == 0:
        return codes, sbytes, gsa
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        y = (x32 / gsa).astype(np.float32)                       # fl32(x / gsa)
        yb = y.reshape(R, D // BLOCK, BLOCK)
        bmax = np.max(np.abs(yb), axis=2).astype(np.float32)
        sy = (bmax / np.float32(6.0)).astype(np.float32)          # fl32(max|y| / 6)
        sbytes = encode_e4m3(sy)
        s = decode_e4m3(sbytes).astype(np.float32)                # exact
        ratio = (yb / s[:, :, None]).astype(np.float32)           # fl32(y / s)
        zero_block = sbytes == 0
        ratio = np.where(zero_block[:, :, None], np.float32(0.0), ratio)
    q = encode_e2m1(ratio.reshape(R, D))
    q = np.where(np.repeat(zero_block, BLOCK, axis=1), np.uint8(0), q).astype(np.uint8)
    return q, sbytes.astype(np.uint8), gsa


def pack_fp4(codes):
    """[R, D] 4-bit codes -> [R, D/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("D must be even")
    lo = c[..., 0::2] & 0xF
    hi = c[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_fp4(packed):
    """[R, D/2] bytes -> [R, D] 4-bit codes (inverse of ``pack_fp4``)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# -------------------------------------------- 128 x 4 scale-factor tile layout
#
# The block-scaled tensor-core GEMM reads scale bytes in tiles ("atoms") of
# 128 rows x 4 consecutive 16-element blocks = 512 bytes.  Inside an atom, the
# byte for (row r, block c) sits at 16*(r % 32) + 4*((r % 128) // 32) + (c % 4):
# 32 lines of 16 bytes, each line holding rows r, r+32, r+64, r+96.  Atoms are
# stored row-tile-major: atom (r // 128, c // 4) starts at
# ((r // 128) * (KB // 4) + c // 4) * 512, KB = D / 16.  Rows are padded up to a
# multiple of 128 with zero bytes.  This is the 1-D block-scaling layout that
# NVIDIA's cuBLAS documentation gives for 16-element (NVFP4) and 32-element
# (MXFP8) scales.

def sf_tile_bytes(rows, D):
    """Size in bytes of the 128x4-tiled scale buffer for [rows, D]."""
    KB = D // BLOCK
    return ((rows + 127) // 128) * 128 * KB


def sf_tile_offset(r, c, KB):
    """Byte offset of scale (row r, block c) in the 128x4-tiled layout."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // 128) * (KB // 4) + c // 4
    return atom * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def sf_to_tiles(sbytes):
    """Linear [R, KB] scale bytes -> the 128x4-tiled flat buffer (zero padded)."""
    s = np.asarray(sbytes, dtype=np.uint8)
    R, KB = s.shape
    if KB % 4:
        raise ValueError("the tiled layout needs D % 64 == 0")
    out = np.zeros(((R + 127) // 128) * 128 * KB, dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(R), np.arange(KB), indexing="ij")
    out[sf_tile_offset(rr, cc, KB)] = s
    return out


def sf_from_tiles(buf, R, KB):
    """Inverse of ``sf_to_tiles`` for the first R rows."""
    b = np.asarray(buf, dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(R), np.arange(KB), indexing="ij")
    return b[sf_tile_offset(rr, cc, KB)]
