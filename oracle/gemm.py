"""Gate logits of two NVFP4 operands, computed exactly enough in float64.

Test infrastructure only (see the package docstring).

Source: "nvfp4-megamoe-kernel commit 04cf8ca: dsv4/layers/router.py", NVFP4
gate section: the router's gate projection x . W_gate^T runs as an NVFP4
block-scaled tensor-core GEMM (Nvfp4Linear) on quantized activations and
quantized gate weights.

The plain definition: each operand dequantizes to
    value[r, i] = e2m1(code[r, i]) * e4m3(scale[r, i // 16]) * gsa,
and the logit is the dot product of the dequantized rows,
    logit[t, n] = sum_i xq[t, i] * wq[n, i].
Every e2m1 * e4m3 product is exact in float64, so the only error here is the
float64 summation over D (relative ~1e-16), far below the GPU's float32.

``abs_logits`` is the same product with |.| on both operands; the parity
tolerance uses it to bound cancellation.
"""

import numpy as np

from .formats import decode_e2m1, decode_e4m3

BLOCK = 16


def dequantize(codes, scale_bytes):
    """float64 [R, D] = e2m1(codes) * e4m3(scale) (the gsa factor is left out)."""
    c = np.asarray(codes)
    s = np.asarray(scale_bytes)
    vals = decode_e2m1(c)
    scl = np.repeat(decode_e4m3(s), BLOCK, axis=1)
    return vals * scl


def logits(x_codes, x_sf, x_gsa, w_codes, w_sf, w_gsa, n_chunk=65536):
    """float64 logits [T, N] and the matching |x| . |w| bound [T, N].

    Computed as (A @ B^T) * (gsa_x * gsa_w) with A, B the dequantized operands
    without their global scales; the scalar product gsa_x * gsa_w is exact in
    float64.  N is processed in chunks to bound memory.
    """
    A = dequantize(x_codes, x_sf)
    g = np.float64(np.float32(x_gsa)) * np.float64(np.float32(w_gsa))
    T = A.shape[0]
    N = np.asarray(w_codes).shape[0]
    out = np.empty((T, N), dtype=np.float64)
    bound = np.empty((T, N), dtype=np.float64)
    Aabs = np.abs(A)
    for n0 in range(0, N, n_chunk):
        n1 = min(N, n0 + n_chunk)
        B = dequantize(w_codes[n0:n1], w_sf[n0:n1])
        out[:, n0:n1] = (A @ B.T) * g
        bound[:, n0:n1] = (Aabs @ np.abs(B).T) * g
    return out, bound
