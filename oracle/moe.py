"""The NVFP4 grouped expert GEMM that consumes the router's output, and the
weighted combine of the expert outputs.

Test infrastructure only (see the package docstring).

Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py"
-- the grouped NVFP4 linear (one weight per group; the groups' rows flattened
into one (G*T, D) activation tensor quantized with ONE runtime global scale
in one launch; expert offsets computed on the GPU) -- and the runtime-gsa
section of "commit 04cf8ca: dsv4/layers/router.py", which applies the same
runtime gsa to Nvfp4GroupedLinear and Nvfp4MoE.

Readings taken where the pages are silent:

* grouping: the router's out_ids [T, k] assign token t's slot j to expert
  ids[t, j]; every (t, j) pair is one row of the grouped GEMM, so a token
  appears in k groups;
* activation scale: one global scale over all rows of the call.  Every token
  is routed k >= 1 times, so the flattened (T*k, D) tensor and x itself have
  the same max|x|: gsa = max|x| / 2688 over x, and each token's codes and
  block scales are its ordinary NVFP4 quantization (identical in all of its
  k rows);
* weights: expert e has its own packed weight [N, D] with its own global
  scale w_gsa[e] (each expert quantized at load time like any NVFP4 linear);
* y[t, j, n] = sum_i xq[t, i] * wq_e[n, i] with e = ids[t, j], both operands
  dequantized (code x block scale x global scale) -- the plain dot product,
  computed exactly enough in float64;
* combine: out[t, n] = sum_j w[t, j] * y[t, j, n] (the routing weights of
  the router's out_w), summed over j in order.
"""

import numpy as np

from . import quantize as Q, gemm


def expert_segments(ids, n_experts):
    """Per-expert row counts of the grouping (the GPU computes the same
    counts; order inside an expert's group is immaterial to any output)."""
    ids = np.asarray(ids, dtype=np.int64)
    return np.bincount(ids.ravel(), minlength=n_experts)


def grouped_gemm(x32, ids, packed_experts):
    """y [T, k, N] float64 and its |x|.|w| bound, for the routed pairs.

    packed_experts: list over experts of (codes [N, D], scale bytes [N, D/16],
    w_gsa) as returned by oracle.quantize.quantize for each expert weight.
    """
    x32 = np.asarray(x32, dtype=np.float32)
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    xq, xs, xg = Q.quantize(x32)
    N = np.asarray(packed_experts[0][0]).shape[0]
    y = np.zeros((T, k, N))
    bound = np.zeros((T, k, N))
    for e in np.unique(ids):
        rows = np.argwhere(ids == e)                    # (t, j) pairs of expert e
        t = rows[:, 0]
        wq, ws, wg = packed_experts[e]
        L, B = gemm.logits(xq[t], xs[t], xg, wq, ws, wg)
        y[rows[:, 0], rows[:, 1]] = L
        bound[rows[:, 0], rows[:, 1]] = B
    return y, bound


def combine(y, w):
    """out [T, N] = sum_j w[t, j] * y[t, j, :] in float64, j in order."""
    y = np.asarray(y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    out = np.zeros((y.shape[0], y.shape[2]))
    for j in range(y.shape[1]):
        out += w[:, j:j + 1] * y[:, j]
    return out
