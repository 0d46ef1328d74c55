"""The whole router call on the CPU: quantize W and x, logits, epilogue.

Test infrastructure only (see the package docstring).

Order of the steps follows the pages' two-kernel path ("nvfp4-megamoe-kernel
commit 04cf8ca: dsv4/layers/router.py", NVFP4 gate section): the gate weight
is quantized once at load with its own runtime global scale, the activations
are quantized per call with theirs, the NVFP4 gate GEMM produces the logits and
the activation_topk epilogue turns them into expert ids and weights.
"""

import numpy as np

from . import quantize as Q, gemm, router


def pack_weight(W32):
    """Load-time weight quantization: (codes [N, D], scale bytes [N, D/16], w_gsa)."""
    return Q.quantize(np.asarray(W32, dtype=np.float32))


def run(x32, W32=None, bias=None, k=8, routed_scaling=1.0, raw=False, packed_w=None):
    """Route one batch.  Returns a dict with every intermediate."""
    if packed_w is None:
        packed_w = pack_weight(W32)
    wq, ws, wg = packed_w
    xq, xs, xg = Q.quantize(np.asarray(x32, dtype=np.float32))
    L, B = gemm.logits(xq, xs, xg, wq, ws, wg)
    ids, w, keys = router.route(L, bias, k, routed_scaling, raw)
    return {"x_codes": xq, "x_sf": xs, "x_gsa": xg, "w_codes": wq, "w_sf": ws, "w_gsa": wg,
            "logits": L, "bound": B, "ids": ids, "weights": w, "keys": keys}
