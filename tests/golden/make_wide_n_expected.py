"""Write tests/golden/wide_n_expected.npz: the oracle's answer for the wide-N
raw-logit head (T=32 tokens, D=7168, N=129280 outputs).

Quantizing the 0.93 G-element weight on the CPU takes minutes, so the parity
test reads these stored oracle values instead of recomputing them.  This
script calls only ``oracle/`` and the seeded ``workloads`` generator; nothing
comes from the CUDA path.  Stored per token: the 64 best outputs by float32
logit (ids, float64 logits, the |x|.|w| bounds) and, over all other outputs,
the largest logit less its slack (``oracle.compare.candidate_summary``) --
enough to check any GPU top-k with k <= 16 under the oracle's comparison
rules (``oracle.compare.check_topk_candidates``).  Checksums of the generated inputs let
the test detect a generator that produces different numbers.

Run:  python tests/golden/make_wide_n_expected.py
"""

import hashlib
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402
from oracle import quantize as Q, gemm, compare  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "wide_n_expected.npz")
TOP = 64
CHUNK = 16384


def input_digest(w):
    """sha256 over x and the first/last weight chunks (generator drift check)."""
    h = hashlib.sha256()
    h.update(WL.make_x(w).tobytes())
    last = None
    for n0, c in WL.iter_w(w, rows_per_chunk=CHUNK):
        if n0 == 0:
            h.update(c.tobytes())
        last = c
    h.update(last.tobytes())
    return h.hexdigest()


def main():
    w = WL.WORKLOADS["wide_n"]
    x32 = WL.bf16_bits_to_float32(WL.make_x(w))
    # pass 1: the weight's global scale
    amax = np.float32(0.0)
    for _, c in WL.iter_w(w, rows_per_chunk=CHUNK):
        amax = max(amax, np.max(np.abs(WL.bf16_bits_to_float32(c))))
    wg = Q.global_scale(np.array([[amax] + [0.0] * 15], np.float32))
    # pass 2: logits of every output
    xq, xs, xg = Q.quantize(x32)
    L = np.empty((w.T, w.N))
    B = np.empty((w.T, w.N))
    for n0, c in WL.iter_w(w, rows_per_chunk=CHUNK):
        wq, ws, _ = Q.quantize(WL.bf16_bits_to_float32(c), gsa=wg)
        L[:, n0:n0 + c.shape[0]], B[:, n0:n0 + c.shape[0]] = gemm.logits(xq, xs, xg, wq, ws, wg)
        print("rows", n0 + c.shape[0], flush=True)
    ids, cand_L, cand_B, rest = compare.candidate_summary(L, B, None, raw=True, top=TOP)
    np.savez_compressed(
        OUT, ids=ids, logits=cand_L, bounds=cand_B, rest_max=rest, x_gsa=np.float32(xg), w_gsa=wg,
        digest=np.array(input_digest(w)))
    print("wrote", OUT)


if __name__ == "__main__":
    main()
