"""The hash router of the first MoE layers: experts looked up by token id.

Test infrastructure only (see the package docstring).

Source: "nvfp4-megamoe-kernel commit df05289: dsv4/layers/grouped_linear.py",
hash-router item: the first layers route without a gate GEMM; ``tid2eid`` is
an int32 table from a token id to its experts, and routing is one lookup.

Readings taken where the page is silent:

* the table is [vocab, k] int32: row ``tid`` holds the k expert ids of token
  id ``tid``, in the order they are emitted (slot j of the output is column j
  of the row);
* weights: with no gate there are no scores, so the router's renormalise and
  scale steps see k equal scores; each selected expert gets
  fl32(routed_scaling / k) (one float32 division);
* inputs outside the table: a token id outside [0, vocab) gives ids -1 and
  weights 0 for its whole row; a table entry outside [0, n_experts) gives id
  -1 and weight 0 in its slot (the other slots keep their weights).
"""

import numpy as np


def route(token_ids, tid2eid, n_experts, routed_scaling=1.0):
    """ids int32 [T, k] and weights float32 [T, k] for the token ids [T]."""
    tids = np.asarray(token_ids, dtype=np.int64)
    table = np.asarray(tid2eid, dtype=np.int64)
    vocab, k = table.shape
    T = tids.shape[0]
    w_each = np.float32(np.float32(routed_scaling) / np.float32(k))
    ids = np.full((T, k), -1, dtype=np.int32)
    w = np.zeros((T, k), dtype=np.float32)
    for t in range(T):
        tid = tids[t]
        if tid < 0 or tid >= vocab:
            continue
        for j in range(k):
            e = table[tid, j]
            if 0 <= e < n_experts:
                ids[t, j] = e
                w[t, j] = w_each
    return ids, w
