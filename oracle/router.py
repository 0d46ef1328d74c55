"""The router epilogue ("activation_topk"): scores, biased top-k, routed weights.

Test infrastructure only (see the package docstring).

Source: "nvfp4-megamoe-kernel commit e0f60b9: dsv4/kernels/router/__init__.py",
activation_topk section: one fused pass of six steps over the gate logits of
each token row.  The pages name the kernel and count its steps but do not list
them; the steps taken here are those of the DeepSeek-style router the pages
belong to:

1. score  s = sigmoid(logit)
2. key    key = s + bias[n]          (score-correction bias, selection only)
3. select the k largest keys of the row
4. gather the unbiased scores s of the selected experts
5. renormalise them by their sum
6. multiply by routed_scaling

Readings taken where the pages are silent:

* Selection runs on float32 keys: l32 = fl32(logit), s32 = fl32(sigmoid(l32))
  (the float64 sigmoid rounded once), key = fl32(s32 + bias32).  Deciding the
  integer outcome (which ids) in the kernel's precision is what lets exact ties
  reproduce (an all-zero token row gives logit 0, s = 0.5 exactly, for every
  expert).
* Order of the k outputs: key descending; equal keys go to the lower expert id
  (the "lower expert id wins" rule of the adversarial workload).
* Weights use the unrounded float64 score of the float64 logit:
  w_j = routed_scaling * s(id_j) / sum_j' s(id_j').  No epsilon; a zero sum
  gives zero weights.
* RAW mode (the wide-N head): no sigmoid, bias, renormalisation or scaling;
  key = l32 and the weight is the logit itself.
* No group-limited routing (absent from the pages).
"""

import numpy as np


def sigmoid64(l):
    """Logistic function in float64."""
    l = np.asarray(l, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-l))


def selection_keys(logits64, bias=None, raw=False):
    """float32 keys the top-k is taken on (see the module docstring)."""
    l32 = np.asarray(logits64, dtype=np.float64).astype(np.float32)
    if raw:
        return l32
    s32 = sigmoid64(l32.astype(np.float64)).astype(np.float32)
    if bias is None:
        return s32
    return (s32 + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)


def topk_order(keys, k):
    """Indices of the k best keys per row: key descending, then id ascending."""
    keys = np.asarray(keys)
    T, N = keys.shape
    ids = np.arange(N)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((ids, -keys[t].astype(np.float64)))
        out[t] = order[:k]
    return out


def routed_weights(logits64, ids, routed_scaling=1.0, raw=False):
    """Weights of the given selected ids (float64 [T, k])."""
    L = np.asarray(logits64, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    sel = np.take_along_axis(L, ids, axis=1)
    if raw:
        return sel
    s = sigmoid64(sel)
    tot = s.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        w = np.where(tot > 0, routed_scaling * s / tot, 0.0)
    return w


def route(logits64, bias=None, k=8, routed_scaling=1.0, raw=False):
    """Full epilogue: returns (ids int32 [T, k], weights float64 [T, k], keys float32 [T, N])."""
    keys = selection_keys(logits64, bias, raw)
    ids = topk_order(keys, k)
    w = routed_weights(logits64, ids, routed_scaling, raw)
    return ids, w, keys
