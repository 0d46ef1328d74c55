"""Tolerance rules for comparing the GPU path with the oracle.

Test infrastructure only (see the package docstring).

The acceptance bar: bit-exact quantized codes, scale bytes and gsa bits;
logits within a relative 1e-3; top-k ids equal except where the oracle's keys
are closer than the logit tolerance allows to separate; routing weights within
1e-5 absolute.  How each is applied:

* Logits: |gpu - exact| <= 1e-3 * |exact| + 2**-15 * bound, where bound is the
  dot product of the absolute dequantized operands.  The second term is the
  worst-case float32 summation error over D = 7168 terms (~D * 2**-24 relative
  to the absolute sum, and 2**-15 > 7168 * 2**-24 * 1.5), so cancellation near
  zero cannot fail a correct kernel.
* Keys: each expert n gets a slack tau_n.  Sigmoid mode:
  tau = sigmoid'(l) * tol(l) + 4 ulp(s32) + 2 ulp(key32) (logit error carried
  through the sigmoid, plus a few ulp for float32 exp / divide / add on the
  GPU).  RAW mode: tau = tol(l) + 2 ulp(l32).  A row whose bound is 0 has an
  exactly computable logit (0) on both sides and gets tau = 0, so exact ties
  there must be broken by the lower id.
* Ids: the GPU's ordered list is accepted when no unselected expert is
  clearly better (key - tau above key + tau) than a selected one, no later slot
  is clearly better than an earlier one, and, where both slacks are zero and
  keys are equal, the lower id comes first.  When all keys are separated by
  more than their slack this forces the exact oracle order.
* Weights: recomputed by the oracle from the GPU's ids (identical to the
  oracle's own ids outside near-ties) and compared within 1e-5 absolute.  In
  RAW mode the weight is the logit and the logit tolerance applies.
"""

import numpy as np

from .router import sigmoid64, routed_weights, selection_keys, topk_order

LOGIT_REL = 1e-3
LOGIT_ABS_FRAC = 2.0 ** -15
WEIGHT_ABS = 1e-5


def logit_tolerance(L64, bound64):
    return LOGIT_REL * np.abs(L64) + LOGIT_ABS_FRAC * np.asarray(bound64)


def check_logits(gpu, L64, bound64):
    """Return the number of logits outside tolerance (0 means pass)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - L64)
    return int(np.count_nonzero(~(err <= logit_tolerance(L64, bound64))))


def check_logits_bf16(gpu, L64, bound64):
    """Logits stored as bf16 (round to nearest even of the float32 result):
    the float32 value obeys the logit tolerance, and rounding it to bf16 moves
    it by at most half a bf16 ulp, 2**-8 of its magnitude (8 significant
    bits).  Returns the number of outputs outside |gpu - exact| <=
    tol + 2**-8 * (|exact| + tol)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    tol = logit_tolerance(L64, bound64)
    err = np.abs(gpu - L64)
    return int(np.count_nonzero(~(err <= tol + 2.0 ** -8 * (np.abs(L64) + tol))))


def check_moe_combine(gpu_out, y64, bound64, w):
    """out[t, n] = sum_j w[t, j] y[t, j, n] against the oracle's float64 y:
    each term carries its y's logit tolerance times |w|, and the float32
    chain of k fused multiply-adds adds at most k roundings of the running
    sum (2**-23 of sum_j |w y| is a generous bound).  Returns the number of
    outputs outside it."""
    y64 = np.asarray(y64, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    ref = np.einsum("tj,tjn->tn", w, y64)
    tol = np.einsum("tj,tjn->tn", np.abs(w), logit_tolerance(y64, bound64))
    tol += 2.0 ** -23 * y64.shape[1] * np.einsum("tj,tjn->tn", np.abs(w), np.abs(y64))
    err = np.abs(np.asarray(gpu_out, dtype=np.float64) - ref)
    return int(np.count_nonzero(~(err <= tol)))


def _ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float32))
    return (np.nextafter(v, np.float32(np.inf)) - v).astype(np.float64)


def key_slack(L64, bound64, keys32, bias=None, raw=False):
    """Per-expert slack tau [T, N] on the float32 selection keys."""
    tol = logit_tolerance(L64, bound64)
    exact = np.asarray(bound64) == 0
    if raw:
        tau = tol + 2.0 * _ulp32(keys32)
    else:
        l32 = np.asarray(L64, dtype=np.float64).astype(np.float32)
        s = sigmoid64(l32.astype(np.float64))
        s32 = s.astype(np.float32)
        tau = s * (1.0 - s) * tol + 4.0 * _ulp32(s32) + 2.0 * _ulp32(keys32)
    return np.where(exact, 0.0, tau)


def check_topk(gpu_ids, gpu_w, L64, bound64, keys32, bias=None, routed_scaling=1.0,
               raw=False):
    """Check one call's ids and weights; returns a dict of failure counts.

    ``keys32`` are the oracle's float32 selection keys [T, N].
    """
    gpu_ids = np.asarray(gpu_ids, dtype=np.int64)
    gpu_w = np.asarray(gpu_w, dtype=np.float64)
    keys = np.asarray(keys32, dtype=np.float64)
    T, N = keys.shape
    k = gpu_ids.shape[1]
    tau = key_slack(L64, bound64, keys32, bias, raw)
    res = {"bad_range": 0, "bad_dup": 0, "bad_order": 0, "bad_set": 0,
           "bad_tie": 0, "bad_weight": 0, "exempt_rows": 0}
    exact_oracle = np.lexsort
    for t in range(T):
        g = gpu_ids[t]
        if np.any((g < 0) | (g >= N)):
            res["bad_range"] += 1
            continue
        if len(set(g.tolist())) != k:
            res["bad_dup"] += 1
            continue
        kt, tt = keys[t], tau[t]
        hi = kt[g] + tt[g]          # best each selected key could really be
        lo = kt[g] - tt[g]          # worst
        # order inside the list
        for i in range(k - 1):
            a, b = g[i], g[i + 1]
            if lo[i + 1] > hi[i]:
                res["bad_order"] += 1
            elif tt[a] == 0 and tt[b] == 0 and kt[a] == kt[b] and a > b:
                res["bad_tie"] += 1
        # nothing left out may be clearly better than something selected
        mask = np.ones(N, dtype=bool)
        mask[g] = False
        u = np.nonzero(mask)[0]
        if u.size:
            if np.any(kt[u] - tt[u] > hi.min()):
                res["bad_set"] += 1
            # exact ties across the cut go to the lower id
            last = g[-1]
            if tt[last] == 0:
                tied = u[(tt[u] == 0) & (kt[u] == kt[last]) & (u < last)]
                if tied.size:
                    res["bad_tie"] += 1
        order = exact_oracle((np.arange(N), -kt))[:k]
        if not np.array_equal(order, g):
            res["exempt_rows"] += 1
    # weights, recomputed from the GPU's ids
    ok_rows = np.all((gpu_ids >= 0) & (gpu_ids < N), axis=1)
    ids_safe = np.where(ok_rows[:, None], gpu_ids, 0)
    if raw:
        sel = np.take_along_axis(np.asarray(L64), ids_safe, axis=1)
        selb = np.take_along_axis(np.asarray(bound64), ids_safe, axis=1)
        bad = ~(np.abs(gpu_w - sel) <= logit_tolerance(sel, selb))
    else:
        exp_w = routed_weights(L64, ids_safe, routed_scaling)
        bad = ~(np.abs(gpu_w - exp_w) <= WEIGHT_ABS)
    res["bad_weight"] = int(np.count_nonzero(bad[ok_rows]))
    return res


def topk_ok(res):
    """True when a ``check_topk`` result has no failures."""
    return all(v == 0 for kk, v in res.items() if kk != "exempt_rows")


def candidate_summary(L64, bound64, bias=None, raw=True, top=64):
    """What a head too wide to keep every logit stores per row for
    ``check_topk_candidates``: the ``top`` best outputs by the oracle's float32
    key (ids in oracle order, their float64 logits and bounds) and, over every
    other output, the largest key - slack (``rest_max``; -inf when there is
    none).  Returns (ids int32 [T, top], logits [T, top], bounds [T, top],
    rest_max [T])."""
    L64 = np.asarray(L64, dtype=np.float64)
    bound64 = np.asarray(bound64, dtype=np.float64)
    T, N = L64.shape
    top = min(top, N)
    keys = selection_keys(L64, bias, raw)
    tau = key_slack(L64, bound64, keys, bias, raw)
    ids = topk_order(keys, top)
    rest = np.full(T, -np.inf)
    for t in range(T):
        mask = np.ones(N, bool)
        mask[ids[t]] = False
        if mask.any():
            rest[t] = np.max(keys[t][mask].astype(np.float64) - tau[t][mask])
    return (ids.astype(np.int32), np.take_along_axis(L64, ids.astype(np.int64), 1),
            np.take_along_axis(bound64, ids.astype(np.int64), 1), rest)


def check_topk_candidates(gpu_ids, gpu_w, cand_ids, cand_L, cand_B, rest_max, raw=True,
                          bias=None, routed_scaling=1.0):
    """``check_topk`` for a head too wide to keep every logit: the oracle keeps,
    per row, its best candidates (ids, float64 logits, bounds) and the largest
    key - slack over all other outputs (``rest_max``).  A GPU id outside the
    candidates counts as a set failure."""
    gpu_ids = np.asarray(gpu_ids, dtype=np.int64)
    T, k = gpu_ids.shape
    res = {"bad_range": 0, "bad_dup": 0, "bad_order": 0, "bad_set": 0, "bad_tie": 0,
           "bad_weight": 0, "exempt_rows": 0}
    for t in range(T):
        cid = np.asarray(cand_ids[t], dtype=np.int64)
        pos = {int(c): i for i, c in enumerate(cid)}
        g = gpu_ids[t]
        if len(set(g.tolist())) != k:
            res["bad_dup"] += 1
            continue
        if any(int(e) not in pos for e in g):
            res["bad_set"] += 1
            continue
        idx = np.array([pos[int(e)] for e in g])
        L = np.asarray(cand_L[t], np.float64)[None, :]
        B = np.asarray(cand_B[t], np.float64)[None, :]
        bc = None if bias is None else np.asarray(bias, np.float32)[cid]   # the candidates' bias
        keys = selection_keys(L, bc, raw)
        # the candidate list (stored in oracle order: among equal keys a lower
        # position is a lower id) plus one stand-in for everything else
        sub = check_topk(idx[None, :], np.asarray(gpu_w[t:t + 1]), L, B, keys, bc,
                         routed_scaling, raw)
        tau = key_slack(L, B, keys, bc, raw)[0]
        hi = keys[0][idx].astype(np.float64) + tau[idx]
        if rest_max[t] > hi.min():
            sub["bad_set"] += 1
        for kk in res:
            res[kk] += sub[kk]
    return res
