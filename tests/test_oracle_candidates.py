"""Pins of the wide-head comparison (``oracle.compare.candidate_summary`` and
``check_topk_candidates``) on CPU-sized heads, where every logit can still be
kept: the candidate checker must reach the same verdict as the full checker
(``check_topk``, itself pinned by planted mistakes in
test_oracle_gemm_router.py) on the oracle's answer and on perturbed answers,
and must catch the mistakes a wrong stored summary or a wrong GPU list would
make.  The parity test of the N = 129280 raw head relies on this checker."""

import numpy as np
import pytest

from oracle import gemm, router, compare


def _wide_case(seed, T=10, N=4096):
    rng = np.random.default_rng(seed)
    xq = rng.integers(0, 16, (T, 64))
    xs = rng.integers(0x30, 0x40, (T, 4))
    wq = rng.integers(0, 16, (N, 64))
    ws = rng.integers(0x30, 0x40, (N, 4))
    xq[0] = 0                                        # all-zero token row: every logit exactly 0
    L, B = gemm.logits(xq, xs, 0.01, wq, ws, 0.02)
    return L, B


def _weights(L, ids, raw, scale):
    return router.routed_weights(L, ids, scale, raw)


def _both(ids, L, B, summ, bias, raw, scale):
    """(full verdict, candidate verdict) for the GPU-like answer `ids`."""
    w = _weights(L, ids, raw, scale)
    keys = router.selection_keys(L, bias, raw)
    full = compare.check_topk(ids, w, L, B, keys, bias, scale, raw)
    cand = compare.check_topk_candidates(ids, w, *summ, raw=raw, bias=bias, routed_scaling=scale)
    return full, cand


@pytest.mark.parametrize("raw", [True, False])
@pytest.mark.parametrize("k", [1, 8])
def test_candidate_checker_agrees_with_full_checker(raw, k):
    L, B = _wide_case(5 + k + raw)
    T, N = L.shape
    bias = None if raw else np.random.default_rng(1).uniform(-0.05, 0.05, N).astype(np.float32)
    scale = 1.0 if raw else 2.5
    summ = compare.candidate_summary(L, B, bias, raw, top=64)
    keys = router.selection_keys(L, bias, raw)
    best = router.topk_order(keys, 64)
    assert np.array_equal(summ[0], best)
    rng = np.random.default_rng(7)
    verdicts = []
    for trial in range(40):
        ids = best[:, :k].copy()
        kind = trial % 5
        for t in range(T):
            if kind == 1 and k > 1:                          # adjacent swap
                i = rng.integers(0, k - 1)
                ids[t, [i, i + 1]] = ids[t, [i + 1, i]]
            elif kind == 2:                                  # a lower-ranked candidate in some slot
                ids[t, rng.integers(0, k)] = best[t, rng.integers(k, 64)]
            elif kind == 3:                                  # the (k+1)-th replaces the k-th
                ids[t, k - 1] = best[t, k]
        full, cand = _both(ids, L, B, summ, bias, raw, scale)
        assert compare.topk_ok(full) == compare.topk_ok(cand), (trial, full, cand)
        assert full["exempt_rows"] == cand["exempt_rows"]
        verdicts.append(compare.topk_ok(full))
    assert any(verdicts) and not all(verdicts)              # both outcomes were exercised


def test_candidate_checker_planted_mistakes():
    L, B = _wide_case(11)
    T, N = L.shape
    k = 8
    summ = compare.candidate_summary(L, B, None, True, top=64)
    ids_c, L_c, B_c, rest = summ
    good = ids_c[:, :k].copy()
    w = _weights(L, good, True, 1.0)
    assert compare.topk_ok(compare.check_topk_candidates(good, w, *summ, raw=True))
    r = 3
    # a swapped pair of well separated outputs
    bad = good.copy()
    bad[r, [0, 1]] = bad[r, [1, 0]]
    res = compare.check_topk_candidates(bad, _weights(L, bad, True, 1.0), *summ, raw=True)
    assert res["bad_order"] > 0
    # an id outside the stored candidates
    outside = np.setdiff1d(np.arange(N), ids_c[r])[0]
    bad = good.copy()
    bad[r, k - 1] = outside
    res = compare.check_topk_candidates(bad, _weights(L, bad, True, 1.0), *summ, raw=True)
    assert res["bad_set"] > 0
    # a stored rest_max that beats the k-th selection: something outside the
    # candidates is clearly better than a selected output
    rest_bad = rest.copy()
    rest_bad[r] = np.float32(L_c[r, k - 1]) + 1.0
    res = compare.check_topk_candidates(good, w, ids_c, L_c, B_c, rest_bad, raw=True)
    assert res["bad_set"] == 1
    # a summary that left the true best output out of its candidates: the
    # answer drawn from those candidates fails through rest_max
    keys = router.selection_keys(L, None, True)
    tau = compare.key_slack(L, B, keys, None, True)
    order = router.topk_order(keys, 65)
    wrong_ids = order[:, 1:65].astype(np.int32)
    wrong_rest = np.array([np.max(np.delete(keys[t].astype(np.float64) - tau[t], order[t, 1:65]))
                           for t in range(T)])
    wrong = (wrong_ids, np.take_along_axis(L, wrong_ids.astype(np.int64), 1),
             np.take_along_axis(B, wrong_ids.astype(np.int64), 1), wrong_rest)
    ans = wrong_ids[:, :k]
    res = compare.check_topk_candidates(ans, _weights(L, ans, True, 1.0), *wrong, raw=True)
    assert res["bad_set"] == T - 1                          # every row but the all-zero one
    # a weight (the raw logit) off by 1 percent
    wb = w.copy()
    wb[r, 2] = wb[r, 2] * 1.01 + 1e-3
    res = compare.check_topk_candidates(good, wb, *summ, raw=True)
    assert res["bad_weight"] == 1


def test_candidate_checker_accepts_near_tie_swap_and_exact_ties():
    L, B = _wide_case(13)
    L = L.copy()
    r = 4
    keys = router.selection_keys(L, None, True)
    o = router.topk_order(keys, 3)[r]
    L[r, o[2]] = L[r, o[1]] * (1 + 1e-7)                  # outputs 2 and 3 of row r: a near tie
    summ = compare.candidate_summary(L, B, None, True, top=64)
    ans = summ[0][:, :8].copy()
    i, j = list(ans[r]).index(o[1]), list(ans[r]).index(o[2])
    ans[r, [i, j]] = ans[r, [j, i]]
    res = compare.check_topk_candidates(ans, _weights(L, ans, True, 1.0), *summ, raw=True)
    assert compare.topk_ok(res) and res["exempt_rows"] == 1, res
    # the all-zero row: logits exactly 0, candidates are ids 0..63, and the
    # lowest ids must win the exact tie
    assert summ[0][0].tolist() == list(range(64)) and np.isneginf(summ[3][0]) is np.False_
    tie = summ[0][:, :8].copy()
    tie[0] = [1, 0, 2, 3, 4, 5, 6, 7]
    res = compare.check_topk_candidates(tie, _weights(L, tie, True, 1.0), *summ, raw=True)
    assert res["bad_tie"] == 1
