"""Pins for the oracle's logits, epilogue and comparison rules (CPU only).

* logits: exact rational brute force (Python Fractions over the decoded
  codes) on tiny random operands, so a dropped scale, a transposed operand or
  a wrong global-scale product fails; plus the |x|.|w| bound.
* epilogue: brute-force full sort on tiny inputs; closed forms of the sigmoid;
  all-equal rows pick ids 0..k-1 with equal weights; weights sum to
  routed_scaling; RAW k=1 is the first argmax.
* comparison rules: planted mistakes in a copy of the oracle's own outputs
  (a swapped pair, a wrong id, a perturbed weight, a broken exact tie) must be
  caught, and legitimate near-tie permutations must pass.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, quantize as Q, gemm, router, compare


def _frac_e2m1(c):
    mag = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
           Fraction(4), Fraction(6)][c & 7]
    return -mag if c & 8 else mag


def _frac_e4m3(b):
    e, m = (b >> 3) & 0xF, b & 7
    v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if b & 0x80 else v


@pytest.mark.parametrize("seed", [0, 1])
def test_logits_exact_rational(seed):
    rng = np.random.default_rng(seed)
    T, N, D = 3, 5, 64
    xq = rng.integers(0, 16, (T, D))
    wq = rng.integers(0, 16, (N, D))
    xs = rng.integers(0, 0x7F, (T, D // 16))
    ws = rng.integers(0, 0x7F, (N, D // 16))
    gx, gw = np.float32(0.0123), np.float32(3.5e-4)
    L, B = gemm.logits(xq, xs, gx, wq, ws, gw)
    for t in range(T):
        for n in range(N):
            acc = Fraction(0)
            accabs = Fraction(0)
            for i in range(D):
                a = _frac_e2m1(int(xq[t, i])) * _frac_e4m3(int(xs[t, i // 16]))
                b = _frac_e2m1(int(wq[n, i])) * _frac_e4m3(int(ws[n, i // 16]))
                acc += a * b
                accabs += abs(a) * abs(b)
            g = Fraction(float(gx)) * Fraction(float(gw))
            exact = acc * g
            assert abs(Fraction(L[t, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
            assert abs(Fraction(B[t, n]) - accabs * g) <= accabs * g * Fraction(1, 2 ** 50)


def test_logits_chunking_invariant():
    rng = np.random.default_rng(5)
    xq = rng.integers(0, 16, (2, 32))
    wq = rng.integers(0, 16, (37, 32))
    xs = rng.integers(0, 0x7F, (2, 2))
    ws = rng.integers(0, 0x7F, (37, 2))
    a, _ = gemm.logits(xq, xs, 1.0, wq, ws, 1.0)
    b, _ = gemm.logits(xq, xs, 1.0, wq, ws, 1.0, n_chunk=7)
    assert np.array_equal(a, b)


def test_sigmoid_closed_forms():
    assert router.sigmoid64(0.0) == 0.5
    assert abs(router.sigmoid64(np.log(3.0)) - 0.75) < 1e-16
    x = np.linspace(-30, 30, 101)
    assert np.allclose(router.sigmoid64(-x), 1 - router.sigmoid64(x), rtol=0, atol=3e-16)
    assert router.sigmoid64(-1000.0) == 0.0 and router.sigmoid64(1000.0) == 1.0


def _brute_topk(keys, k):
    out = []
    for row in keys:
        order = sorted(range(len(row)), key=lambda n: (-float(row[n]), n))
        out.append(order[:k])
    return np.array(out)


@pytest.mark.parametrize("N,k", [(16, 2), (16, 1), (33, 8), (64, 8), (9, 9)])
def test_topk_brute_force(N, k):
    rng = np.random.default_rng(N * 100 + k)
    L = rng.standard_normal((20, N)) * 3
    L[3] = 0.0                                       # all-equal row
    L[4, ::2] = L[4, 1::2][: len(L[4, ::2])] if N % 2 == 0 else L[4, ::2]   # pairwise ties
    bias = rng.uniform(-0.1, 0.1, N).astype(np.float32)
    keys = router.selection_keys(L, bias)
    ids = router.topk_order(keys, k)
    assert np.array_equal(ids, _brute_topk(keys, k))


def test_epilogue_special_rows():
    N, k, scale = 16, 4, 2.5
    L = np.zeros((2, N))
    L[1] = np.linspace(-1, 1, N)
    ids, w, keys = router.route(L, np.zeros(N, np.float32), k, scale)
    assert ids[0].tolist() == [0, 1, 2, 3]
    assert np.allclose(w[0], scale / k)
    assert ids[1].tolist() == [15, 14, 13, 12]
    assert abs(w[1].sum() - scale) < 1e-12


def test_raw_mode_is_argmax():
    rng = np.random.default_rng(9)
    L = rng.standard_normal((6, 50))
    L[2, 7] = L[2, 30] = 10.0                        # tie: first index wins
    ids, w, keys = router.route(L, None, 1, 1.0, raw=True)
    assert np.array_equal(ids[:, 0], np.argmax(L.astype(np.float32), axis=1))
    assert ids[2, 0] == 7
    assert np.array_equal(w[:, 0], L[np.arange(6), ids[:, 0]])


def test_bias_changes_selection_not_weights():
    L = np.array([[1.0, 0.9, -3.0]])
    bias = np.array([0.0, 0.0, 1.0], np.float32)
    ids, w, _ = router.route(L, bias, 1, 1.0)
    assert ids[0, 0] == 2                            # biased key wins
    assert w[0, 0] == 1.0                            # renormalised unbiased score of one expert


# ------------------------------------------------------------ comparison rules

def _case(seed=0, T=12, N=32, k=4):
    rng = np.random.default_rng(seed)
    xq = rng.integers(0, 16, (T, 64))
    xs = rng.integers(0x30, 0x40, (T, 4))
    wq = rng.integers(0, 16, (N, 64))
    ws = rng.integers(0x30, 0x40, (N, 4))
    xq[0] = 0                                        # an all-zero token row: exact ties
    L, B = gemm.logits(xq, xs, 0.01, wq, ws, 0.02)
    bias = np.zeros(N, np.float32)
    ids, w, keys = router.route(L, bias, k, 2.5)
    return L, B, bias, ids, w, keys


def test_compare_accepts_oracle_and_rejects_planted_mistakes():
    L, B, bias, ids, w, keys = _case()
    ok = compare.check_topk(ids, w.astype(np.float32), L, B, keys, bias, 2.5)
    assert compare.topk_ok(ok), ok
    assert compare.check_logits(L.astype(np.float32), L, B) == 0
    # swapped pair in a row with well separated keys
    bad = ids.copy()
    r = 5
    bad[r, [0, 1]] = bad[r, [1, 0]]
    res = compare.check_topk(bad, w, L, B, keys, bias, 2.5)
    assert res["bad_order"] > 0
    # an id replaced by a clearly worse expert
    bad = ids.copy()
    worst = int(np.argmin(keys[r]))
    bad[r, 0] = worst
    assert compare.check_topk(bad, w, L, B, keys, bias, 2.5)["bad_set"] > 0
    # exact tie in the all-zero row broken the wrong way
    bad = ids.copy()
    bad[0] = [1, 0, 2, 3]
    assert compare.check_topk(bad, w, L, B, keys, bias, 2.5)["bad_tie"] > 0
    bad[0] = [0, 1, 2, 5]
    assert compare.check_topk(bad, w, L, B, keys, bias, 2.5)["bad_tie"] > 0
    # a weight off by 1e-4
    ww = w.copy()
    ww[3, 2] += 1e-4
    assert compare.check_topk(ids, ww, L, B, keys, bias, 2.5)["bad_weight"] == 1
    # a logit off by 1 percent
    Lb = L.astype(np.float32).copy()
    Lb[4, 4] = Lb[4, 4] * 1.01 + 1e-3
    assert compare.check_logits(Lb, L, B) == 1


def test_compare_accepts_near_tie_swap():
    L, B, bias, ids, w, keys = _case(seed=3)
    r = 6
    L = L.copy()
    a, b = ids[r, 1], ids[r, 2]
    L[r, b] = L[r, a] * (1 + 1e-7)                   # make two experts a near tie
    ids2, w2, keys2 = router.route(L, bias, ids.shape[1], 2.5)
    swapped = ids2.copy()
    i = list(ids2[r]).index(a)
    j = list(ids2[r]).index(b)
    swapped[r, [i, j]] = swapped[r, [j, i]]
    w_sw = router.routed_weights(L, swapped, 2.5)
    res = compare.check_topk(swapped, w_sw, L, B, keys2, bias, 2.5)
    assert compare.topk_ok(res) and res["exempt_rows"] == 1, res


def test_compare_bf16_logits_rule():
    """bf16-stored logits: the oracle's float64 logits rounded to bf16 (an
    independent RNE rounding, workloads.float32_to_bf16_bits) pass; a value
    two bf16 ulps off fails; the float32 rule alone would reject bf16 output."""
    import workloads as WL
    L, B, *_ = _case(seed=5)
    bits = WL.float32_to_bf16_bits(L.astype(np.float32))
    g = WL.bf16_bits_to_float32(bits).astype(np.float64)
    assert compare.check_logits_bf16(g, L, B) == 0
    assert compare.check_logits(g, L, B) > 0
    bad = bits.copy()
    r, c = np.unravel_index(np.argmax(np.abs(L)), L.shape)
    bad[r, c] = np.uint16(int(bad[r, c]) + 2)
    assert compare.check_logits_bf16(WL.bf16_bits_to_float32(bad), L, B) == 1
