"""Pins of the grouped expert GEMM oracle (oracle/moe.py): each routed pair's
row against an exact rational dot product of the dequantized operands, the
grouping against a pair-by-pair computation, the one-scale-for-all-rows
reading, and the combine against its closed forms."""

from fractions import Fraction

import numpy as np

from oracle import quantize as Q, gemm, formats, moe


def _experts(rng, E, N, D, scale=0.05):
    return [Q.quantize((rng.standard_normal((N, D)) * scale).astype(np.float32)) for _ in range(E)]


def test_grouped_rows_match_pairwise_and_exact_rationals():
    rng = np.random.default_rng(3)
    T, D, N, E, k = 6, 64, 8, 5, 3
    x = rng.standard_normal((T, D)).astype(np.float32)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    ex = _experts(rng, E, N, D)
    y, B = moe.grouped_gemm(x, ids, ex)
    xq, xs, xg = Q.quantize(x)
    for t in range(T):
        for j in range(k):
            wq, ws, wg = ex[ids[t, j]]
            L, Bt = gemm.logits(xq[t:t + 1], xs[t:t + 1], xg, wq, ws, wg)
            assert np.array_equal(y[t, j], L[0]) and np.array_equal(B[t, j], Bt[0])
    # one pair exactly: sum over i of e2m1 * e4m3 products times both global scales
    t, j, n = 4, 1, 3
    wq, ws, wg = ex[ids[t, j]]
    acc = Fraction(0)
    for i in range(D):
        a = Fraction(float(formats.decode_e2m1(xq[t, i]))) * Fraction(float(formats.decode_e4m3(xs[t, i // 16])))
        b = Fraction(float(formats.decode_e2m1(wq[n, i]))) * Fraction(float(formats.decode_e4m3(ws[n, i // 16])))
        acc += a * b
    exact = acc * Fraction(float(xg)) * Fraction(float(wg))
    assert abs(Fraction(y[t, j, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def test_one_global_scale_over_the_routed_rows():
    """The flattened (T*k, D) tensor of routed rows has the same max|x| as x
    (every token is routed k >= 1 times): the reading 'quantize x once' and
    'quantize the flattened groups once' give identical codes per row."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((9, 128)) * np.exp(rng.standard_normal((9, 1)))).astype(np.float32)
    k = 4
    flat = np.repeat(x, k, axis=0)
    assert Q.global_scale(flat) == Q.global_scale(x)
    q1, s1, _ = Q.quantize(x)
    q2, s2, _ = Q.quantize(flat)
    assert np.array_equal(np.repeat(q1, k, axis=0), q2) and np.array_equal(np.repeat(s1, k, axis=0), s2)


def test_grouping_detects_a_wrong_expert_and_counts():
    rng = np.random.default_rng(5)
    T, D, N, E, k = 5, 64, 4, 4, 2
    x = rng.standard_normal((T, D)).astype(np.float32)
    ids = np.array([[0, 1], [2, 3], [1, 0], [3, 2], [0, 3]])
    ex = _experts(rng, E, N, D)
    y, _ = moe.grouped_gemm(x, ids, ex)
    bad = ids.copy()
    bad[2, 0] = 2
    y2, _ = moe.grouped_gemm(x, bad, ex)
    assert not np.array_equal(y[2, 0], y2[2, 0]) and np.array_equal(y[3], y2[3])
    assert moe.expert_segments(ids, E).tolist() == [3, 2, 2, 3]


def test_combine_closed_forms():
    rng = np.random.default_rng(6)
    y = rng.standard_normal((7, 3, 5))
    onehot = np.zeros((7, 3))
    onehot[:, 1] = 1.0
    assert np.array_equal(moe.combine(y, onehot), y[:, 1])
    w = rng.random((7, 3))
    assert np.allclose(moe.combine(y, w), np.einsum("tj,tjn->tn", w, y), rtol=0, atol=1e-12)
    same = np.repeat(y[:, :1], 3, axis=1)
    assert np.allclose(moe.combine(same, np.full((7, 3), 1 / 3)), y[:, 0], atol=1e-12)


def test_compare_moe_combine_rule():
    """The combine tolerance accepts the float32 fused multiply-add chain of
    the oracle's own rows (an independent float32 evaluation) and rejects a
    term dropped or a weight misapplied."""
    from oracle import compare
    rng = np.random.default_rng(8)
    T, D, N, E, k = 6, 64, 16, 4, 3
    x = rng.standard_normal((T, D)).astype(np.float32)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    ex = _experts(rng, E, N, D)
    y, B = moe.grouped_gemm(x, ids, ex)
    w = rng.random((T, k)).astype(np.float32)
    acc = np.zeros((T, N), np.float32)
    for j in range(k):
        acc = (acc + w[:, j:j + 1] * y[:, j].astype(np.float32)).astype(np.float32)
    assert compare.check_moe_combine(acc, y, B, w) == 0
    dropped = np.zeros((T, N), np.float32)
    for j in range(k - 1):
        dropped = (dropped + w[:, j:j + 1] * y[:, j].astype(np.float32)).astype(np.float32)
    assert compare.check_moe_combine(dropped, y, B, w) > 0
    swapped = (acc + (w[:, 1:2] - w[:, 0:1]) * (y[:, 0] - y[:, 1]).astype(np.float32)).astype(np.float32)
    assert compare.check_moe_combine(swapped, y, B, w) > 0
