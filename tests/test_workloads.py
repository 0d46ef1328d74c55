"""The seeded input generators: determinism, chunking, bf16 rounding, structure."""

import numpy as np

import workloads as WL


def test_bf16_rounding_rne():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 1e4], np.float32)
    b = WL.float32_to_bf16_bits(v)
    back = WL.bf16_bits_to_float32(b)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins;
    # 1+3*2^-8 is a tie between 1+2^-7 and 1+2^-6: even is 1+2^-6
    assert back.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 9984.0]


def test_deterministic_and_chunk_invariant():
    w = WL.WORKLOADS["tiny"]
    assert np.array_equal(WL.make_x(w), WL.make_x(w))
    full = WL.make_w(w)
    parts = np.concatenate([c for _, c in WL.iter_w(w, rows_per_chunk=5)])
    assert np.array_equal(full, parts)


def test_shapes_and_structure():
    d = WL.WORKLOADS["decode"].with_T(8)
    x = WL.x_as_float32(WL.make_x(d), d)
    assert x.shape == (8, 7168)
    big = np.abs(x).max(axis=0) > 20
    assert 60 <= big.sum() <= 72                    # the 72 outlier channels stand out
    a = WL.WORKLOADS["adversarial"].with_T(16)
    xa = WL.x_as_float32(WL.make_x(a), a)
    assert not xa[1::4].any()                       # class 1: all-zero rows
    assert np.all(np.sort(np.abs(xa[2::4]), axis=1)[:, -1] == 9984.0)   # class 2: one huge element
    assert np.all(xa[3::4] == xa[3::4, :1])         # class 3: constant rows
    assert np.all(WL.make_bias(a) == 0)
    assert WL.make_bias(WL.WORKLOADS["wide_n"]) is None
