"""Pins for the linear-layer oracle: a hand-worked example, the operand
orientation, the bias axis, closed forms and brute force, chosen so that a
transposed weight, a bias added along the wrong axis, a dropped term or a
row that leaks into another row fails."""
import numpy as np
import pytest

import oracle


def test_hand_worked_example():
    # y = x w^T + b with w stored [out, in]:
    #   row 0: [1*1 + 2*0 + 3*0, 1*0 + 2*0 + 3*1, 1*1 + 2*1 + 3*1] + b
    #   row 1: [4, 6, 15] + b
    x = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    w = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0], [1.0, 1.0, 1.0]])
    b = np.array([10.0, 20.0, 30.0])
    assert oracle.linear(x, w).tolist() == [[1.0, 3.0, 6.0], [4.0, 6.0, 15.0]]
    assert oracle.linear(x, w, b).tolist() == [[11.0, 23.0, 36.0], [14.0, 26.0, 45.0]]


def test_orientation_rejects_transposed_weight():
    x = np.ones((4, 3))
    with pytest.raises(ValueError):
        oracle.linear(x, np.ones((3, 5)))          # [K, N] instead of [N, K]
    assert oracle.linear(x, np.ones((5, 3))).shape == (4, 5)


def test_identity_and_permutation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 6))
    assert np.array_equal(oracle.linear(x, np.eye(6)), x)
    perm = [3, 0, 5, 1, 4, 2]
    assert np.array_equal(oracle.linear(x, np.eye(6)[perm]), x[:, perm])


def test_brute_force_integers():
    rng = np.random.default_rng(1)
    x = rng.integers(-5, 6, size=(5, 9)).astype(np.float64)
    w = rng.integers(-5, 6, size=(4, 9)).astype(np.float64)
    b = rng.integers(-5, 6, size=4).astype(np.float64)
    got = oracle.linear(x, w, b)
    for m in range(5):
        for n in range(4):
            acc = int(b[n])
            for k in range(9):
                acc += int(x[m, k]) * int(w[n, k])
            assert got[m, n] == acc


def test_rank_one_closed_form():
    rng = np.random.default_rng(2)
    u, v = rng.standard_normal(8), rng.standard_normal(5)
    x = rng.standard_normal((3, 5))
    got = oracle.linear(x, np.outer(u, v))
    assert np.allclose(got, np.outer(x @ v, u), rtol=1e-13, atol=1e-13)


def test_rows_are_independent():
    # the property the packed path relies on: a row's output depends on that
    # row only, so packed rows equal the rows computed alone, in any order
    # (here up to float64 rounding: the library matmul may sum a lone row in
    # another order than a block of rows)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 16))
    w = rng.standard_normal((12, 16))
    b = rng.standard_normal(12)
    full = oracle.linear(x, w, b)
    for m in range(10):
        assert np.allclose(oracle.linear(x[m:m + 1], w, b)[0], full[m], rtol=1e-13, atol=1e-13)
    rows = [9, 2, 5]
    assert np.allclose(oracle.linear_rows(x, w, b, rows), full[rows], rtol=1e-13, atol=1e-13)
    # changing one row changes that row only
    x2 = x.copy()
    x2[4] += 1.0
    diff = np.abs(oracle.linear(x2, w, b) - full).max(axis=1)
    assert diff[4] > 1e-3 and np.all(np.delete(diff, 4) < 1e-12)


def test_flops():
    assert oracle.linear_flops(3, 4, 5) == 120
