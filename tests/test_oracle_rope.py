"""Pins for the request-local RoPE oracle: brute force from the rotation
definition, and properties of rotary embeddings that fail for a wrong pair
convention, sign or frequency."""
import math

import numpy as np
import pytest

import oracle


def _x(T, H, D, seed):
    return np.random.default_rng(seed).standard_normal((T, H, D))


def test_positions_request_local():
    pos = oracle.rope_positions([3, 0, 2], pos_offset=[5, 9, 0], total=7)
    assert pos.tolist() == [5, 6, 7, 0, 1, -1, -1]
    assert oracle.rope_positions([2, 2]).tolist() == [0, 1, 0, 1]


def test_brute_force():
    x = _x(4, 2, 6, 1)
    pos = np.array([0, 3, 17, -1])
    got = oracle.rope(x, pos, 100.0)
    for t in range(4):
        for h in range(2):
            for i in range(3):
                a, b = x[t, h, 2 * i], x[t, h, 2 * i + 1]
                if pos[t] < 0:
                    want = (a, b)
                else:
                    ang = pos[t] * 100.0 ** (-2 * i / 6)
                    want = (a * math.cos(ang) - b * math.sin(ang),
                            a * math.sin(ang) + b * math.cos(ang))
                assert abs(got[t, h, 2 * i] - want[0]) < 1e-12
                assert abs(got[t, h, 2 * i + 1] - want[1]) < 1e-12


def test_position_zero_is_identity_and_norms_kept():
    x = _x(5, 3, 16, 2)
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(5, dtype=np.int64), 1e4), x)
    y = oracle.rope(x, np.arange(5) * 1000, 1e4)
    pair = lambda z: np.hypot(z[..., 0::2], z[..., 1::2])
    np.testing.assert_allclose(pair(y), pair(x), rtol=1e-12)


def test_relative_position_property():
    # <R(p) q, R(p') k> depends only on p - p'
    q, k = _x(1, 1, 32, 3), _x(1, 1, 32, 4)
    dots = []
    for p in (0, 7, 300, 12345):
        rq = oracle.rope(q, np.array([p + 11]), 1e4)
        rk = oracle.rope(k, np.array([p]), 1e4)
        dots.append(float((rq * rk).sum()))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)
    # and it does depend on the offset
    rq = oracle.rope(q, np.array([12]), 1e4)
    rk = oracle.rope(k, np.array([0]), 1e4)
    assert abs(float((rq * rk).sum()) - dots[0]) > 1e-6


def test_rotation_composes():
    # rotating by p then by p' (two calls) equals rotating by p + p'
    x = _x(3, 2, 8, 5)
    a = oracle.rope(oracle.rope(x, np.array([4, 50, 900]), 10.0), np.array([3, 7, 11]), 10.0)
    b = oracle.rope(x, np.array([7, 57, 911]), 10.0)
    np.testing.assert_allclose(a, b, atol=1e-10)


def test_packed_equals_alone():
    L = [5, 9, 2]
    x = _x(sum(L), 2, 8, 6)
    packed = oracle.rope(x, oracle.rope_positions(L, [0, 3, 1]), 1e4)
    alone = oracle.rope(x[5:14], oracle.rope_positions([9], [3]), 1e4)
    np.testing.assert_array_equal(packed[5:14], alone)
