"""Pins for the segment-aware unpack + CFG combine oracle: the page's formula
on its own scales, brute force, closed forms and the packed-equals-alone
invariant."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _layout():
    # two CFG requests (sequences 0/1 and 2/3) and one without CFG (sequence 4)
    text = [5, 3, 7, 2, 4]
    img = [6, 6, 4, 4, 3]
    lengths = [t + i for t, i in zip(text, img)]
    return lengths, text, [0, 2, 4], [1, 3, -1], img


def _flat(lengths, C, seed):
    return np.random.default_rng(seed).standard_normal((sum(lengths), C))


def test_golden_formula_with_page_scales():
    with open(os.path.join(GOLDEN, "cfg_combine.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        flat = np.array([[c["positive"]], [c["negative"]]])
        out = oracle.cfg_combine(flat, [1, 1], [0, 0], [0], [1], [c["true_cfg_scale"]], [0], 1)
        assert out[0, 0, 0] == c["combined"]


def test_brute_force():
    lengths, text, pos, neg, img = _layout()
    C = 5
    flat = _flat(lengths, C, 1)
    scales, norm = [2.0, 7.0, 3.0], [0, 1, 0]
    out = oracle.cfg_combine(flat, lengths, text, pos, neg, scales, norm, 8)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    for r in range(3):
        p = pos[r]
        for i in range(img[p]):
            pr = flat[starts[p] + text[p] + i]
            if neg[r] < 0:
                want = pr
            else:
                nr = flat[starts[neg[r]] + text[neg[r]] + i]
                want = [nr[c] + scales[r] * (pr[c] - nr[c]) for c in range(C)]
                if norm[r]:
                    pn = sum(v * v for v in pr) ** 0.5
                    cn = sum(v * v for v in want) ** 0.5
                    want = [v * pn / cn for v in want]
            np.testing.assert_allclose(out[r, i], want, rtol=0, atol=1e-12)
        assert (out[r, img[p]:] == 0).all()


def test_closed_forms():
    lengths, text, pos, neg, img = _layout()
    flat = _flat(lengths, 4, 2)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    one = oracle.cfg_combine(flat, lengths, text, pos, neg, [1.0, 1.0, 1.0], [0, 0, 0], 8)
    zero = oracle.cfg_combine(flat, lengths, text, pos, neg, [0.0, 0.0, 0.0], [0, 0, 0], 8)
    for r in range(2):
        p, q = pos[r], neg[r]
        n = img[p]
        # scale 1 returns the positive rows, scale 0 the negative rows
        np.testing.assert_allclose(one[r, :n], flat[starts[p] + text[p]:starts[p] + text[p] + n])
        np.testing.assert_allclose(zero[r, :n], flat[starts[q] + text[q]:starts[q] + text[q] + n])
    # normalised output keeps the positive row norms
    nrm = oracle.cfg_combine(flat, lengths, text, pos, neg, [5.0, 5.0, 5.0], [1, 1, 1], 8)
    for r in range(2):
        p = pos[r]
        n = img[p]
        prow = flat[starts[p] + text[p]:starts[p] + text[p] + n]
        np.testing.assert_allclose(np.linalg.norm(nrm[r, :n], axis=1),
                                   np.linalg.norm(prow, axis=1), rtol=1e-12)


def test_linearity_and_identical_branches():
    lengths, text, pos, neg, img = _layout()
    flat = _flat(lengths, 3, 3)
    a = oracle.cfg_combine(flat, lengths, text, pos, neg, [2.0, 4.0, 1.0], [0, 0, 0], 8)
    b = oracle.cfg_combine(flat, lengths, text, pos, neg, [3.0, 5.0, 1.0], [0, 0, 0], 8)
    c = oracle.cfg_combine(flat, lengths, text, pos, neg, [4.0, 6.0, 1.0], [0, 0, 0], 8)
    np.testing.assert_allclose(b - a, c - b, atol=1e-12)   # affine in the scale
    # identical positive and negative image rows: any scale returns them
    flat2 = flat.copy()
    starts = np.concatenate([[0], np.cumsum(lengths)])
    flat2[starts[1] + text[1]:starts[2]] = flat2[starts[0] + text[0]:starts[1]]
    d = oracle.cfg_combine(flat2, lengths, text, pos, neg, [9.0, 1.0, 1.0], [0, 0, 0], 8)
    np.testing.assert_allclose(d[0, :img[0]], flat2[starts[0] + text[0]:starts[1]], atol=1e-12)


def test_request_alone_equals_packed():
    lengths, text, pos, neg, img = _layout()
    flat = _flat(lengths, 4, 4)
    packed = oracle.cfg_combine(flat, lengths, text, pos, neg, [2.0, 7.0, 3.0], [1, 0, 0], 8)
    starts = np.concatenate([[0], np.cumsum(lengths)])
    alone = oracle.cfg_combine(flat[starts[2]:starts[4]], lengths[2:4], text[2:4], [0], [1],
                               [7.0], [0], 8)
    np.testing.assert_array_equal(packed[1], alone[0])


def test_mismatched_image_spans_rejected():
    with pytest.raises(ValueError):
        oracle.cfg_combine(np.zeros((7, 2)), [4, 3], [1, 1], [0], [1], [2.0], [0], 4)
