"""Segment-aware unpack with per-request CFG combine (TEST INFRASTRUCTURE, oracle).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  Pinned by ``tests/test_oracle_cfg.py``.

A CFG-active request r runs as two packed sequences: the positive one (its
text, then its image tokens) and the negative one (the negative text, then
the same number of image tokens).  After the per-request split, the image
span of each request is combined as

    out = negative + true_cfg_scale * (positive - negative)

with the scale kept per request ("feat: Support dynamic batching for
heterogeneous diffusion requests", CFG behavior; AttentionSegment for the
text / image / negative-text spans).  A request without CFG (no negative
sequence) gets its positive image rows unchanged.

``cfg_normalize`` is named on the page as a per-request value but not
defined there.  Reading taken: when set, every combined token row is
rescaled to the L2 norm (over the row's channels) of its positive row,
out *= ||positive|| / ||out|| (rows whose combined norm is zero stay zero).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .attention import to_f64
from .packing import cu_seqlens_from_lengths


def cfg_combine(flat, lengths: Sequence[int], img_off: Sequence[int],
                pos_seq: Sequence[int], neg_seq: Sequence[int],
                cfg_scale: Sequence[float], cfg_normalize: Sequence[int],
                img_max: int, out_init: Optional[np.ndarray] = None) -> np.ndarray:
    """Scatter each request's image span and combine it with its negative.

    flat: [T, C] packed rows (any float dtype; computed in float64).
    lengths: per packed sequence; img_off[b]: first image row of sequence b
    (its text length).  Request r's positive sequence is pos_seq[r] and its
    negative one neg_seq[r] (< 0: none).  Returns float64 [R, img_max, C]:
    rows [0, n_img(r)) of slot r hold the result; the other rows keep
    out_init (zeros if not given).
    """
    x = to_f64(flat)
    cu = cu_seqlens_from_lengths(lengths)
    R, C = len(pos_seq), x.shape[1]
    out = np.zeros((R, img_max, C)) if out_init is None else to_f64(out_init).copy()
    for r in range(R):
        p = pos_seq[r]
        p0 = cu[p] + img_off[p]
        n_img = int(cu[p + 1] - p0)
        pos = x[p0:p0 + n_img]
        if neg_seq[r] < 0:
            comb = pos.copy()
        else:
            q = neg_seq[r]
            q0 = cu[q] + img_off[q]
            if int(cu[q + 1] - q0) != n_img:
                raise ValueError("positive and negative image spans differ in length")
            neg = x[q0:q0 + n_img]
            comb = neg + cfg_scale[r] * (pos - neg)
            if cfg_normalize[r]:
                pn = np.sqrt((pos * pos).sum(axis=1, keepdims=True))
                cn = np.sqrt((comb * comb).sum(axis=1, keepdims=True))
                comb = np.where(cn > 0, comb * (pn / np.where(cn > 0, cn, 1.0)), 0.0)
        out[r, :n_img] = comb
    return out
