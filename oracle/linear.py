"""Packed-M linear layer (TEST INFRASTRUCTURE, oracle).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  Pinned by ``tests/test_oracle_linear.py``.

The packed path runs its projections (QKV, output) as GEMMs over the flat
[total_tokens, C] activations of every request at once, and the batched
result equals the per-request result bit for bit because those GEMMs are
batch invariant ("feat: Support dynamic batching for heterogeneous diffusion
requests", packed varlen step batching: Summary, Setup (Determinism) and
Notes, item 1).  The pages give no formula; the plainest reading is the
linear layer of the model's projections:

    y[m, n] = sum_k x[m, k] * w[n, k] + bias[n]

with w stored [out_features, in_features].  Each output row is a function of
its own input row alone, which is the property the packed path relies on.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .attention import to_f64


def linear(x, w, bias=None) -> np.ndarray:
    """x [M, K], w [N, K], bias [N] or None -> float64 [M, N]."""
    x, w = to_f64(x), to_f64(w)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x must be [M, K] and w [N, K]")
    y = x @ w.T
    if bias is not None:
        b = to_f64(bias)
        if b.shape != (w.shape[0],):
            raise ValueError("bias must be [N]")
        y = y + b[None, :]
    return y


def linear_rows(x, w, bias, rows) -> np.ndarray:
    """Rows `rows` of linear(x, w, bias), computed one row at a time (for
    sampled checks of large problems)."""
    x = to_f64(x)
    return linear(x[np.asarray(rows, dtype=np.int64)], w, bias)


def linear_flops(M: int, N: int, K: int) -> int:
    """2 M N K: one multiply and one add per (m, n, k)."""
    return 2 * int(M) * int(N) * int(K)
