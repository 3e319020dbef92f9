"""Rotary position embedding with request-local positions (TEST INFRASTRUCTURE,
oracle).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  Pinned by ``tests/test_oracle_rope.py``.

The dynamic path rebuilds RoPE per request from request-local state: the
model never infers positions from packed global offsets, so a request gets
the same RoPE alone or inside a mixed batch ("feat: Support dynamic batching
for heterogeneous diffusion requests", Main changes and Correctness model;
"[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop ...", the RoPE
of the packed path moved into a fused operator).  The pages give no formula,
so the plainest reading is taken: the rotary embedding of Su et al.
(RoFormer) on interleaved pairs,

    theta_i = base ** (-2 i / D),   i = 0 .. D/2 - 1
    (x_2i, x_2i+1) -> (x_2i cos(p theta_i) - x_2i+1 sin(p theta_i),
                       x_2i sin(p theta_i) + x_2i+1 cos(p theta_i))

applied to every head of q and k, where token j of packed sequence b has the
request-local position p = pos_offset[b] + j.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .attention import to_f64
from .packing import cu_seqlens_from_lengths


def rope_positions(lengths: Sequence[int], pos_offset: Optional[Sequence[int]] = None,
                   total: Optional[int] = None) -> np.ndarray:
    """Request-local position of every packed row (-1 for rows past the last
    sequence): row cu[b] + j of sequence b sits at pos_offset[b] + j."""
    cu = cu_seqlens_from_lengths(lengths)
    T = int(cu[-1]) if total is None else total
    pos = np.full(T, -1, dtype=np.int64)
    for b, L in enumerate(lengths):
        off = 0 if pos_offset is None else int(pos_offset[b])
        pos[cu[b]:cu[b] + L] = off + np.arange(L)
    return pos


def rope(x, positions: np.ndarray, base: float) -> np.ndarray:
    """x [T, H, D] rotated per row by its position (rows with position -1 are
    returned unchanged).  float64."""
    x = to_f64(x)
    T, H, D = x.shape
    i = np.arange(D // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / D)
    out = x.copy()
    live = positions >= 0
    ang = positions[live, None].astype(np.float64) * theta[None, :]   # [T', D/2]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    xe, xo = x[live, :, 0::2], x[live, :, 1::2]
    out[live, :, 0::2] = xe * c - xo * s
    out[live, :, 1::2] = xe * s + xo * c
    return out
