"""Integer and copy steps of the packed layout (TEST INFRASTRUCTURE, oracle).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  Parity for every function here is pinned by brute-force
loops in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def cu_seqlens_from_lengths(lengths: Sequence[int]) -> np.ndarray:
    """Sequence boundaries of a flat packed batch.

    The flat path builds its boundaries from the real token count of every
    request (the text-mask sum plus the image tokens) ("[Perf][Diffusion]
    [Qwen-Image] Replace per-bucket varlen loop with flat varlen attention for
    mixfusion", Key changes).  Sequence b owns flat rows [cu[b], cu[b+1]):
    cu[0] = 0 and cu[b+1] = cu[b] + lengths[b].  int32, length B + 1.
    """
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    for b, n in enumerate(lengths):
        if n < 0:
            raise ValueError("negative sequence length")
        cu[b + 1] = cu[b] + int(n)
    if cu[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length does not fit int32")
    return cu.astype(np.int32)


def pack(padded: np.ndarray, lengths: Sequence[int]) -> np.ndarray:
    """Copy the real tokens of a padded batch into the flat layout.

    ``padded`` is [B, S_max, ...]; the real tokens of request b are its rows
    [0, lengths[b]).  Only real tokens enter the flat tensor; padding never
    does ("feat: Support dynamic batching for heterogeneous diffusion
    requests", How batching works).  Output: [sum(lengths), ...], request b at
    rows [cu[b], cu[b+1]).  A pure copy: values keep their bits.
    """
    cu = cu_seqlens_from_lengths(lengths)
    out = np.empty((int(cu[-1]),) + padded.shape[2:], dtype=padded.dtype)
    for b, n in enumerate(lengths):
        if n > padded.shape[1]:
            raise ValueError("length exceeds S_max")
        out[cu[b]:cu[b + 1]] = padded[b, :n]
    return out


def unpack(flat: np.ndarray, lengths: Sequence[int], padded_out: np.ndarray) -> np.ndarray:
    """Scatter flat rows back to a padded batch (the output split by
    cu_seqlens, "[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop
    with flat varlen attention for mixfusion", Key changes).

    Rows [0, lengths[b]) of slot b of a copy of ``padded_out`` receive flat rows
    [cu[b], cu[b+1]); every padding row keeps the value it had.
    """
    cu = cu_seqlens_from_lengths(lengths)
    out = padded_out.copy()
    for b, n in enumerate(lengths):
        out[b, :n] = flat[cu[b]:cu[b + 1]]
    return out


def work_order(lengths_q: Sequence[int], lengths_k: Sequence[int], H: int,
               tile_m: int) -> List[Tuple[int, int, int]]:
    """Length-ordered list of attention work items (sequence, head, q_tile).

    The per-bucket loop left bubbles and a mixed batch is dominated by its
    largest request ("[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen
    loop ...", Purpose; "feat: Support dynamic batching ...", online serving
    evaluation), so the longest work goes first: sequences are taken in order
    of key length, longest first, equal lengths by lower index; within a
    sequence heads in order, within a head q-tiles in order.  A sequence with
    no queries has no items; one with queries but no keys has items (their
    rows are all zero).
    """
    B = len(lengths_q)
    order = sorted(range(B), key=lambda b: (-int(lengths_k[b]), b))
    items = []
    for b in order:
        n_tiles = (int(lengths_q[b]) + tile_m - 1) // tile_m
        for h in range(H):
            for t in range(n_tiles):
                items.append((b, h, t))
    return items
