"""Plain float64 attention under explicit boolean masks (TEST INFRASTRUCTURE, oracle).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.

The flat varlen path computes ordinary (exact) softmax attention, only with
request boundaries taken from cu_seqlens, and the block-window path computes
the same result as dense attention under the block-difference mask ("[Perf]
[Model] Use block-sparse attention in Qwen2.5-Omni Token2Wav DiT", Change:
"the math is the same as the dense masked SDPA").  So the oracle is the plain
definition written out:

    s_j   = scale * <q_i, k_j>              for every key j with allowed[i, j]
    p_j   = exp(s_j - max s) / sum exp(s - max s)
    out_i = sum_j p_j * v_j

in float64 on the exact values of the bf16 inputs.  A query with no allowed
key gets an all-zero row (fully masked positions contribute nothing).

Readings taken where the pages are silent: attention is non-causal inside a
sequence (joint text+image attention is bidirectional); the default scale is
1/sqrt(D); query and key lengths may differ per sequence.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .packing import cu_seqlens_from_lengths


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a (bf16/fp16/fp32) torch tensor or numpy array."""
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     allowed: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one head under an explicit boolean mask.

    q [M, D], k [N, D], v [N, Dv] (float64), allowed [M, N] bool -> [M, Dv].
    Rows with no allowed key are zero.
    """
    s = (q @ k.T) * scale
    s = np.where(allowed, s, -np.inf)
    row_max = s.max(axis=1, keepdims=True) if s.shape[1] else np.full((s.shape[0], 1), -np.inf)
    row_max = np.where(np.isfinite(row_max), row_max, 0.0)
    e = np.where(allowed, np.exp(s - row_max), 0.0)
    denom = e.sum(axis=1, keepdims=True)
    num = e @ v
    safe = np.where(denom > 0, denom, 1.0)
    return np.where(denom > 0, num / safe, 0.0)


def varlen_mask(cu_q: Sequence[int], cu_k: Sequence[int]) -> np.ndarray:
    """Dense [T_q, T_k] mask of a packed batch: query row i may see key row j
    exactly when both lie in the same sequence (tokens never attend across
    requests, "feat: Support dynamic batching for heterogeneous diffusion
    requests", AttentionMetadata)."""
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_k = np.asarray(cu_k, dtype=np.int64)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    seq_of_q = np.full(Tq, -1, dtype=np.int64)
    seq_of_k = np.full(Tk, -2, dtype=np.int64)
    for b in range(len(cu_q) - 1):
        seq_of_q[cu_q[b]:cu_q[b + 1]] = b
        seq_of_k[cu_k[b]:cu_k[b + 1]] = b
    return seq_of_q[:, None] == seq_of_k[None, :]


def varlen_attention(q, k, v, cu_q: Sequence[int], cu_k: Sequence[int],
                     scale: Optional[float] = None,
                     rows: Optional[Sequence[int]] = None,
                     chunk: int = 1024) -> np.ndarray:
    """Packed varlen attention, one sequence at a time.

    q [T_q, H, D], k/v [T_k, H, D]; sequence b owns query rows
    [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]).  For each sequence
    the explicit mask is the sequence's block of ``varlen_mask`` (all keys of
    the same sequence, non-causal); it is applied to the sequence's own keys.
    Returns float64 [T_q, H, D]; rows of queries that belong to no sequence
    (beyond cu_q[-1]) are zero.  With ``rows`` given, returns only those query
    rows, [len(rows), H, D].
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_k = np.asarray(cu_k, dtype=np.int64)
    H, D = q.shape[1], q.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    want = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(want), H, v.shape[2]), dtype=np.float64)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        sel = np.nonzero((want >= q0) & (want < q1))[0]
        if len(sel) == 0:
            continue
        for c0 in range(0, len(sel), chunk):
            idx = sel[c0:c0 + chunk]
            qrows = want[idx]
            allowed = np.ones((len(qrows), int(k1 - k0)), dtype=bool)
            for h in range(H):
                out[idx, h, :] = masked_attention(q[qrows, h, :], k[k0:k1, h, :],
                                                  v[k0:k1, h, :], allowed, scale)
    return out


def key_padding_attention(q, k, v, valid: int, scale: Optional[float] = None,
                          rows: Optional[Sequence[int]] = None,
                          chunk: int = 1024) -> np.ndarray:
    """Dense attention of one sequence whose buffer holds ``valid`` real tokens
    followed by padding tokens, with the padding keys masked out (the masked
    reference for an auto-padded sequence, "[Perf][qwen-image-edit] Skip
    attention-mask to avoid varlen path", Test Result).  q/k/v [T, H, D];
    key j is allowed iff j < valid.  Returns [T or len(rows), H, D]."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, H, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    want = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(want), H, v.shape[2]), dtype=np.float64)
    key_ok = np.arange(k.shape[0]) < valid
    for c0 in range(0, len(want), chunk):
        qrows = want[c0:c0 + chunk]
        allowed = np.broadcast_to(key_ok[None, :], (len(qrows), k.shape[0]))
        for h in range(H):
            out[c0:c0 + len(qrows), h, :] = masked_attention(q[qrows, h, :], k[:, h, :],
                                                             v[:, h, :], allowed, scale)
    return out


def block_window_mask(n: int, block: int, look_back: int, look_ahead: int,
                      rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Dense block-difference mask of the Token2Wav DiT.

    The sequence is padded up to a whole number of blocks; with
    diff[i, j] = block(j) - block(i) (an int64 tensor), key j is allowed for
    query i iff -look_back <= diff <= look_ahead (look_back blocks before,
    look_ahead blocks after) and j is not a padding position, j < n ("[Perf]
    [Model] Use block-sparse attention in Qwen2.5-Omni Token2Wav DiT",
    Purpose: mask built from the block-difference tensor; review: "own block
    plus look_backward_block before and look_ahead_block after ... masking the
    shifted-out and padded positions").  Returns [n or len(rows), n] bool.
    """
    n_pad = ((n + block - 1) // block) * block
    qi = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    kj = np.arange(n_pad, dtype=np.int64)
    diff = (kj[None, :] // block) - (qi[:, None].astype(np.int64) // block)
    allowed = (diff >= -look_back) & (diff <= look_ahead)
    allowed &= (kj < n)[None, :]
    return allowed[:, :n]


def block_window_attention(q, k, v, block: int, look_back: int, look_ahead: int,
                           scale: Optional[float] = None,
                           rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Dense attention under ``block_window_mask`` for q/k/v [batch, n, H, D].

    Every batch entry and head attends over all n keys with the block-window
    mask applied.  Returns float64 [batch, n (or len(rows)), H, D]."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    batch, n, H, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    want = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    allowed = block_window_mask(n, block, look_back, look_ahead, rows=want)
    out = np.zeros((batch, len(want), H, v.shape[3]), dtype=np.float64)
    for bi in range(batch):
        for h in range(H):
            out[bi, :, h, :] = masked_attention(q[bi, want, h, :], k[bi, :, h, :],
                                                v[bi, :, h, :], allowed, scale)
    return out


def varlen_useful_flops(lengths_q: Sequence[int], lengths_k: Sequence[int],
                        H: int, D: int) -> int:
    """Useful attention FLOPs 4 * H * D * sum_b Lq[b] * Lk[b] (QK^T and PV,
    two FLOPs per multiply-add, only allowed query/key pairs)."""
    return 4 * H * D * int(sum(int(a) * int(b) for a, b in zip(lengths_q, lengths_k)))


def block_window_useful_flops(batch: int, n: int, H: int, D: int, block: int,
                              look_back: int, look_ahead: int) -> int:
    """Useful FLOPs of one block-window layer: 4 * H * D * (allowed pairs)."""
    pairs = int(block_window_mask(n, block, look_back, look_ahead).sum())
    return 4 * batch * H * D * pairs
