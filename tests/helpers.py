"""Shared test helpers: run the CUDA path through the binding, compare with the
oracle under the tolerance the attention kernels are held to."""
import numpy as np
import torch

# bf16 outputs against the exact fp64 oracle
MAX_ABS_TOL = 2e-2
MEAN_ABS_TOL = 2e-3


def assert_close_to_oracle(got: np.ndarray, want: np.ndarray, what: str = ""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    max_abs, mean_abs = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert max_abs <= MAX_ABS_TOL and mean_abs <= MEAN_ABS_TOL, \
        f"{what}: max_abs={max_abs:.3e} mean_abs={mean_abs:.3e}"
    return max_abs, mean_abs


def gpu_varlen(pv, w, out_fill=float("nan"), scale=None):
    """Run the full GPU path for a VarlenWorkload: boundaries from lengths on
    the device, then attention.  Returns the output (CPU bf16) and cu arrays."""
    dev = "cuda"
    lq = torch.tensor(w.lengths_q, dtype=torch.int32, device=dev)
    lk = torch.tensor(w.lengths_k, dtype=torch.int32, device=dev)
    cu_q = pv.cu_seqlens_from_lengths(lq)
    cu_k = pv.cu_seqlens_from_lengths(lk)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    out = torch.full_like(q, out_fill)
    pv.varlen_attn_fwd(q, k, v, cu_q, cu_k, max(w.lengths_q), max(w.lengths_k),
                       scale=w.scale if scale is None else scale, out=out)
    torch.cuda.synchronize()
    return out.cpu(), cu_q.cpu(), cu_k.cpu()


def sample_rows(lengths, per_seq=12, seed=0, tile=128):
    """Query rows that cover each sequence's ends, tile edges and random rows."""
    rng = np.random.default_rng(seed)
    rows, start = [], 0
    for L in lengths:
        if L > 0:
            cand = {0, L - 1, min(L - 1, tile - 1), min(L - 1, tile), L // 2,
                    (L - 1) // tile * tile}
            cand |= set(rng.integers(0, L, size=per_seq).tolist())
            rows += [start + r for r in sorted(cand)]
        start += L
    return np.array(rows, dtype=np.int64)


def item_rows(lengths, item=256, tile=128, seed=0):
    """One random query row from every 128-row tile of every sequence (so
    both tiles of every 256-row work item of the varlen kernel), plus each
    sequence's first and last rows and the rows on either side of every tile
    edge that a sequence's last tile creates.  The oracle computes all heads
    of a row, so every (sequence, head, work item) is checked."""
    rng = np.random.default_rng(seed)
    rows, start = [], 0
    for L in lengths:
        if L > 0:
            cand = {0, L - 1, (L - 1) // tile * tile, max(0, (L - 1) // tile * tile - 1)}
            for t0 in range(0, L, tile):
                cand.add(int(rng.integers(t0, min(L, t0 + tile))))
            rows += [start + r for r in sorted(cand)]
        start += L
    return np.array(rows, dtype=np.int64)


def items_covered(rows, lengths, item=256, tile=128):
    """Per sequence, the sets of (item, tile) indices the given global rows
    fall in, and the full sets they should cover."""
    got, want, start = [], [], 0
    rows = np.asarray(rows)
    for L in lengths:
        local = rows[(rows >= start) & (rows < start + L)] - start
        got.append({(int(r) // item, (int(r) % item) // tile) for r in local})
        want.append({(t // item, (t % item) // tile) for t in range(0, L, tile)})
        start += L
    return got, want
