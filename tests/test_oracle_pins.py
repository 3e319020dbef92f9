"""Pins for the CPU oracle: brute force, closed forms, a library routine, the
pages' invariants and the values the pages print.  None of these call the
CUDA library; they check the oracle against something other than itself."""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Brute force written from the definitions, independently of the oracle:
# pure Python loops, math.exp and math.fsum, key sets built as index ranges.
# ----------------------------------------------------------------------------

def _brute_row(qrow, keys, vals, scale, dv):
    if not keys:
        return [0.0] * dv
    s = [scale * math.fsum(a * b for a, b in zip(qrow, kr)) for kr in keys]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = math.fsum(e)
    return [math.fsum(ei * vr[d] for ei, vr in zip(e, vals)) / z for d in range(dv)]


def brute_varlen(q, k, v, lengths_q, lengths_k, scale):
    q, k, v = q.tolist(), k.tolist(), v.tolist()
    H, dv = len(q[0]) if q else 0, len(v[0][0]) if v else 0
    out = []
    qs = ks = 0
    for lq, lk in zip(lengths_q, lengths_k):
        for i in range(qs, qs + lq):
            row = []
            for h in range(H):
                keys = [k[j][h] for j in range(ks, ks + lk)]
                vals = [v[j][h] for j in range(ks, ks + lk)]
                row.append(_brute_row(q[i][h], keys, vals, scale, dv))
            out.append(row)
        qs += lq
        ks += lk
    return np.array(out, dtype=np.float64).reshape(qs, H, dv)


def brute_block_window(q, k, v, block, look_back, look_ahead, scale):
    """q/k/v [batch, n, H, D]; query i sees key rows of blocks
    block(i) - look_back .. block(i) + look_ahead that exist in [0, n)."""
    qq, kk, vv = q.tolist(), k.tolist(), v.tolist()
    batch, n, H, dv = len(qq), len(qq[0]), len(qq[0][0]), len(vv[0][0][0])
    out = np.zeros((batch, n, H, dv))
    for b in range(batch):
        for i in range(n):
            bi = i // block
            lo = max(0, (bi - look_back) * block)
            hi = min(n, (bi + look_ahead + 1) * block)
            for h in range(H):
                keys = [kk[b][j][h] for j in range(lo, hi)]
                vals = [vv[b][j][h] for j in range(lo, hi)]
                out[b, i, h] = _brute_row(qq[b][i][h], keys, vals, scale, dv)
    return out


def _bf16_f64(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)
    return t.double().numpy()


# ----------------------------------------------------------------------------
# Integer / copy steps
# ----------------------------------------------------------------------------

def test_cu_seqlens_brute():
    rng = random.Random(1)
    for _ in range(50):
        L = [rng.choice([0, 1, 7, 128, 129, 300]) for _ in range(rng.randint(1, 9))]
        cu = oracle.cu_seqlens_from_lengths(L)
        assert cu.dtype == np.int32 and len(cu) == len(L) + 1 and cu[0] == 0
        run = 0
        for b, n in enumerate(L):
            assert cu[b] == run
            run += n
        assert cu[-1] == run
    with pytest.raises(ValueError):
        oracle.cu_seqlens_from_lengths([3, -1])


def test_pack_unpack_brute():
    rng = np.random.default_rng(3)
    L = [5, 0, 9, 1]
    padded = rng.integers(-30000, 30000, size=(4, 9, 2, 3)).astype(np.int16)
    flat = oracle.pack(padded, L)
    assert flat.shape == (15, 2, 3)
    row = 0
    for b, n in enumerate(L):
        for i in range(n):
            assert np.array_equal(flat[row], padded[b, i])
            row += 1
    fill = np.full_like(padded, 7)
    back = oracle.unpack(flat, L, fill)
    for b, n in enumerate(L):
        assert np.array_equal(back[b, :n], padded[b, :n])
        assert (back[b, n:] == 7).all()


def test_work_order_brute():
    rng = random.Random(5)
    for _ in range(30):
        B = rng.randint(1, 7)
        Lq = [rng.choice([0, 1, 127, 128, 129, 500]) for _ in range(B)]
        Lk = [rng.choice([0, 5, 128, 500]) if rng.random() < 0.3 else Lq[b] for b in range(B)]
        H, tile = rng.randint(1, 4), 128
        items = oracle.work_order(Lq, Lk, H, tile)
        # every (b, h, t) exactly once
        expect = {(b, h, t) for b in range(B) for h in range(H)
                  for t in range(-(-Lq[b] // tile))}
        assert len(items) == len(expect) and set(items) == expect
        # sequences in non-increasing key length, ties by lower index,
        # and each sequence's items contiguous, heads then tiles in order
        seq_seen = []
        for b, _, _ in items:
            if not seq_seen or seq_seen[-1] != b:
                assert b not in seq_seen
                seq_seen.append(b)
        for a, c in zip(seq_seen, seq_seen[1:]):
            assert (Lk[a] > Lk[c]) or (Lk[a] == Lk[c] and a < c)
        for b in seq_seen:
            mine = [(h, t) for bb, h, t in items if bb == b]
            assert mine == sorted(mine)


# ----------------------------------------------------------------------------
# Attention: brute force on tiny inputs
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("case", [
    dict(Lq=[3, 5], Lk=[3, 5], H=2, D=4, scale=None),
    dict(Lq=[1], Lk=[1], H=1, D=8, scale=0.7),
    dict(Lq=[4, 0, 2], Lk=[6, 3, 1], H=2, D=3, scale=1.3),   # Lq != Lk, empty queries
    dict(Lq=[2, 3], Lk=[0, 4], H=1, D=5, scale=None),         # queries with no keys
    dict(Lq=[8, 7, 2], Lk=[8, 7, 2], H=2, D=8, scale=3.0),
])
def test_varlen_matches_brute_force(case):
    Tq, Tk = sum(case["Lq"]), sum(case["Lk"])
    H, D = case["H"], case["D"]
    q = _bf16_f64((Tq, H, D), 11)
    k = _bf16_f64((Tk, H, D), 12)
    v = _bf16_f64((Tk, H, D + 1), 13)
    scale = case["scale"] if case["scale"] is not None else 1 / math.sqrt(D)
    cu_q = oracle.cu_seqlens_from_lengths(case["Lq"])
    cu_k = oracle.cu_seqlens_from_lengths(case["Lk"])
    got = oracle.varlen_attention(q, k, v, cu_q, cu_k, scale)
    want = brute_varlen(q, k, v, case["Lq"], case["Lk"], scale)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_varlen_large_scores_stable():
    # scores of order 1e3: needs the max subtraction to stay finite
    q = _bf16_f64((6, 1, 4), 21, scale=30.0)
    k = _bf16_f64((6, 1, 4), 22, scale=30.0)
    v = _bf16_f64((6, 1, 4), 23)
    cu = [0, 6]
    got = oracle.varlen_attention(q, k, v, cu, cu, 1.0)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, brute_varlen(q, k, v, [6], [6], 1.0), atol=1e-12)


@pytest.mark.parametrize("n", [10, 96, 101])
@pytest.mark.parametrize("look", [(0, 0), (1, 0), (0, 1), (1, 1), (2, 1)])
def test_block_window_matches_brute_force(n, look):
    # the pages' unit matrix: shorter than a block, a whole number of blocks,
    # a partial last block; plain / look-backward / look-ahead layers
    q = _bf16_f64((1, n, 1, 4), 31)
    k = _bf16_f64((1, n, 1, 4), 32)
    v = _bf16_f64((1, n, 1, 4), 33)
    got = oracle.block_window_attention(q, k, v, 24, look[0], look[1], 0.5)
    want = brute_block_window(q, k, v, 24, look[0], look[1], 0.5)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_block_window_direction():
    # look_back = earlier frames, look_ahead = later frames
    m = oracle.block_window_mask(72, 24, 1, 0)
    assert m[30, 0] and m[30, 47] and not m[30, 48]       # block 1 sees blocks 0, 1
    m = oracle.block_window_mask(72, 24, 0, 1)
    assert not m[30, 23] and m[30, 24] and m[30, 71]      # block 1 sees blocks 1, 2
    m = oracle.block_window_mask(50, 24, 0, 1)
    assert m[30].sum() == 26                              # 24 + 2 valid of the partial block


def test_block_window_key_counts_golden():
    with open(os.path.join(GOLDEN, "block_window_key_counts.json")) as f:
        g = json.load(f)
    n, block = g["n"], g["block"]
    full_blocks = n // block
    for case in g["cases"]:
        m = oracle.block_window_mask(n, block, case["look_back"], case["look_ahead"])
        counts = m.sum(axis=1)
        # queries away from both ends, whose window holds only whole blocks
        interior = np.arange(block, (full_blocks - 1) * block)
        assert (counts[interior] == case["keys_per_query"]).all()
        assert counts[: full_blocks * block].min() >= g["min_keys_any_full_block_query"]
        assert counts.max() <= g["max_keys_any_query_one_neighbour"]


# ----------------------------------------------------------------------------
# A library routine as a special case: torch SDPA in float64 with a bool mask
# ----------------------------------------------------------------------------

def _sdpa(q, k, v, mask, scale):
    # q [M, H, D] -> [H, M, D]
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2)
    vt = torch.from_numpy(v).permute(1, 0, 2)
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask), scale=scale)
    return out.permute(1, 0, 2).numpy()


def test_varlen_matches_sdpa_fp64():
    L = [57, 130, 1, 200]
    T = sum(L)
    q, k, v = (_bf16_f64((T, 3, 32), s) for s in (41, 42, 43))
    cu = oracle.cu_seqlens_from_lengths(L)
    got = oracle.varlen_attention(q, k, v, cu, cu, 0.2)
    want = _sdpa(q, k, v, oracle.varlen_mask(cu, cu), 0.2)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-10)


def test_block_window_matches_sdpa_fp64():
    n = 250
    q, k, v = (_bf16_f64((1, n, 2, 16), s) for s in (51, 52, 53))
    for lb, la in [(0, 0), (1, 1), (2, 0)]:
        got = oracle.block_window_attention(q, k, v, 24, lb, la, 0.25)
        mask = oracle.block_window_mask(n, 24, lb, la)
        want = _sdpa(q[0], k[0], v[0], mask, 0.25)
        np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-10)


# ----------------------------------------------------------------------------
# Closed forms
# ----------------------------------------------------------------------------

def test_scale_zero_is_mean_of_values():
    L = [5, 9]
    q, k, v = (_bf16_f64((14, 2, 8), s) for s in (61, 62, 63))
    cu = oracle.cu_seqlens_from_lengths(L)
    got = oracle.varlen_attention(q, k, v, cu, cu, 0.0)
    np.testing.assert_allclose(got[:5], np.broadcast_to(v[:5].mean(0), (5, 2, 8)), atol=1e-14)
    np.testing.assert_allclose(got[5:], np.broadcast_to(v[5:].mean(0), (9, 2, 8)), atol=1e-14)


def test_identical_keys_give_mean():
    q = _bf16_f64((7, 1, 8), 64)
    k = np.repeat(_bf16_f64((1, 1, 8), 65), 7, axis=0)
    v = _bf16_f64((7, 1, 8), 66)
    got = oracle.varlen_attention(q, k, v, [0, 7], [0, 7], 0.3)
    np.testing.assert_allclose(got, np.broadcast_to(v.mean(0), (7, 1, 8)), atol=1e-14)


def test_constant_values():
    q, k = _bf16_f64((20, 2, 8), 71), _bf16_f64((20, 2, 8), 72)
    v = np.full((20, 2, 8), 0.375)
    got = oracle.varlen_attention(q, k, v, [0, 11, 20], [0, 11, 20], 1.0)
    np.testing.assert_allclose(got, 0.375, atol=1e-15)
    got = oracle.block_window_attention(q[None], k[None], v[None], 4, 1, 1, 1.0)
    np.testing.assert_allclose(got, 0.375, atol=1e-15)


def test_single_key_returns_its_value():
    # block 1, no neighbours: each query sees only its own key row
    q, k, v = (_bf16_f64((1, 13, 2, 8), s) for s in (81, 82, 83))
    got = oracle.block_window_attention(q, k, v, 1, 0, 0, 0.9)
    np.testing.assert_array_equal(got, v)
    # one key per sequence in varlen
    q2, k2, v2 = (_bf16_f64((3, 1, 4), s) for s in (84, 85, 86))
    got = oracle.varlen_attention(q2, k2, v2, [0, 1, 2, 3], [0, 1, 2, 3], 1.0)
    np.testing.assert_array_equal(got, v2)


def test_block_at_least_n_is_full_attention():
    n = 40
    q, k, v = (_bf16_f64((1, n, 2, 8), s) for s in (91, 92, 93))
    got = oracle.block_window_attention(q, k, v, 64, 0, 0, 0.4)
    want = oracle.varlen_attention(q[0], k[0], v[0], [0, n], [0, n], 0.4)
    np.testing.assert_allclose(got[0], want, atol=1e-14)


def test_fully_masked_rows_are_zero():
    q, k, v = (_bf16_f64((4, 1, 4), s) for s in (94, 95, 96))
    got = oracle.varlen_attention(q, k[:0], v[:0], [0, 4], [0, 0], 1.0)
    assert (got == 0).all()


# ----------------------------------------------------------------------------
# Invariants the pages state
# ----------------------------------------------------------------------------

def test_packed_equals_each_request_alone_and_dense_mask():
    # packed == per-request (the pages' bitwise batch-vs-serial check), and the
    # per-sequence evaluation == one dense attention under the packed mask
    L = [33, 1, 90, 64]
    w = workloads.random_varlen(L, None, 2, 16, seed=7)
    q, k, v = oracle.to_f64(w.q), oracle.to_f64(w.k), oracle.to_f64(w.v)
    cu = oracle.cu_seqlens_from_lengths(L)
    packed = oracle.varlen_attention(q, k, v, cu, cu, 0.25)
    for b in range(len(L)):
        s = slice(cu[b], cu[b + 1])
        alone = oracle.varlen_attention(q[s], k[s], v[s], [0, L[b]], [0, L[b]], 0.25)
        assert np.array_equal(packed[s], alone)
    mask = oracle.varlen_mask(cu, cu)
    for h in range(2):
        dense = oracle.masked_attention(q[:, h], k[:, h], v[:, h], mask, 0.25)
        np.testing.assert_allclose(packed[:, h], dense, atol=1e-13)


def test_masked_positions_contribute_nothing():
    L = [20, 30]
    cu = oracle.cu_seqlens_from_lengths(L)
    q, k, v = (_bf16_f64((50, 2, 8), s) for s in (101, 102, 103))
    base = oracle.varlen_attention(q, k, v, cu, cu, 0.3)
    k2, v2 = k.copy(), v.copy()
    k2[20:] += 1e4
    v2[20:] -= 1e4
    pert = oracle.varlen_attention(q, k2, v2, cu, cu, 0.3)
    assert np.array_equal(base[:20], pert[:20])
    # block window: keys outside a query's window do not matter
    n = 96
    qb, kb, vb = (_bf16_f64((1, n, 1, 8), s) for s in (104, 105, 106))
    base = oracle.block_window_attention(qb, kb, vb, 24, 1, 0, 0.3)
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[0, 48:] = 1e4    # blocks 2, 3 are invisible to queries of blocks 0, 1
    vb2[0, 48:] = -1e4
    pert = oracle.block_window_attention(qb, kb2, vb2, 24, 1, 0, 0.3)
    assert np.array_equal(base[0, :48], pert[0, :48])


def test_request_permutation():
    L = [12, 40, 7]
    cu = oracle.cu_seqlens_from_lengths(L)
    q, k, v = (_bf16_f64((59, 1, 8), s) for s in (111, 112, 113))
    base = oracle.varlen_attention(q, k, v, cu, cu, 0.5)
    perm = [2, 0, 1]
    segs = [slice(cu[b], cu[b + 1]) for b in perm]
    qp, kp, vp = (np.concatenate([x[s] for s in segs]) for x in (q, k, v))
    cup = oracle.cu_seqlens_from_lengths([L[b] for b in perm])
    got = oracle.varlen_attention(qp, kp, vp, cup, cup, 0.5)
    np.testing.assert_array_equal(got, np.concatenate([base[s] for s in segs]))


def test_trimmed_padded_tail_equals_key_padding_mask():
    # an auto-padded sequence (6889 -> 6896 at 1328x1328 with 8 ranks, from the
    # golden file): trimming cu_seqlens equals dense attention with the padding
    # keys masked
    with open(os.path.join(GOLDEN, "token_counts.json")) as f:
        g = json.load(f)
    case = g["sp_pad"][1]
    valid, total = case["seq_len"], case["padded"]
    assert total - valid == case["pad_size"] == (-valid) % case["world_size"]
    q, k, v = (_bf16_f64((total, 1, 8), s) for s in (121, 122, 123))
    rows = list(range(0, valid, 97)) + [valid - 1]
    masked = oracle.key_padding_attention(q, k, v, valid, 0.35, rows=rows)
    trimmed = oracle.varlen_attention(q, k, v, [0, valid], [0, valid], 0.35, rows=rows)
    np.testing.assert_allclose(masked, trimmed, atol=1e-13)


def _block_local_fp32(q, k, v, block, lb, la, scale):
    """Per-block formulation the Token2Wav change describes, in float32: each
    query block attends to the concatenation of its window's key blocks, with
    positions beyond either end or beyond n masked."""
    batch, n, H, D = q.shape
    nb = -(-n // block)
    out = np.zeros(q.shape, dtype=np.float32)
    q32, k32, v32 = (x.astype(np.float32) for x in (q, k, v))
    for bi in range(nb):
        qs = slice(bi * block, min(n, (bi + 1) * block))
        lo, hi = max(0, bi - lb) * block, min(n, (bi + la + 1) * block)
        for b in range(batch):
            for h in range(H):
                s = (q32[b, qs, h] @ k32[b, lo:hi, h].T) * np.float32(scale)
                s = s - s.max(axis=1, keepdims=True)
                e = np.exp(s)
                out[b, qs, h] = (e @ v32[b, lo:hi, h]) / e.sum(axis=1, keepdims=True)
    return out


def test_block_window_within_pages_fp32_bound():
    # block-local vs dense differed by <= 6e-6 in fp32 on the pages' 4000-frame
    # sample ("... Token2Wav DiT", Test Result); the oracle is exact, so the
    # fp32 block-local result must sit within that bound of it
    n = 4000
    q, k, v = (_bf16_f64((1, n, 2, 64), s) for s in (131, 132, 133))
    for lb, la in [(0, 0), (1, 0), (0, 1)]:
        exact = oracle.block_window_attention(q, k, v, 24, lb, la, 0.125)
        local = _block_local_fp32(q, k, v, 24, lb, la, 0.125)
        assert np.abs(exact - local).max() <= 6e-6


# ----------------------------------------------------------------------------
# Input recipe pinned to the pages' printed token counts
# ----------------------------------------------------------------------------

def test_token_counts_golden():
    with open(os.path.join(GOLDEN, "token_counts.json")) as f:
        g = json.load(f)
    for e in g["image_tokens"]:
        assert workloads.image_tokens(e["height"], e["width"]) == e["tokens"]
    assert 2 * workloads.image_tokens(2048, 2048) == g["edit_tokens_2048"]
    assert workloads.lengths_single_edit() == [256 + g["edit_tokens_2048"]]
    plan = g["mixfusion_plan"]
    toks = [workloads.image_tokens(h, w) for h, w in plan["sizes"]]
    assert math.gcd(*toks) == plan["chunk_size"]
    assert sum(toks) // plan["chunk_size"] == plan["chunk_count"]
    assert workloads.IMAGE_TOKENS == tuple(workloads.image_tokens(s, s) for s in (768, 1024, 1328, 2048))


def test_useful_flops():
    assert oracle.varlen_useful_flops([37, 64], [37, 64], 2, 64) == 4 * 2 * 64 * (37 * 37 + 64 * 64)
    # own-block layer of Token2Wav: n = 2400 = 100 blocks of 24 -> 100 * 24 * 24 pairs
    assert oracle.block_window_useful_flops(1, 2400, 16, 64, 24, 0, 0) == 4 * 16 * 64 * 57600
    # one neighbour each side: 100 blocks * 24 rows * 72 keys minus the two ends
    assert oracle.block_window_useful_flops(1, 2400, 16, 64, 24, 1, 1) == \
        4 * 16 * 64 * (57600 * 3 - 2 * 24 * 24)
