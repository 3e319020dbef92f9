"""Seeded random sweeps: many small shapes drawn from fixed seeds, each
compared element by element with the fp64 oracle through the C ABI.

The hand-picked cases in the other files aim at known edges; these draw
lengths, head counts, head dims, blocks and looks at random (within sizes the
oracle computes in a moment), so that combinations nobody listed are also
checked: varlen batches with cross lengths and empty sequences, block
windows in bf16 and fp32 with any block, look and partial last block, the
packed-M linear layer with ragged M, N and K, pack/unpack (bit-exact) and
request-local RoPE with random offsets and bases."""
import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_close_to_oracle, gpu_varlen

pytestmark = pytest.mark.gpu

F32_MAX_ABS = 6e-6
F32_MEAN_ABS = 5e-7


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    return pv


def _varlen_case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 7))
    D = int(rng.choice([64, 128]))
    H = int(rng.integers(1, 4))
    lq = [int(x) for x in rng.integers(0, 400, size=B)]
    cross = bool(rng.integers(0, 2))
    lk = [int(x) for x in rng.integers(0, 400, size=B)] if cross else None
    if sum(lq) == 0:
        lq[0] = 1
    return lq, lk, H, D


@pytest.mark.parametrize("seed", range(40))
def test_varlen_random_shapes(pv, seed):
    lq, lk, H, D = _varlen_case(seed)
    w = workloads.random_varlen(lq, lk, H, D, seed=seed)
    out, cu_q, cu_k = gpu_varlen(pv, w)
    ocq = oracle.cu_seqlens_from_lengths(w.lengths_q)
    ock = oracle.cu_seqlens_from_lengths(w.lengths_k)
    want = oracle.varlen_attention(w.q, w.k, w.v, ocq, ock, w.scale)
    T = int(ocq[-1])
    assert_close_to_oracle(oracle.to_f64(out)[:T], want[:T], f"seed={seed} Lq={lq} Lk={lk}")
    assert pv.get_device_status() == 0


def _window_case(seed):
    rng = np.random.default_rng(2000 + seed)
    block = int(rng.choice([1, 3, 8, 13, 20, 24, 31, 32, 40, 64, 100]))
    n = int(rng.integers(1, 6 * block + 200))
    look = (int(rng.integers(0, 4)), int(rng.integers(0, 4)))
    batch = int(rng.integers(1, 3))
    H = int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    return block, n, look, batch, H, D


@pytest.mark.parametrize("seed", range(40))
def test_block_window_random_shapes(pv, seed):
    block, n, look, batch, H, D = _window_case(seed)
    w = workloads.random_block_window(batch, n, H, D, block, seed=seed)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    got = pv.block_window_attn_fwd(q, k, v, block, look[0], look[1], scale=w.scale)
    want = oracle.block_window_attention(w.q, w.k, w.v, block, look[0], look[1], w.scale)
    assert_close_to_oracle(oracle.to_f64(got.cpu()), want,
                           f"seed={seed} block={block} n={n} look={look} D={D}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("seed", range(40))
def test_block_window_f32_random_shapes(pv, seed):
    block, n, look, batch, H, D = _window_case(seed + 100)
    w = workloads.random_block_window_f32(batch, n, H, D, block, seed=seed)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    got = oracle.to_f64(pv.block_window_attn_fwd_f32(q, k, v, block, look[0], look[1],
                                                     scale=w.scale).cpu())
    want = oracle.block_window_attention(w.q, w.k, w.v, block, look[0], look[1], w.scale)
    err = np.abs(got - want)
    what = f"seed={seed} block={block} n={n} look={look} D={D}"
    assert np.isfinite(got).all(), what
    assert err.max() <= F32_MAX_ABS, f"{what}: max abs {err.max():.3e}"
    assert err.mean() <= F32_MEAN_ABS, f"{what}: mean abs {err.mean():.3e}"
    assert pv.get_device_status() == 0


def _linear_case(seed):
    rng = np.random.default_rng(3000 + seed)
    M = int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 150))
    K = 8 * int(rng.integers(1, 80))
    return M, N, K, bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(40))
def test_linear_random_shapes(pv, seed):
    # bound: one bf16 rounding of the result plus an fp32 accumulation
    # allowance of 2^-14 * sum_k |x_k w_k| (as the linear layer's own tests)
    M, N, K, with_bias = _linear_case(seed)
    c = workloads.linear_case([M], N, K, seed=seed, bias=with_bias)
    y = pv.linear_bf16(c.x.cuda(), c.w.cuda(), None if c.bias is None else c.bias.cuda()).cpu()
    want = oracle.linear(c.x, c.w, c.bias)
    absdot = np.abs(oracle.to_f64(c.x)) @ np.abs(oracle.to_f64(c.w)).T
    if c.bias is not None:
        absdot = absdot + np.abs(oracle.to_f64(c.bias))[None, :]
    excess = np.abs(oracle.to_f64(y) - want) - (2.0 ** -8 * np.abs(want) + 2.0 ** -14 * absdot)
    assert excess.max() <= 0, f"seed={seed} M={M} N={N} K={K}: max excess {excess.max():.3e}"
    assert pv.get_device_status() == 0


def _rows_case(seed, base_seed):
    rng = np.random.default_rng(base_seed + seed)
    B = int(rng.integers(1, 7))
    lengths = [int(x) for x in rng.integers(0, 300, size=B)]
    H = int(rng.integers(1, 5))
    D = int(rng.choice([8, 16, 64, 128]))
    return lengths, H, D, rng


@pytest.mark.parametrize("seed", range(20))
def test_pack_unpack_random_shapes(pv, seed):
    # bit-exact: padded -> flat -> padded, padding rows of the target kept
    import torch
    lengths, H, D, _ = _rows_case(seed, 4000)
    if sum(lengths) == 0:   # (empty buffers have null pointers; not this test's case)
        lengths[0] = 1
    pw = workloads.padded(lengths, H, D, seed=seed)
    cu = pv.cu_seqlens_from_lengths(torch.tensor(lengths, dtype=torch.int32, device="cuda"))
    i16 = lambda t: t.view(torch.int16).cpu().numpy()
    flat = pv.pack(pw.q.cuda(), cu, sum(lengths))
    want = oracle.pack(i16(pw.q), lengths)
    assert np.array_equal(i16(flat), want), f"seed={seed} L={lengths}"
    target = torch.full_like(pw.q, -2.0).cuda()
    pv.unpack(flat, cu, target)
    want_pad = oracle.unpack(want, lengths, i16(torch.full_like(pw.q, -2.0)))
    assert np.array_equal(i16(target), want_pad), f"seed={seed} L={lengths}"
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("seed", range(20))
def test_rope_random_shapes(pv, seed):
    # within one bf16 rounding of a result computed to ~1e-5 of its pair's norm
    import torch
    lengths, H, D, rng = _rows_case(seed, 5000)
    if sum(lengths) == 0:
        lengths[0] = 1
    offsets = [int(x) for x in rng.integers(0, 5000, size=len(lengths))]
    base = float(rng.choice([500.0, 1e4, 1e6]))
    w = workloads.random_varlen(lengths, None, H, D, seed=seed)
    dev = "cuda"
    cu = pv.cu_seqlens_from_lengths(torch.tensor(lengths, dtype=torch.int32, device=dev))
    q, k = w.q.to(dev), w.k.to(dev)
    pv.rope_packed(q, k, cu, cu, torch.tensor(offsets, dtype=torch.int32, device=dev), base)
    pos = oracle.rope_positions(lengths, offsets)
    for got, x in ((q.cpu(), w.q), (k.cpu(), w.k)):
        want = oracle.rope(x, pos, base)
        xx = oracle.to_f64(x)
        pair = np.repeat(np.hypot(xx[..., 0::2], xx[..., 1::2]), 2, axis=-1)
        excess = np.abs(oracle.to_f64(got) - want) - (2.0 ** -8 * np.abs(want) + 1e-5 * pair)
        assert excess.max() <= 0, f"seed={seed} L={lengths} D={D}: {excess.max():.3e}"
    assert pv.get_device_status() == 0
