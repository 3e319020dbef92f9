"""Parity of the batch-invariant packed-M linear layer with the fp64 oracle,
and its batch invariance (packed rows equal rows computed alone, bit for
bit), through the C ABI.

Bound per element: one bf16 rounding of the result (at most 2^-8 of its
magnitude) plus an fp32 accumulation allowance of 2^-14 * sum_k |x_k w_k|
(tensor-core fp32 accumulation over K terms, bias added in fp32).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    return pv


def _bound(x, w, bias, want):
    absdot = np.abs(oracle.to_f64(x)) @ np.abs(oracle.to_f64(w)).T
    if bias is not None:
        absdot = absdot + np.abs(oracle.to_f64(bias))[None, :]
    return 2.0 ** -8 * np.abs(want) + 2.0 ** -14 * absdot


def _check(got, x, w, bias, rows=None):
    want = oracle.linear(x, w, bias) if rows is None else oracle.linear_rows(x, w, bias, rows)
    xx = x if rows is None else x[torch.as_tensor(rows)]
    excess = np.abs(oracle.to_f64(got) - want) - _bound(xx, w, bias, want)
    assert excess.max() <= 0, f"max excess {excess.max():.3e}"


def _run(pv, x, w, bias=None):
    y = pv.linear_bf16(x.cuda(), w.cuda(), None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    return y.cpu()


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (37, 264, 72), (300, 520, 200), (129, 256, 64),
                                   (256, 512, 128), (200, 1032, 3072)])
@pytest.mark.parametrize("with_bias", [False, True])
def test_against_oracle(pv, M, N, K, with_bias):
    # ragged M, N and K tails: partial 128-row, 256-column and 64-deep tiles
    w = workloads.linear_case([M], N, K, seed=M + N + K, bias=with_bias)
    _check(_run(pv, w.x, w.w, w.bias), w.x, w.w, w.bias)
    assert pv.get_device_status() == 0


def test_packed_equals_per_request_bitwise(pv):
    w = workloads.linear_case([37, 300, 1, 129, 512, 128], 776, 328, seed=7)
    packed = _run(pv, w.x, w.w, w.bias)
    r0 = 0
    for L in w.lengths:
        alone = _run(pv, w.x[r0:r0 + L].contiguous(), w.w, w.bias)
        assert torch.equal(packed[r0:r0 + L].view(torch.int16), alone.view(torch.int16)), L
        r0 += L


def test_row_offset_does_not_change_bits(pv):
    # the same rows at every offset within a 256-row pair tile give the same
    # bits (a shift of 128 moves a row from one CTA of the pair to the other)
    w = workloads.linear_case([400], 512, 256, seed=8)
    base = _run(pv, w.x, w.w, w.bias)
    for shift in (1, 5, 64, 127, 128, 200, 255, 256):
        moved = _run(pv, w.x[shift:].contiguous(), w.w, w.bias)
        assert torch.equal(moved.view(torch.int16), base[shift:].view(torch.int16)), shift


def test_repeatable_and_guard_band(pv):
    w = workloads.linear_case([333], 264, 136, seed=9)
    x, wt, b = w.x.cuda(), w.w.cuda(), w.bias.cuda()
    buf = torch.full((333 * 264 + 64,), 5.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:333 * 264].view(333, 264)
    pv.linear_bf16(x, wt, b, out=out)
    y2 = pv.linear_bf16(x, wt, b)
    torch.cuda.synchronize()
    assert (buf[333 * 264:].float() == 5.0).all()
    assert torch.equal(out.cpu().view(torch.int16), y2.cpu().view(torch.int16))


def test_zero_rows_is_a_no_op(pv):
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(16, 64, dtype=torch.bfloat16, device="cuda")
    y = pv.linear_bf16(x, w)
    torch.cuda.synchronize()
    assert y.shape == (0, 16)


@pytest.mark.parametrize("kind", ["qkv", "out"])
def test_mmdit_projection_full_size(pv, kind):
    # the full mixed-resolution batch: sampled rows against the oracle (tile
    # edges, request edges, the last row) and every request bit-identical alone
    w = workloads.mmdit_projection(kind)
    x, wt, b = w.x.cuda(), w.w.cuda(), w.bias.cuda()
    y = pv.linear_bf16(x, wt, b)
    torch.cuda.synchronize()
    cu = np.cumsum([0] + w.lengths)
    rows = sorted(set([0, 1, 127, 128, 255, 256, w.M - 1] + [int(c) for c in cu[1:-1]] +
                      [int(c) - 1 for c in cu[1:]] +
                      np.random.default_rng(0).integers(0, w.M, 24).tolist()))
    _check(y[torch.as_tensor(rows)].cpu(), w.x, w.w, w.bias, rows=rows)
    for bi, L in enumerate(w.lengths):
        alone = pv.linear_bf16(x[cu[bi]:cu[bi + 1]].contiguous(), wt, b)
        torch.cuda.synchronize()
        assert torch.equal(y[cu[bi]:cu[bi + 1]].view(torch.int16), alone.view(torch.int16))
    assert pv.get_device_status() == 0
