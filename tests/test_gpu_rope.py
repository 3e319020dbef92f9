"""Parity of the CUDA request-local RoPE with the fp64 oracle, through the C ABI."""
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


def _check(got, want, x):
    """Within one bf16 rounding of a result computed to ~1e-6 of its pair's norm."""
    g = oracle.to_f64(got)
    xx = oracle.to_f64(x)
    pair = np.repeat(np.hypot(xx[..., 0::2], xx[..., 1::2]), 2, axis=-1)
    bound = 2.0 ** -8 * np.abs(want) + 1e-5 * pair
    excess = np.abs(g - want) - bound
    assert excess.max() <= 0, f"max excess {excess.max():.3e}"


def _run(pv, w, pos_offset=None, base=1e4, extra_rows=0):
    dev = "cuda"
    cu_q = pv.cu_seqlens_from_lengths(torch.tensor(w.lengths_q, dtype=torch.int32, device=dev))
    cu_k = pv.cu_seqlens_from_lengths(torch.tensor(w.lengths_k, dtype=torch.int32, device=dev))
    q = torch.cat([w.q, torch.full((extra_rows, w.H, w.D), 3.0).to(torch.bfloat16)]).to(dev)
    k = torch.cat([w.k, torch.full((extra_rows, w.H, w.D), 3.0).to(torch.bfloat16)]).to(dev)
    po = None if pos_offset is None else torch.tensor(pos_offset, dtype=torch.int32, device=dev)
    pv.rope_packed(q, k, cu_q, cu_k, po, base)
    torch.cuda.synchronize()
    return q.cpu(), k.cpu()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths,offsets", [([37, 64], None), ([0, 300, 1, 129], [5, 0, 77, 2]),
                                             ([1000], [250])])
def test_against_oracle(pv, D, lengths, offsets):
    w = workloads.random_varlen(lengths, None, 3, D, seed=D + len(lengths))
    q, k = _run(pv, w, offsets, extra_rows=4)
    T = sum(lengths)
    pos = oracle.rope_positions(lengths, offsets)
    _check(q[:T], oracle.rope(w.q, pos, 1e4), w.q)
    _check(k[:T], oracle.rope(w.k, pos, 1e4), w.k)
    assert (q[T:].float() == 3.0).all() and (k[T:].float() == 3.0).all()
    assert pv.get_device_status() == 0


def test_cross_lengths_and_base(pv):
    w = workloads.random_varlen([10, 200], [300, 7], 2, 64, seed=3)
    q, k = _run(pv, w, [1, 2], base=500.0)
    _check(q, oracle.rope(w.q, oracle.rope_positions(w.lengths_q, [1, 2]), 500.0), w.q)
    _check(k, oracle.rope(w.k, oracle.rope_positions(w.lengths_k, [1, 2]), 500.0), w.k)


def test_large_positions(pv):
    # exact angle reduction keeps positions around 10^6 accurate
    w = workloads.random_varlen([256], None, 2, 128, seed=4)
    q, _ = _run(pv, w, [1_000_000])
    _check(q, oracle.rope(w.q, oracle.rope_positions([256], [1_000_000]), 1e4), w.q)


def test_packed_equals_alone_bitwise(pv):
    w = workloads.random_varlen([130, 64, 257], None, 4, 128, seed=5)
    q, k = _run(pv, w, [3, 0, 11])
    one = workloads.VarlenWorkload("one", [257], [257], 4, 128, w.q[194:].clone(),
                                   w.k[194:].clone(), w.v[194:].clone(), 5)
    q1, k1 = _run(pv, one, [11])
    assert torch.equal(q[194:].view(torch.int16), q1.view(torch.int16))
    assert torch.equal(k[194:].view(torch.int16), k1.view(torch.int16))


def test_bad_boundaries_recorded(pv):
    q = torch.zeros(20, 2, 64, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 15, 10], dtype=torch.int32, device="cuda")
    pv.rope_packed(q, q.clone(), cu, cu)
    assert pv.get_device_status() == 1
