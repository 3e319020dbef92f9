"""Bit-exact parity of the integer and copy steps (boundaries, pack, unpack,
work order) with the oracle, through the C ABI."""
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


@pytest.mark.parametrize("lengths", [[37, 64], [0], [5, 0, 9, 1], list(range(2000)),
                                     [16384 + 100, 2304 + 20, 6889 + 255, 4096 + 16]])
def test_cu_seqlens(pv, lengths):
    lt = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    got = pv.cu_seqlens_from_lengths(lt).cpu().numpy()
    assert np.array_equal(got, oracle.cu_seqlens_from_lengths(lengths))
    assert pv.get_device_status() == 0


def test_cu_seqlens_negative_length_recorded(pv):
    lt = torch.tensor([3, -2, 4], dtype=torch.int32, device="cuda")
    got = pv.cu_seqlens_from_lengths(lt).cpu().numpy()
    assert got.tolist() == [0, 3, 3, 7]
    assert pv.get_device_status() == 4


def _i16(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("lengths,H,D", [([5, 0, 9, 1], 2, 64), ([128, 127, 1], 24, 128),
                                         ([300, 300], 1, 8)])
def test_pack_unpack(pv, lengths, H, D):
    pw = workloads.padded(lengths, H, D, seed=sum(lengths))
    cu = pv.cu_seqlens_from_lengths(torch.tensor(lengths, dtype=torch.int32, device="cuda"))
    T = sum(lengths)
    padded = pw.q.cuda()
    flat = pv.pack(padded, cu, T)
    want = oracle.pack(_i16(pw.q), lengths)
    assert np.array_equal(_i16(flat), want)
    # unpack into a buffer whose padding rows hold a sentinel: they stay
    target = torch.full_like(padded, 7.0)
    pv.unpack(flat, cu, target)
    want_pad = oracle.unpack(want, lengths, _i16(torch.full_like(pw.q, 7.0)))
    assert np.array_equal(_i16(target), want_pad)
    assert pv.get_device_status() == 0


def test_pack_full_mixed_res(pv):
    pw = workloads.mixed_res_padded()
    cu = pv.cu_seqlens_from_lengths(torch.tensor(pw.lengths, dtype=torch.int32, device="cuda"))
    T = sum(pw.lengths)
    flat = pv.pack(pw.k.cuda(), cu, T)
    assert np.array_equal(_i16(flat), oracle.pack(_i16(pw.k), pw.lengths))


@pytest.mark.parametrize("lengths,H,D", [
    (np.random.default_rng(3).integers(0, 300, 200).tolist(), 2, 64),   # many sequences
    ([3, 1, 2], 24, 512),                                              # 24 KB rows: one per chunk
])
def test_pack_unpack_chunking(pv, lengths, H, D):
    # the copy is split into chunks of ~16 KB of one sequence's rows; every
    # sequence, chunk tail and row size must land exactly
    pw = workloads.padded(lengths, H, D, seed=len(lengths))
    cu = pv.cu_seqlens_from_lengths(torch.tensor(lengths, dtype=torch.int32, device="cuda"))
    T = sum(lengths)
    flat = pv.pack(pw.q.cuda(), cu, T)
    want = oracle.pack(_i16(pw.q), lengths)
    assert np.array_equal(_i16(flat), want)
    target = torch.full_like(pw.q, 3.0).cuda()
    pv.unpack(flat, cu, target)
    assert np.array_equal(_i16(target), oracle.unpack(want, lengths, _i16(torch.full_like(pw.q, 3.0))))
    assert pv.get_device_status() == 0


def test_pack_skips_only_the_bad_sequence(pv):
    # sequence 1 ends past `total`: it is skipped and reported, sequence 0 is copied
    padded = torch.arange(2 * 8 * 8, dtype=torch.float32).to(torch.bfloat16).view(2, 8, 8).cuda()
    cu = torch.tensor([0, 3, 9], dtype=torch.int32, device="cuda")
    flat = torch.full((7, 8), -1.0, dtype=torch.bfloat16, device="cuda")
    pv.pack(padded, cu, 7, out=flat)
    assert pv.get_device_status() == 1   # PA_DEVICE_ERR_CU_SEQLENS
    assert torch.equal(flat[:3].cpu(), padded[0, :3].cpu())
    assert (flat[3:].float() == -1.0).all()


def test_pack_rejects_long_sequence(pv):
    padded = torch.zeros(2, 4, 8, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 5, 7], dtype=torch.int32, device="cuda")   # 5 > s_max = 4
    flat = torch.full((7, 8), 2.0, dtype=torch.bfloat16, device="cuda")
    pv.pack(padded, cu, 7, out=flat)
    assert pv.get_device_status() == 2
    assert (flat[:5].float() == 2.0).all() and (flat[5:].float() == 0.0).all()


@pytest.mark.parametrize("lq,lk,H", [([37, 64], [37, 64], 2), ([0, 129, 128, 1, 500], None, 3),
                                     ([5, 300], [400, 0], 4)])
def test_work_order(pv, lq, lk, H):
    lk = lq if lk is None else lk
    cu_q = torch.tensor(oracle.cu_seqlens_from_lengths(lq), device="cuda")
    cu_k = torch.tensor(oracle.cu_seqlens_from_lengths(lk), device="cuda")
    want = oracle.work_order(lq, lk, H, pv.VARLEN_TILE_M)
    got = pv.varlen_work_order(cu_q, cu_k, H, len(want))
    assert [tuple(r) for r in got.cpu().tolist()] == want
    assert pv.get_device_status() == 0


def test_work_order_large_batch(pv):
    rng = np.random.default_rng(3)
    lq = rng.integers(0, 700, size=1024).tolist()
    lk = rng.integers(0, 50, size=1024).tolist()   # many ties
    cu_q = torch.tensor(oracle.cu_seqlens_from_lengths(lq), device="cuda")
    cu_k = torch.tensor(oracle.cu_seqlens_from_lengths(lk), device="cuda")
    want = oracle.work_order(lq, lk, 2, pv.VARLEN_TILE_M)
    got = pv.varlen_work_order(cu_q, cu_k, 2, len(want))
    assert [tuple(r) for r in got.cpu().tolist()] == want


def test_work_order_capacity(pv):
    cu = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    got = pv.varlen_work_order(cu, cu, 2, 4, tile_m=128)
    assert got.cpu().tolist() == [[0, 0, 0], [0, 0, 1], [0, 0, 2], [0, 1, 0]]
    assert pv.get_device_status() == 5
