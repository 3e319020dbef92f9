"""Parity of the CUDA segment-aware unpack + CFG combine with the fp64 oracle,
through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

# fp32 arithmetic rounded once to bf16: within one bf16 ulp (2^-7 relative)
REL_TOL = 2.0 ** -7


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    return pv


def _gpu(pv, seg, out_fill=None):
    dev = "cuda"
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=dev)
    cu = pv.cu_seqlens_from_lengths(i32(seg.lengths))
    out = None
    if out_fill is not None:
        out = torch.full((len(seg.pos_seq), seg.img_max) + tuple(seg.flat.shape[1:]), out_fill,
                         dtype=torch.bfloat16, device=dev)
    out = pv.cfg_combine(seg.flat.to(dev), cu, i32(seg.text), i32(seg.pos_seq),
                         i32(seg.neg_seq), torch.tensor(seg.cfg_scale, device=dev),
                         i32(seg.cfg_normalize), seg.img_max, out=out)
    torch.cuda.synchronize()
    return out.cpu()


def _check(got, want, what):
    g = oracle.to_f64(got)
    err = np.abs(g - want)
    bound = REL_TOL * np.abs(want) + 1e-6
    worst = float((err - bound).max())
    assert worst <= 0, f"{what}: max excess {worst:.3e}, max err {err.max():.3e}"


def _small(C, normalize):
    lengths = [9, 7, 30, 20, 5, 130, 129]
    text = [3, 1, 10, 0, 2, 2, 1]          # image rows: 6, 6, 20, 20, 3, 128, 128
    seg = workloads.CfgSegments(lengths, text, [0, 2, 4, 5], [1, 3, -1, 6],
                                [2.0, 7.0, 3.0, 4.5], [normalize, 0, 0, normalize],
                                None, 128)
    g = torch.Generator().manual_seed(C + normalize)
    seg.flat = torch.randn(sum(lengths), C, generator=g).to(torch.bfloat16)
    return seg


@pytest.mark.parametrize("C", [8, 64, 136, 256, 1000, 3072])
@pytest.mark.parametrize("normalize", [0, 1])
def test_small_layouts(pv, C, normalize):
    # rows of 1, 8, 17, 32, 125 and 384 sixteen-byte vectors: several rows per
    # warp, one row per warp with fewer vectors than lanes, exactly one vector
    # per lane, and ragged last batches of the four vectors a lane loads at once
    seg = _small(C, normalize)
    got = _gpu(pv, seg, out_fill=5.0)
    want = oracle.cfg_combine(seg.flat, seg.lengths, seg.text, seg.pos_seq, seg.neg_seq,
                              seg.cfg_scale, seg.cfg_normalize, seg.img_max,
                              out_init=np.full((4, 128, C), 5.0))
    _check(got, want, f"C={C} normalize={normalize}")
    assert pv.get_device_status() == 0


@pytest.mark.slow
@pytest.mark.parametrize("normalize_every", [0, 3])
def test_cfg_batch_layout(pv, normalize_every):
    seg = workloads.cfg_segments(C=64, normalize_every=normalize_every)
    got = _gpu(pv, seg)
    want = oracle.cfg_combine(seg.flat, seg.lengths, seg.text, seg.pos_seq, seg.neg_seq,
                              seg.cfg_scale, seg.cfg_normalize, seg.img_max)
    _check(got, want, "cfg batch")


def test_no_cfg_rows_copied_bit_exact(pv):
    seg = _small(64, 0)
    got = _gpu(pv, seg)
    starts = np.concatenate([[0], np.cumsum(seg.lengths)])
    p = seg.pos_seq[2]               # request 2 has no negative pass
    n = seg.lengths[p] - seg.text[p]
    src = seg.flat[starts[p] + seg.text[p]:starts[p] + seg.text[p] + n]
    assert torch.equal(got[2, :n].view(torch.int16), src.view(torch.int16))


def test_packed_equals_request_alone(pv):
    seg = _small(64, 1)
    full = _gpu(pv, seg)
    starts = np.concatenate([[0], np.cumsum(seg.lengths)])
    alone = workloads.CfgSegments(seg.lengths[5:7], seg.text[5:7], [0], [1], [4.5], [1],
                                  seg.flat[starts[5]:starts[7]].clone(), 128)
    one = _gpu(pv, alone)
    assert torch.equal(full[3].view(torch.int16), one[0].view(torch.int16))


def test_bad_segments_recorded_and_skipped(pv):
    seg = _small(8, 0)
    seg.neg_seq = [1, 4, -1, 6]      # request 1: 20 positive vs 3 negative image rows
    got = _gpu(pv, seg, out_fill=9.0)
    assert pv.get_device_status() == 7
    assert (got[1].float() == 9.0).all()
    assert not (got[0, :6].float() == 9.0).all()
