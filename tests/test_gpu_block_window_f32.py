"""Parity of the fp32 block-window attention with the fp64 dense
block-difference mask oracle, through the C ABI.

The bound is the one the pages saw between the fp32 block-local and the fp32
dense masked attention of the Token2Wav DiT: 6e-6 ("[Perf][Model] Use
block-sparse attention in Qwen2.5-Omni Token2Wav DiT", Test Result).  With
unit-normal inputs an fp32 result carries a few 1e-7 of rounding (64-term dot
products, exp, a 24-72-term weighted sum), so the max-abs bound is 6e-6 and
the mean-abs bound 5e-7.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

MAX_ABS = 6e-6
MEAN_ABS = 5e-7


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    return pv


def _run(pv, w, lb, la):
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    out = pv.block_window_attn_fwd_f32(q, k, v, w.block, lb, la, scale=w.scale)
    torch.cuda.synchronize()
    return out.cpu()


def _close(got, want, what):
    err = np.abs(oracle.to_f64(got) - want)
    assert np.isfinite(oracle.to_f64(got)).all(), what
    assert err.max() <= MAX_ABS, f"{what}: max abs {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs {err.mean():.3e}"


LOOKS = [(0, 0), (1, 0), (0, 1), (1, 1), (2, 3)]


@pytest.mark.parametrize("n", [1, 10, 24, 96, 101])
@pytest.mark.parametrize("look", LOOKS)
def test_pages_unit_cases(pv, n, look):
    # one frame, shorter than a block, one block, whole blocks, a partial last block
    w = workloads.random_block_window_f32(1, n, 4, 64, 24, seed=n + 10 * look[0] + look[1])
    want = oracle.block_window_attention(w.q, w.k, w.v, 24, look[0], look[1], w.scale)
    _close(_run(pv, w, *look), want, f"n={n} look={look}")


@pytest.mark.parametrize("n", [2400, 2390])
@pytest.mark.parametrize("look", [(0, 0), (1, 1)])
def test_token2wav_cfg_batch(pv, n, look):
    w = workloads.token2wav_f32(n=n)
    want = oracle.block_window_attention(w.q, w.k, w.v, w.block, look[0], look[1], w.scale)
    _close(_run(pv, w, *look), want, f"token2wav f32 n={n} look={look}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("block,D", [(1, 64), (7, 128), (64, 64), (200, 128), (24, 128),
                                     (13, 64)])
def test_other_blocks_and_head_dims(pv, block, D):
    w = workloads.random_block_window_f32(2, 333, 3, D, block, seed=block + D)
    for lb, la in [(0, 0), (1, 2), (4, 0)]:
        want = oracle.block_window_attention(w.q, w.k, w.v, block, lb, la, w.scale)
        _close(_run(pv, w, lb, la), want, f"block={block} D={D} look=({lb},{la})")


def test_window_covers_everything_is_dense(pv):
    # look-back and look-ahead past both ends: plain dense attention
    w = workloads.random_block_window_f32(1, 150, 2, 128, 24, seed=9)
    for h in range(2):
        dense = oracle.masked_attention(oracle.to_f64(w.q[0, :, h]), oracle.to_f64(w.k[0, :, h]),
                                        oracle.to_f64(w.v[0, :, h]),
                                        np.ones((150, 150), dtype=bool), w.scale)
        got = _run(pv, w, 100, 100)[0, :, h]
        err = np.abs(oracle.to_f64(got) - dense)
        assert err.max() <= MAX_ABS


def test_cfg_rows_match_single_batch_bitwise(pv):
    # batch 2 (CFG) gives each entry exactly what a batch-1 call gives it
    w = workloads.token2wav_f32(n=480)
    both = _run(pv, w, 1, 1)
    for b in range(2):
        one = workloads.BlockWindowWorkload("one", 1, 480, 16, 64, 24, [(1, 1)],
                                            w.q[b:b + 1].clone(), w.k[b:b + 1].clone(),
                                            w.v[b:b + 1].clone(), 0)
        assert torch.equal(both[b:b + 1].view(torch.int32), _run(pv, one, 1, 1).view(torch.int32))


def test_repeatable_with_guard_band(pv):
    w = workloads.random_block_window_f32(2, 257, 4, 64, 24, seed=11)
    a = _run(pv, w, 1, 1)
    b = _run(pv, w, 1, 1)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # rows outside out's extent are never written: a guard band stays intact
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    buf = torch.full((2 * 257 * 4 * 64 + 64,), 7.0, device="cuda")
    out = buf[:2 * 257 * 4 * 64].view(2, 257, 4, 64)
    pv.block_window_attn_fwd_f32(q, k, v, 24, 1, 1, scale=w.scale, out=out)
    torch.cuda.synchronize()
    assert (buf[2 * 257 * 4 * 64:] == 7.0).all()
    assert torch.equal(out.cpu().view(torch.int32), a.view(torch.int32))


@pytest.mark.parametrize("block,n,look", [(24, 2400, (1, 0)), (20, 507, (0, 0)), (32, 300, (0, 0)),
                                          (16, 300, (1, 1)), (8, 250, (0, 0)), (40, 333, (0, 0)),
                                          (48, 500, (0, 0)), (24, 23, (1, 1))])
def test_block_and_window_shapes(pv, block, n, look):
    # one neighbour block on one side; blocks of 20 frames (a 24-row task
    # split over lanes that cover fewer rows), 32, 16 and 8 frames (several
    # blocks per 32-row span), 40 and 48 frames (tasks of part of a block),
    # and a sequence shorter than its block with neighbours on both sides
    w = workloads.random_block_window_f32(2, n, 3, 64, block, seed=block * 5 + n)
    want = oracle.block_window_attention(w.q, w.k, w.v, block, look[0], look[1], w.scale)
    _close(_run(pv, w, *look), want, f"block={block} n={n} look={look}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("n,look", [(2390, (1, 1)), (101, (0, 0)), (333, (2, 3))])
def test_batch_entries_do_not_leak(pv, n, look):
    # entry 1 is all NaN / +-Inf: entry 0 (whose last rows end where entry 1
    # begins in memory) must equal its run alone bit for bit and the oracle
    w = workloads.random_block_window_f32(2, n, 2, 64, 24, seed=n)
    bad = [t.clone() for t in (w.q, w.k, w.v)]
    vals = torch.tensor([float("nan"), float("inf"), float("-inf")])
    for t in bad:
        t[1] = vals.repeat(t[1].numel() // 3 + 1)[:t[1].numel()].view(t[1].shape)
    w2 = workloads.BlockWindowWorkload("poisoned", 2, n, 2, 64, 24, [look], *bad, w.seed)
    got = _run(pv, w2, *look)
    one = workloads.BlockWindowWorkload("alone", 1, n, 2, 64, 24, [look], w.q[:1].contiguous(),
                                        w.k[:1].contiguous(), w.v[:1].contiguous(), w.seed)
    assert torch.equal(got[0].view(torch.int32), _run(pv, one, *look)[0].view(torch.int32))
    want = oracle.block_window_attention(w.q[:1], w.k[:1], w.v[:1], 24, look[0], look[1], w.scale)
    _close(got[:1], want, f"entry 0 n={n} look={look}")
    assert pv.get_device_status() == 0


def test_chained_layers_respect_stream_order(pv):
    # Each layer reads the previous layer's output (read after write), and in
    # the second chain writes over the buffer the previous layer read (write
    # after read); no host sync between launches.  The result must equal the
    # same chain with a sync after every launch.
    w = workloads.token2wav_f32(n=960)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    looks = [(0, 0), (1, 1), (0, 0), (1, 1), (2, 3), (0, 0)]

    def chain(sync):
        x = q.clone()
        for lb, la in looks:
            x = pv.block_window_attn_fwd_f32(x, k, v, w.block, lb, la)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return x

    def chain_in_place(sync):
        a, b = q.clone(), torch.empty_like(q)
        for lb, la in looks:
            pv.block_window_attn_fwd_f32(a, k, v, w.block, lb, la, out=b)
            a, b = b, a
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return a

    assert torch.equal(chain(False).view(torch.int32), chain(True).view(torch.int32))
    assert torch.equal(chain_in_place(False).view(torch.int32),
                       chain_in_place(True).view(torch.int32))
    assert pv.get_device_status() == 0


def test_graph_replay_matches_eager(pv):
    # the 22 Token2Wav layers captured in a CUDA graph give the eager launches' bits
    w = workloads.token2wav_f32(n=480)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    eager = [pv.block_window_attn_fwd_f32(q, k, v, w.block, lb, la) for lb, la in w.layers]
    outs = [torch.empty_like(q) for _ in w.layers]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for o, (lb, la) in zip(outs, w.layers):
            pv.block_window_attn_fwd_f32(q, k, v, w.block, lb, la, out=o)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("block", [14, 15, 16, 17, 18, 19, 21, 22, 23])
def test_every_partial_stage_length(pv, block):
    # keys come in stages of 12; an own-block window of 14-23 keys leaves
    # 2-11 valid keys in its last stage (and the sequence's last block fewer)
    n = 4 * block + 5
    w = workloads.random_block_window_f32(1, n, 2, 64, block, seed=block)
    for lb, la in [(0, 0), (1, 0)]:
        want = oracle.block_window_attention(w.q, w.k, w.v, block, lb, la, w.scale)
        _close(_run(pv, w, lb, la), want, f"block={block} look=({lb},{la})")
