"""Parity of the CUDA block-window attention with the dense block-difference
mask oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close_to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    return pv


def _run(pv, w, lb, la):
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    out = pv.block_window_attn_fwd(q, k, v, w.block, lb, la, scale=w.scale)
    torch.cuda.synchronize()
    return out.cpu()


LOOKS = [(0, 0), (1, 0), (0, 1), (1, 1), (2, 3)]


@pytest.mark.parametrize("n", [10, 24, 96, 101])
@pytest.mark.parametrize("look", LOOKS)
def test_pages_unit_cases(pv, n, look):
    # shorter than a block, exactly one block, whole blocks, a partial last block
    w = workloads.random_block_window(1, n, 4, 64, 24, seed=n + 10 * look[0] + look[1])
    got = oracle.to_f64(_run(pv, w, *look))
    want = oracle.block_window_attention(w.q, w.k, w.v, 24, look[0], look[1], w.scale)
    assert_close_to_oracle(got, want, f"n={n} look={look}")


@pytest.mark.parametrize("n", [2400, 2390])
@pytest.mark.parametrize("look", [(0, 0), (1, 1)])
def test_token2wav_config(pv, n, look):
    w = workloads.token2wav(n=n)
    got = oracle.to_f64(_run(pv, w, *look))
    want = oracle.block_window_attention(w.q, w.k, w.v, w.block, look[0], look[1], w.scale)
    assert_close_to_oracle(got, want, f"token2wav n={n} look={look}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("block,D", [(1, 64), (7, 128), (64, 64), (200, 128), (24, 128), (13, 64)])
def test_other_blocks_and_head_dims(pv, block, D):
    w = workloads.random_block_window(2, 333, 3, D, block, seed=block + D)
    for lb, la in [(0, 0), (1, 2), (4, 0)]:
        got = oracle.to_f64(_run(pv, w, lb, la))
        want = oracle.block_window_attention(w.q, w.k, w.v, block, lb, la, w.scale)
        assert_close_to_oracle(got, want, f"block={block} D={D} look=({lb},{la})")


def test_block_one_returns_values(pv):
    # block 1, no neighbours: every query sees only its own key, out = v
    w = workloads.random_block_window(1, 77, 2, 64, 1, seed=5)
    got = _run(pv, w, 0, 0)
    assert torch.equal(got.view(torch.int16), w.v.view(torch.int16))


def test_window_keys_outside_do_not_matter(pv):
    w = workloads.random_block_window(1, 96, 2, 64, 24, seed=6)
    base = _run(pv, w, 1, 0)
    k2, v2 = w.k.clone(), w.v.clone()
    k2[0, 48:] = 100.0
    v2[0, 48:] = -100.0
    w2 = workloads.BlockWindowWorkload("p", 1, 96, 2, 64, 24, [(1, 0)], w.q, k2, v2, 6)
    pert = _run(pv, w2, 1, 0)
    assert torch.equal(base[0, :48].view(torch.int16), pert[0, :48].view(torch.int16))


def test_graph_replay_matches_eager(pv):
    # the 22 Token2Wav layers captured in a CUDA graph give the eager launches' bits
    w = workloads.token2wav(n=480)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    eager = [pv.block_window_attn_fwd(q, k, v, w.block, lb, la) for lb, la in w.layers]
    outs = [torch.empty_like(q) for _ in w.layers]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for o, (lb, la) in zip(outs, w.layers):
            pv.block_window_attn_fwd(q, k, v, w.block, lb, la, out=o)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("n,look", [(2390, (1, 1)), (101, (0, 0)), (333, (1, 2))])
def test_batch_entries_do_not_leak(pv, D, n, look):
    # entry 1 is all NaN / +-Inf: entry 0 (whose last blocks end where entry
    # 1 begins in memory) must equal its run alone bit for bit and the oracle
    w = workloads.random_block_window(2, n, 2, D, 24, seed=n + D)
    bad = [t.clone() for t in (w.q, w.k, w.v)]
    vals = torch.tensor([float("nan"), float("inf"), float("-inf")], dtype=torch.bfloat16)
    for t in bad:
        t[1] = vals.repeat(t[1].numel() // 3 + 1)[:t[1].numel()].view(t[1].shape)
    w2 = workloads.BlockWindowWorkload("poisoned", 2, n, 2, D, 24, [look], *bad, w.seed)
    got = _run(pv, w2, *look)
    one = workloads.BlockWindowWorkload("alone", 1, n, 2, D, 24, [look], w.q[:1].contiguous(),
                                        w.k[:1].contiguous(), w.v[:1].contiguous(), w.seed)
    alone = _run(pv, one, *look)
    assert torch.equal(got[0].view(torch.int16), alone[0].view(torch.int16))
    want = oracle.block_window_attention(w.q[:1], w.k[:1], w.v[:1], 24, look[0], look[1],
                                         w.scale)
    assert_close_to_oracle(oracle.to_f64(got[:1]), want, f"entry 0 n={n} look={look} D={D}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("block,n,look", [(24, 2400, (0, 0)), (24, 2400, (1, 1)),
                                          (128, 1000, (1, 1)), (300, 1200, (0, 1)),
                                          (5, 700, (9, 0))])
def test_window_shapes_against_oracle(pv, block, n, look):
    # single-chunk and multi-chunk windows (a window above 256 keys is taken
    # in 256-key chunks with an online softmax), H = 16 like the DiT
    w = workloads.random_block_window(1, n, 16, 64, block, seed=block * 7 + n)
    got = oracle.to_f64(_run(pv, w, *look))
    want = oracle.block_window_attention(w.q, w.k, w.v, block, look[0], look[1], w.scale)
    assert_close_to_oracle(got, want, f"block={block} n={n} look={look}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("block,n,look,D", [(20, 507, (0, 0), 64), (28, 333, (0, 0), 128),
                                            (32, 300, (0, 0), 64), (24, 250, (0, 0), 64),
                                            (20, 507, (1, 0), 64)])
def test_one_window_path_edges(pv, block, n, look, D):
    # A warp whose rows share one key interval that starts on an 8-column
    # boundary and is at most 32 keys wide reads exactly that interval; here
    # intervals that end inside an 8-column group (20- and 28-frame blocks, a
    # window clipped at n), that start off an 8-column boundary (so the warp
    # takes the masked path beside warps that take the exact one), that are
    # exactly 32 wide, and that are wider than 32 (the masked path only)
    w = workloads.random_block_window(2, n, 3, D, block, seed=block * 3 + n)
    got = oracle.to_f64(_run(pv, w, *look))
    want = oracle.block_window_attention(w.q, w.k, w.v, block, look[0], look[1], w.scale)
    assert_close_to_oracle(got, want, f"block={block} n={n} look={look} D={D}")
    assert pv.get_device_status() == 0


def test_chained_layers_respect_stream_order(pv):
    # The kernel is launched so that it may start while the previous kernel
    # on the stream drains; its copies and stores must still wait for that
    # kernel.  Layer i reads layer i-1's output (read after write), and in
    # the second chain each layer writes over the buffer the previous layer
    # read (write after read).  No host sync between launches; the result
    # must equal the same chain run with a sync after every launch.
    w = workloads.token2wav(n=2400)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    looks = [(0, 0), (1, 1), (0, 0), (1, 1), (0, 0)]

    def chain(sync):
        x = q.clone()
        for lb, la in looks:
            x = pv.block_window_attn_fwd(x, k, v, w.block, lb, la)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return x

    def chain_in_place(sync):
        a, b = q.clone(), torch.empty_like(q)
        for lb, la in looks:
            pv.block_window_attn_fwd(a, k, v, w.block, lb, la, out=b)
            a, b = b, a   # the next layer writes over the buffer just read
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return a

    assert torch.equal(chain(False).view(torch.int16), chain(True).view(torch.int16))
    assert torch.equal(chain_in_place(False).view(torch.int16),
                       chain_in_place(True).view(torch.int16))
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_multi_chunk_rescale_on_growing_scores(pv, D):
    # windows of up to 700 keys are taken in 256-key chunks; keys of later
    # chunks are scaled up so that rows' maxima grow from chunk to chunk and
    # the running output (in TMEM at D = 128, in registers at D = 64) is
    # rescaled before each later chunk's PV
    w = workloads.random_block_window(1, 700, 2, D, 100, seed=77 + D)
    k = w.k.clone()
    grow = (1.0 + 1.5 * (torch.arange(700) // 256).float()).to(torch.bfloat16)
    k = (k.float() * grow.float()[None, :, None, None]).to(torch.bfloat16)
    w2 = workloads.BlockWindowWorkload("growing", 1, 700, 2, D, 100, [(3, 3)], w.q, k, w.v, w.seed)
    for lb, la in [(3, 3), (6, 0), (0, 6)]:
        got = oracle.to_f64(_run(pv, w2, lb, la))
        want = oracle.block_window_attention(w.q, k, w.v, 100, lb, la, w.scale)
        assert_close_to_oracle(got, want, f"D={D} look=({lb},{la})")
    assert pv.get_device_status() == 0
