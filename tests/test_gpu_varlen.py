"""Parity of the CUDA varlen attention path with the fp64 oracle, through the
C ABI, plus the packed-vs-alone bit identity the pages require."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close_to_oracle, gpu_varlen, item_rows, items_covered, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pv():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()  # clear any earlier record
    return pv


def _check_full(pv, w, what):
    out, cu_q, cu_k = gpu_varlen(pv, w)
    ocq = oracle.cu_seqlens_from_lengths(w.lengths_q)
    ock = oracle.cu_seqlens_from_lengths(w.lengths_k)
    assert np.array_equal(cu_q.numpy(), ocq) and np.array_equal(cu_k.numpy(), ock)
    want = oracle.varlen_attention(w.q, w.k, w.v, ocq, ock, w.scale)
    T = int(ocq[-1])
    got = oracle.to_f64(out)
    assert_close_to_oracle(got[:T], want[:T], what)
    assert np.isnan(got[T:]).all(), "rows outside every sequence were written"
    assert pv.get_device_status() == 0


def test_tiny_config(pv):
    _check_full(pv, workloads.tiny(), "tiny")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [
    [1], [127], [128], [129], [300, 17, 256, 1],        # tails around the 128-row tile
    [0, 200, 0, 5],                                      # empty sequences
    [513, 1000],                                         # several tiles, ragged
])
def test_random_self_attention(pv, D, lengths):
    w = workloads.random_varlen(lengths, None, 3, D, seed=sum(lengths) + D)
    _check_full(pv, w, f"L={lengths} D={D}")


@pytest.mark.parametrize("lq,lk", [([5, 300, 128], [400, 7, 128]), ([200, 3], [0, 260])])
def test_cross_lengths_and_empty_keys(pv, lq, lk):
    w = workloads.random_varlen(lq, lk, 2, 128, seed=99)
    _check_full(pv, w, f"Lq={lq} Lk={lk}")


@pytest.mark.parametrize("D", [64, 128])
def test_many_sequences(pv, D):
    # a long work list of short and empty sequences: many items per CTA (pair),
    # single-tile items, items without keys between items with keys
    rng = np.random.default_rng(7)
    L = rng.integers(0, 200, size=300).tolist()
    w = workloads.random_varlen(L, None, 2, D, seed=8)
    _check_full(pv, w, f"300 sequences D={D}")


def test_every_item_single_tile(pv):
    # no sequence reaches a second 128-row tile: the odd CTA of each pair
    # computes only rows past its item and stores none, and every item has a
    # single key tile
    w = workloads.random_varlen([100, 50, 128, 7, 64, 128, 1], None, 3, 128, seed=12)
    _check_full(pv, w, "single-tile items")


@pytest.mark.parametrize("D", [64, 128])
def test_max_batch(pv, D):
    L = ([1, 2, 0, 130] * 256)[:1024]
    w = workloads.random_varlen(L, None, 1, D, seed=9)
    _check_full(pv, w, f"1024 sequences D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_rescale_on_growing_scores(pv, D):
    # Key rows grow with their key tile, so the row maximum jumps by far more
    # than 2^8 between tiles and O is rescaled on most tiles (including a
    # sequence's last tile and the last tiles of a CTA's stream); the tile
    # order starts at a rotated tile, so maxima also stay flat for a while.
    L = [700, 1300, 260]
    w = workloads.random_varlen(L, None, 2, D, seed=21)
    k = w.k.float()
    start = 0
    for n in L:
        grow = 1.0 + 1.5 * (torch.arange(n, dtype=torch.float32) // 128)
        k[start:start + n] *= grow[:, None, None]
        start += n
    w.k = k.to(torch.bfloat16)
    for scale in (0.3, None):
        out, _, _ = gpu_varlen(pv, w, scale=scale)
        cu = oracle.cu_seqlens_from_lengths(w.lengths_q)
        sc = w.scale if scale is None else scale
        want = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, sc)
        assert_close_to_oracle(oracle.to_f64(out), want, f"growing scores D={D} scale={sc}")


def test_scale_argument(pv):
    w = workloads.random_varlen([150, 40], None, 2, 128, seed=11)
    for scale in (0.0, 0.02, 0.3, -0.1):   # negative: the scaled-first softmax path
        out, _, _ = gpu_varlen(pv, w, scale=scale)
        cu = oracle.cu_seqlens_from_lengths(w.lengths_q)
        want = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, scale)
        assert_close_to_oracle(oracle.to_f64(out), want, f"scale={scale}")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixed_res_mmdit", "single_edit", "cfg_dynamic_batch"])
def test_full_size_configs_every_item(pv, name):
    # one query row of every 128-row tile of every sequence, all heads: every
    # (sequence, head, 256-row work item) the scheduler hands out, and both
    # of its tiles, is compared with the oracle
    w = workloads.VARLEN_CONFIGS[name]()
    out, cu_q, _ = gpu_varlen(pv, w)
    rows = item_rows(w.lengths_q, seed=1)
    got_items, want_items = items_covered(rows, w.lengths_q)
    assert got_items == want_items
    cu = oracle.cu_seqlens_from_lengths(w.lengths_q)
    want = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, w.scale, rows=rows)
    assert_close_to_oracle(oracle.to_f64(out[rows]), want, name)
    assert pv.get_device_status() == 0


@pytest.mark.slow
def test_padded_tail_equals_masked_oracle(pv):
    # 7 auto-padded rows after the edit request: trimmed by cu_seqlens, never
    # read as keys, never written; equal to the key-padding-masked oracle
    w = workloads.single_edit(pad_rows=7)
    T = sum(w.lengths_q)
    out, _, _ = gpu_varlen(pv, w)
    assert out.shape[0] == T + 7
    assert torch.isnan(out[T:].float()).all()
    rows = sample_rows(w.lengths_q, per_seq=8, seed=2)
    want = oracle.key_padding_attention(w.q, w.k, w.v, T, w.scale, rows=rows)
    assert_close_to_oracle(oracle.to_f64(out[rows]), want, "padded tail")


def _alone(pv, w, b):
    s0, s1 = sum(w.lengths_q[:b]), sum(w.lengths_q[:b + 1])
    k0, k1 = sum(w.lengths_k[:b]), sum(w.lengths_k[:b + 1])
    one = workloads.VarlenWorkload("one", [w.lengths_q[b]], [w.lengths_k[b]], w.H, w.D,
                                   w.q[s0:s1].clone(), w.k[k0:k1].clone(), w.v[k0:k1].clone(),
                                   w.seed)
    out, _, _ = gpu_varlen(pv, one)
    return out


@pytest.mark.parametrize("name", ["mixed_res_mmdit", "small"])
def test_packed_bit_identical_to_alone(pv, name):
    if name == "small":
        w = workloads.random_varlen([300, 1, 129, 64, 700], None, 4, 128, seed=12)
    else:
        w = workloads.mixed_res()
    packed, _, _ = gpu_varlen(pv, w)
    start = 0
    for b, L in enumerate(w.lengths_q):
        alone = _alone(pv, w, b)
        assert torch.equal(packed[start:start + L].view(torch.int16), alone.view(torch.int16)), \
            f"sequence {b} differs packed vs alone"
        start += L


def test_request_permutation_bit_identical(pv):
    w = workloads.random_varlen([200, 333, 64, 129], None, 2, 128, seed=13)
    base, _, _ = gpu_varlen(pv, w)
    perm = [3, 1, 0, 2]
    cu = [0]
    for L in w.lengths_q:
        cu.append(cu[-1] + L)
    segs = [slice(cu[b], cu[b + 1]) for b in perm]
    wp = workloads.VarlenWorkload("perm", [w.lengths_q[b] for b in perm],
                                  [w.lengths_k[b] for b in perm], w.H, w.D,
                                  torch.cat([w.q[s] for s in segs]),
                                  torch.cat([w.k[s] for s in segs]),
                                  torch.cat([w.v[s] for s in segs]), w.seed)
    got, _, _ = gpu_varlen(pv, wp)
    want = torch.cat([base[s] for s in segs])
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_device_checks_record_errors(pv):
    dev = "cuda"
    q = torch.randn(64, 2, 64, device=dev).to(torch.bfloat16)
    out = torch.full_like(q, 3.0)
    bad = torch.tensor([0, 40, 30], dtype=torch.int32, device=dev)   # decreasing
    pv.varlen_attn_fwd(q, q, q, bad, bad, 64, 64, out=out)
    assert pv.get_device_status() == 1
    assert (out[40:].float() == 3.0).all()   # the bad sequence was skipped
    assert (out[:40].float() != 3.0).any()   # the good one was not
    out.fill_(3.0)
    ok = torch.tensor([0, 40, 64], dtype=torch.int32, device=dev)
    pv.varlen_attn_fwd(q, q, q, ok, ok, 30, 64, out=out)              # 40 > max_q
    assert pv.get_device_status() == 2
    assert (out[:40].float() == 3.0).all()
    assert (out[40:].float() != 3.0).any()
    assert pv.get_device_status() == 0      # cleared by the read


def _poison(t: torch.Tensor, rows: slice) -> torch.Tensor:
    """Copy of t whose given rows hold NaN, +Inf and -Inf in turn (element by
    element), so no finite factor can cancel them."""
    bad = t.clone()
    block = bad[rows]
    vals = torch.tensor([float("nan"), float("inf"), float("-inf")], dtype=t.dtype)
    flat = vals.repeat(block.numel() // 3 + 1)[:block.numel()].view(block.shape)
    bad[rows] = flat
    return bad


@pytest.mark.parametrize("D", [64, 128])
def test_nonfinite_padded_tail(pv, D):
    # The auto-padded tail of "[Perf][qwen-image-edit] Skip attention-mask to
    # avoid varlen path" (Test Result: a 1328x1328 image, 6889 tokens padded
    # to 6896).  6889 = 53 * 128 + 105, so the last key tile loads the 7 pad
    # rows; filled with NaN / +-Inf they must contribute nothing.
    L, T = 6889, 6896
    base = workloads.random_varlen([T], None, 2, D, seed=6889 + D)
    fin = workloads.VarlenWorkload("tail", [L], [L], 2, D, base.q, base.k, base.v, 0, pad_rows=7)
    bad = workloads.VarlenWorkload("tail_nonfinite", [L], [L], 2, D,
                                   _poison(base.q, slice(L, T)), _poison(base.k, slice(L, T)),
                                   _poison(base.v, slice(L, T)), 0, pad_rows=7)
    got_fin, _, _ = gpu_varlen(pv, fin)
    got_bad, _, _ = gpu_varlen(pv, bad)
    assert torch.isnan(got_bad[L:].float()).all(), "pad rows were written"
    assert torch.equal(got_bad[:L].view(torch.int16), got_fin[:L].view(torch.int16)), \
        "non-finite pad rows changed the valid rows"
    # key-padding-masked dense attention over the finite buffer
    want = oracle.key_padding_attention(base.q, base.k, base.v, L, fin.scale,
                                        rows=np.arange(L))
    assert_close_to_oracle(oracle.to_f64(got_bad[:L]), want, f"6889->6896 tail D={D}")
    assert pv.get_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lengths", [[300, 200], [129, 1000, 44]])
def test_nonfinite_neighbour_rows_do_not_leak(pv, D, lengths):
    # The first 127 key/value rows of sequence 1 (and the query rows) are
    # non-finite; sequence 0's last key tile spans some of them.  Sequence 0
    # must still match the oracle and equal its run alone bit for bit.
    w = workloads.random_varlen(lengths, None, 3, D, seed=41 + D)
    s1 = slice(lengths[0], lengths[0] + min(127, lengths[1]))
    bad = workloads.VarlenWorkload("neighbour_nonfinite", w.lengths_q, w.lengths_k, w.H, w.D,
                                   _poison(w.q, s1), _poison(w.k, s1), _poison(w.v, s1), w.seed)
    packed, _, _ = gpu_varlen(pv, bad)
    L0 = lengths[0]
    alone = _alone(pv, w, 0)
    assert torch.equal(packed[:L0].view(torch.int16), alone.view(torch.int16))
    cu = oracle.cu_seqlens_from_lengths(lengths)
    want = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, w.scale, rows=np.arange(L0))
    assert_close_to_oracle(oracle.to_f64(packed[:L0]), want, f"sequence 0 of {lengths}")
    if len(lengths) > 2:   # a sequence after the poisoned one is unaffected too
        s2 = sum(lengths[:2])
        want2 = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, w.scale,
                                        rows=np.arange(s2, s2 + lengths[2]))
        assert_close_to_oracle(oracle.to_f64(packed[s2:s2 + lengths[2]]), want2, "sequence 2")
    assert pv.get_device_status() == 0


@pytest.mark.slow
def test_mixed_batch_every_row_of_two_heads(pv):
    # every query row of heads 0 and 23 of the full mixed-resolution batch
    # against the oracle; heads are independent, so the oracle runs on those
    # two heads' slices of q, k and v
    w = workloads.mixed_res()
    out, cu_q, _ = gpu_varlen(pv, w)
    cu = oracle.cu_seqlens_from_lengths(w.lengths_q)
    heads = [0, w.H - 1]
    want = oracle.varlen_attention(w.q[:, heads], w.k[:, heads], w.v[:, heads], cu, cu, w.scale)
    assert_close_to_oracle(oracle.to_f64(out[:, heads]), want, "mixed batch, heads 0 and 23")
    assert pv.get_device_status() == 0
