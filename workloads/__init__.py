"""Seeded synthetic workloads for packed variable-length attention.

This module only draws numbers: sequence lengths and bf16 N(0, 1) tensors of
the shapes the pages' workloads have. It holds none of the method's
arithmetic (no prefix sums, no packing, no attention), so both the CPU oracle
and the CUDA path can take their inputs from here without sharing any of the
computation they are compared on.

Recipe (every draw on the CPU from ``torch.Generator().manual_seed(seed)``):
lengths first, with ``torch.randint`` (inclusive bounds written as
``randint(lo, hi + 1)``), then q, k, v in that order, each
``torch.randn(..., dtype=float32)`` rounded to bf16.

Image token counts are the Qwen-Image latent grid sizes: one token per 16x16
pixel patch, so 768x768 -> 48*48 = 2304, 1024x1024 -> 4096, 1328x1328 -> 6889
and 2048x2048 -> 16384 ("[Perf][qwen-image-edit] Skip attention-mask to avoid
varlen path", Test Result: 16,384 tokens at 2048x2048, 16,384*2 for the edit
model's noise + source latents, 6889 -> 6896 at 1328x1328).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch

# Qwen-Image latent token counts for 768^2, 1024^2, 1328^2 and 2048^2 images.
IMAGE_TOKENS = (2304, 4096, 6889, 16384)


def image_tokens(height: int, width: int, patch: int = 16) -> int:
    """Tokens of a (height x width) image: one per patch x patch pixel tile."""
    return (height // patch) * (width // patch)


@dataclass
class VarlenWorkload:
    """A packed batch: per-sequence query/key lengths and flat bf16 tensors.

    q is [sum(lengths_q), H, D]; k and v are [sum(lengths_k), H, D], with the
    tokens of sequence b stored contiguously in order b = 0, 1, ...  ``pad_rows``
    extra rows (if any) sit after the last sequence and belong to no sequence.
    """
    name: str
    lengths_q: List[int]
    lengths_k: List[int]
    H: int
    D: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seed: int
    pad_rows: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.lengths_q)

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5


@dataclass
class BlockWindowWorkload:
    """Token2Wav-style block-window attention input, layout [batch, n, H, D]."""
    name: str
    batch: int
    n: int
    H: int
    D: int
    block: int
    layers: List[Tuple[int, int]]  # (look_back, look_ahead) per DiT layer
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5


@dataclass
class PaddedWorkload:
    """A padded batch [B, S_max, H, D]: sequence b's real tokens are rows
    [0, lengths[b]) of slot b; the remaining rows are padding."""
    name: str
    lengths: List[int]
    s_max: int
    H: int
    D: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    seed: int


def _randn_bf16(g: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _qkv(g, tq, tk, H, D):
    q = _randn_bf16(g, (tq, H, D))
    k = _randn_bf16(g, (tk, H, D))
    v = _randn_bf16(g, (tk, H, D))
    return q, k, v


# --------------------------------------------------------------------------
# Lengths of the five workloads (drawn first from each workload's generator)
# --------------------------------------------------------------------------

def lengths_tiny() -> List[int]:
    """Two packed sequences of 37 and 64 tokens, H=2, D=64, seed 0."""
    return [37, 64]


def lengths_mixed_res(g: torch.Generator) -> List[int]:
    """Four joint text+image requests: text ~ U[16, 256] + 2304/4096/6889/16384."""
    text = torch.randint(16, 257, (4,), generator=g).tolist()
    return [t + img for t, img in zip(text, IMAGE_TOKENS)]


def lengths_single_edit() -> List[int]:
    """One edit request: 256 text + 2 * 16384 image tokens (noise + source)."""
    return [256 + 2 * 16384]


def lengths_cfg_batch_detail(g: torch.Generator) -> Tuple[List[int], List[int], List[int]]:
    """Eight requests, image tokens chosen uniformly from IMAGE_TOKENS; each
    becomes two sequences (positive text + image, negative text + image) with
    independent text lengths ~ U[8, 256].  Returns (lengths, request index,
    text lengths); sequence 2r is request r's positive pass, 2r + 1 its
    negative pass."""
    img_idx = torch.randint(0, len(IMAGE_TOKENS), (8,), generator=g).tolist()
    text = torch.randint(8, 257, (16,), generator=g).tolist()
    lengths, owner = [], []
    for r in range(8):
        for s in range(2):
            lengths.append(text[2 * r + s] + IMAGE_TOKENS[img_idx[r]])
            owner.append(r)
    return lengths, owner, text


def lengths_cfg_batch(g: torch.Generator) -> Tuple[List[int], List[int]]:
    """(lengths, request index) of the CFG batch; see lengths_cfg_batch_detail."""
    lengths, owner, _ = lengths_cfg_batch_detail(g)
    return lengths, owner


# --------------------------------------------------------------------------
# Full workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> VarlenWorkload:
    g = torch.Generator().manual_seed(seed)
    L = lengths_tiny()
    q, k, v = _qkv(g, sum(L), sum(L), 2, 64)
    return VarlenWorkload("tiny", L, list(L), 2, 64, q, k, v, seed)


def mixed_res(seed: int = 2) -> VarlenWorkload:
    g = torch.Generator().manual_seed(seed)
    L = lengths_mixed_res(g)
    q, k, v = _qkv(g, sum(L), sum(L), 24, 128)
    return VarlenWorkload("mixed_res_mmdit", L, list(L), 24, 128, q, k, v, seed)


def single_edit(seed: int = 3, pad_rows: int = 0) -> VarlenWorkload:
    """The edit request; ``pad_rows`` > 0 adds that many trailing rows that
    belong to no sequence (an auto-padded tail that trimming leaves out)."""
    g = torch.Generator().manual_seed(seed)
    L = lengths_single_edit()
    T = sum(L) + pad_rows
    q, k, v = _qkv(g, T, T, 24, 128)
    return VarlenWorkload("single_edit" + ("_padded_tail" if pad_rows else ""),
                          L, list(L), 24, 128, q, k, v, seed, pad_rows=pad_rows)


def cfg_batch(seed: int = 5) -> VarlenWorkload:
    g = torch.Generator().manual_seed(seed)
    L, owner = lengths_cfg_batch(g)
    q, k, v = _qkv(g, sum(L), sum(L), 24, 128)
    return VarlenWorkload("cfg_dynamic_batch", L, list(L), 24, 128, q, k, v, seed,
                          meta={"request_of_sequence": owner})


TOKEN2WAV_LAYERS = [(0, 0)] * 19 + [(1, 1)] * 3


def token2wav(n: int = 2400, seed: int = 4) -> BlockWindowWorkload:
    """Token2Wav DiT block-window attention: batch 1, H=16, D=64, block 24;
    19 own-block layers and 3 layers with one neighbour block each side."""
    g = torch.Generator().manual_seed(seed)
    shape = (1, n, 16, 64)
    q = _randn_bf16(g, shape)
    k = _randn_bf16(g, shape)
    v = _randn_bf16(g, shape)
    return BlockWindowWorkload("token2wav_block_window", 1, n, 16, 64, 24,
                               list(TOKEN2WAV_LAYERS), q, k, v, seed)


def token2wav_f32(n: int = 2400, seed: int = 6) -> BlockWindowWorkload:
    """The Token2Wav DiT's attention in its own dtype: fp32, classifier-free
    guidance as batch 2 (conditional and unconditional rows), H=16, D=64,
    block 24, the same 22 layers."""
    g = torch.Generator().manual_seed(seed)
    shape = (2, n, 16, 64)
    q = torch.randn(*shape, generator=g, dtype=torch.float32)
    k = torch.randn(*shape, generator=g, dtype=torch.float32)
    v = torch.randn(*shape, generator=g, dtype=torch.float32)
    return BlockWindowWorkload("token2wav_block_window_f32", 2, n, 16, 64, 24,
                               list(TOKEN2WAV_LAYERS), q, k, v, seed)


def random_block_window_f32(batch: int, n: int, H: int, D: int, block: int, seed: int,
                            layers=None) -> BlockWindowWorkload:
    g = torch.Generator().manual_seed(seed)
    shape = (batch, n, H, D)
    q, k, v = (torch.randn(*shape, generator=g, dtype=torch.float32) for _ in range(3))
    return BlockWindowWorkload(f"block_window_f32_n{n}", batch, n, H, D, block,
                               list(layers or [(0, 0)]), q, k, v, seed)


def padded(lengths: List[int], H: int, D: int, seed: int,
           s_max: Optional[int] = None, name: str = "padded") -> PaddedWorkload:
    """Padded [B, S_max, H, D] q/k/v for the given lengths (every row drawn,
    padding rows included)."""
    g = torch.Generator().manual_seed(seed)
    s = max(lengths) if s_max is None else s_max
    B = len(lengths)
    q = _randn_bf16(g, (B, s, H, D))
    k = _randn_bf16(g, (B, s, H, D))
    v = _randn_bf16(g, (B, s, H, D))
    return PaddedWorkload(name, list(lengths), s, H, D, q, k, v, seed)


def mixed_res_padded(seed: int = 2, value_seed: Optional[int] = None) -> PaddedWorkload:
    """The mixed-resolution batch in the padded layout the pack step reads.
    Lengths come from ``seed``; values from ``value_seed`` (default seed + 1000),
    so several ranks can hold batches of one shape with different values."""
    g = torch.Generator().manual_seed(seed)
    L = lengths_mixed_res(g)
    vs = seed + 1000 if value_seed is None else value_seed
    return padded(L, 24, 128, vs, name="mixed_res_mmdit_padded")


def config_lengths(name: str) -> List[int]:
    """Sequence lengths of a named varlen config, drawn exactly as the flat
    workload of that name draws them."""
    if name == "tiny":
        return lengths_tiny()
    if name == "mixed_res_mmdit":
        return lengths_mixed_res(torch.Generator().manual_seed(2))
    if name == "single_edit":
        return lengths_single_edit()
    if name == "cfg_dynamic_batch":
        return lengths_cfg_batch(torch.Generator().manual_seed(5))[0]
    raise KeyError(name)


def varlen_padded(name: str, value_seed: int) -> PaddedWorkload:
    """A named varlen config in the padded [B, S_max, H, D] layout the pack
    step reads, with S_max the longest sequence.  Only real rows are drawn:
    from ``value_seed``, sequence by sequence, the q rows of every sequence,
    then k, then v; padding rows are zero.  (Drawing only the real rows keeps
    the host cost of the 121k-token CFG batch to its 121k rows.)"""
    L = config_lengths(name)
    H, D = (2, 64) if name == "tiny" else (24, 128)
    g = torch.Generator().manual_seed(value_seed)
    s = max(L)
    out = []
    for _ in range(3):
        t = torch.zeros((len(L), s, H, D), dtype=torch.bfloat16)
        for b, n in enumerate(L):
            t[b, :n] = _randn_bf16(g, (n, H, D))
        out.append(t)
    return PaddedWorkload(name + "_padded", list(L), s, H, D, out[0], out[1], out[2], value_seed)


def random_varlen(lengths_q: List[int], lengths_k: Optional[List[int]], H: int, D: int,
                  seed: int, name: str = "random") -> VarlenWorkload:
    """Arbitrary lengths (tests): flat q [sum Lq, H, D], k/v [sum Lk, H, D]."""
    lk = list(lengths_q) if lengths_k is None else list(lengths_k)
    g = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(g, sum(lengths_q), sum(lk), H, D)
    return VarlenWorkload(name, list(lengths_q), lk, H, D, q, k, v, seed)


def random_block_window(batch: int, n: int, H: int, D: int, block: int, seed: int,
                        layers=None) -> BlockWindowWorkload:
    g = torch.Generator().manual_seed(seed)
    shape = (batch, n, H, D)
    q = _randn_bf16(g, shape)
    k = _randn_bf16(g, shape)
    v = _randn_bf16(g, shape)
    return BlockWindowWorkload(f"block_window_n{n}", batch, n, H, D, block,
                               list(layers or [(0, 0)]), q, k, v, seed)


@dataclass
class LinearWorkload:
    """A packed-M projection: x [M, K] (the flat tokens of every request),
    w [N, K], bias [N]; `lengths` are the requests' row counts in x."""
    name: str
    lengths: List[int]
    x: torch.Tensor
    w: torch.Tensor
    bias: Optional[torch.Tensor]
    seed: int

    @property
    def M(self) -> int:
        return self.x.shape[0]

    @property
    def N(self) -> int:
        return self.w.shape[0]

    @property
    def K(self) -> int:
        return self.x.shape[1]


def linear_case(lengths: List[int], N: int, K: int, seed: int, bias: bool = True,
                name: str = "linear") -> LinearWorkload:
    """x ~ N(0, 1), w ~ N(0, 1/K) (unit-variance outputs), bias ~ N(0, 0.1^2),
    all rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    M = int(sum(lengths))
    x = _randn_bf16(g, (M, K))
    w = (torch.randn(N, K, generator=g) / float(K) ** 0.5).to(torch.bfloat16)
    b = (0.1 * torch.randn(N, generator=g)).to(torch.bfloat16) if bias else None
    return LinearWorkload(name, list(lengths), x, w, b, seed)


def mmdit_projection(kind: str = "qkv", seed: int = 2) -> LinearWorkload:
    """A projection of the mixed-resolution MMDiT batch: x is the batch's
    packed [T, 3072] hidden states (24 heads x 128); "qkv" multiplies by the
    fused [9216, 3072] QKV weight, "out" by the [3072, 3072] output weight."""
    g = torch.Generator().manual_seed(seed)
    L = lengths_mixed_res(g)
    N = {"qkv": 3 * 3072, "out": 3072}[kind]
    return linear_case(L, N, 3072, seed + 2000, bias=True, name=f"mmdit_{kind}_projection")


VARLEN_CONFIGS = {
    "tiny": tiny,
    "mixed_res_mmdit": mixed_res,
    "single_edit": single_edit,
    "cfg_dynamic_batch": cfg_batch,
}


@dataclass
class CfgSegments:
    """Model output rows of a CFG-doubled packed batch and its segment layout:
    flat [sum(lengths), C]; sequence b holds text rows [0, text[b]) then image
    rows; request r's positive pass is pos_seq[r], its negative pass
    neg_seq[r] (-1: no CFG); per-request guidance scale and normalize flag."""
    lengths: List[int]
    text: List[int]
    pos_seq: List[int]
    neg_seq: List[int]
    cfg_scale: List[float]
    cfg_normalize: List[int]
    flat: torch.Tensor
    img_max: int


def cfg_segments(C: int = 64, seed: int = 5, scales=(2.0, 7.0), normalize_every: int = 0
                 ) -> CfgSegments:
    """The CFG dynamic batch's lengths (drawn as in cfg_batch) with bf16
    N(0, 1) rows of width C drawn after them; request r uses guidance scale
    scales[r % len(scales)] (the page's example pair 2.0 / 7.0 by default) and
    normalizes when normalize_every > 0 and r % normalize_every == 0."""
    g = torch.Generator().manual_seed(seed)
    L, owner, text = lengths_cfg_batch_detail(g)
    flat = _randn_bf16(g, (sum(L), C))
    R = len(L) // 2
    img = [L[2 * r] - text[2 * r] for r in range(R)]
    return CfgSegments(L, text, [2 * r for r in range(R)], [2 * r + 1 for r in range(R)],
                       [float(scales[r % len(scales)]) for r in range(R)],
                       [1 if normalize_every and r % normalize_every == 0 else 0
                        for r in range(R)],
                       flat, max(img))
