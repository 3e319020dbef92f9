"""CPU oracle for packed variable-length attention (TEST INFRASTRUCTURE).

This package is test infrastructure, not part of the product.  Only the test
suite, the smoke check and the benchmark's CPU-baseline leg may import it.  The
CUDA library never calls into it and it never calls into the CUDA library; the
two share no code.  Everything here is plain NumPy in float64 (integers for
the integer steps), written for a reader to check against the definitions:

* ``cu_seqlens_from_lengths``, ``pack``, ``unpack``: the flat-packing steps
  ("[Perf][Diffusion][Qwen-Image] Replace per-bucket varlen loop with flat
  varlen attention for mixfusion", Key changes; "feat: Support dynamic
  batching for heterogeneous diffusion requests", How batching works).
* ``masked_attention``: softmax attention under an explicit boolean mask.
* ``varlen_attention``: per-sequence attention with the block-diagonal mask
  the cu_seqlens define ("feat: Support dynamic batching ...",
  AttentionMetadata).
* ``block_window_attention``: attention under the dense block-difference mask
  ("[Perf][Model] Use block-sparse attention in Qwen2.5-Omni Token2Wav DiT",
  Purpose and Change).
* ``work_order``: the length-ordered enumeration of (sequence, head, q-tile)
  work items.
* ``rope``, ``rope_positions``: rotary embedding with request-local
  positions ("feat: Support dynamic batching ...", Correctness model).
* ``cfg_combine``: segment-aware unpack of each request's image span with the
  per-request classifier-free-guidance combine ("feat: Support dynamic
  batching for heterogeneous diffusion requests", CFG behavior).
* ``linear``: the packed-M projection y = x w^T + bias ("feat: Support
  dynamic batching ...", packed varlen step batching, Determinism).

Every function is pinned by tests in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_cfg.py``, ``tests/test_oracle_rope.py`` and
``tests/test_oracle_linear.py`` against
brute force, closed forms, a library routine and the pages' invariants.
"""
from .packing import cu_seqlens_from_lengths, pack, unpack, work_order
from .cfg import cfg_combine
from .rope import rope, rope_positions
from .linear import linear, linear_rows, linear_flops
from .attention import (
    masked_attention,
    varlen_mask,
    varlen_attention,
    key_padding_attention,
    block_window_mask,
    block_window_attention,
    to_f64,
    varlen_useful_flops,
    block_window_useful_flops,
)

__all__ = [
    "cu_seqlens_from_lengths", "pack", "unpack", "work_order",
    "masked_attention", "varlen_mask", "varlen_attention", "key_padding_attention",
    "block_window_mask", "block_window_attention", "to_f64",
    "varlen_useful_flops", "block_window_useful_flops", "cfg_combine", "rope", "rope_positions",
    "linear", "linear_rows", "linear_flops",
]
