"""Python binding of libpackedattn (packed variable-length attention, sm_103a).

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, passes raw device pointers and the current CUDA stream to the C ABI
declared in ``include/packedattn.h`` and raises ``PackedAttnError`` on a
non-OK status.  Every step runs in the library's CUDA kernels; there is no
other implementation behind these names.  Names are the C entry points
without their ``pa_`` prefix.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libpackedattn.so")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                3: "PA_ERR_MISALIGNED", 4: "PA_ERR_CUDA", 5: "PA_ERR_DEVICE"}
DEVICE_ERRORS = {0: "PA_DEVICE_OK", 1: "PA_DEVICE_ERR_CU_SEQLENS", 2: "PA_DEVICE_ERR_MAX_LEN",
                 3: "PA_DEVICE_ERR_TIMEOUT", 4: "PA_DEVICE_ERR_LENGTH",
                 5: "PA_DEVICE_ERR_CAPACITY", 6: "PA_DEVICE_ERR_SMEM_ALIGN",
                 7: "PA_DEVICE_ERR_SEGMENT"}
MAX_BATCH = 1024
VARLEN_TILE_M = 256


class PackedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        msg = f"{fn} returned {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


_lib = None

_c_i32 = ctypes.c_int32
_c_i64 = ctypes.c_int64
_c_ptr = ctypes.c_void_p
_c_f32 = ctypes.c_float

_SIGNATURES = {
    "pa_varlen_attn_fwd": ([_c_ptr] * 6 + [_c_i32] * 7 + [_c_f32, _c_ptr], _c_i32),
    "pa_block_window_attn_fwd": ([_c_ptr] * 4 + [_c_i32] * 7 + [_c_f32, _c_ptr], _c_i32),
    "pa_block_window_attn_fwd_f32": ([_c_ptr] * 4 + [_c_i32] * 7 + [_c_f32, _c_ptr], _c_i32),
    "pa_cu_seqlens_from_lengths": ([_c_ptr, _c_ptr, _c_i32, _c_ptr], _c_i32),
    "pa_pack": ([_c_ptr, _c_ptr, _c_ptr, _c_i32, _c_i32, _c_i32, _c_i64, _c_ptr], _c_i32),
    "pa_unpack": ([_c_ptr, _c_ptr, _c_ptr, _c_i32, _c_i32, _c_i32, _c_i64, _c_ptr], _c_i32),
    "pa_varlen_num_work_items": ([_c_ptr, _c_i32, _c_i32, _c_i32], _c_i64),
    "pa_varlen_work_order": ([_c_ptr, _c_ptr, _c_i32, _c_i32, _c_i32, _c_ptr, _c_i64, _c_ptr],
                             _c_i32),
    "pa_get_device_status": ([ctypes.POINTER(_c_i32)], _c_i32),
    "pa_status_string": ([_c_i32], ctypes.c_char_p),
    "pa_selftest_wait_timeout": ([_c_i32, _c_ptr], _c_i32),
    "pa_last_cuda_error": ([], ctypes.c_char_p),
    "pa_cfg_combine": ([_c_ptr] * 8 + [_c_i32] * 5 + [_c_ptr], _c_i32),
    "pa_rope_packed": ([_c_ptr] * 5 + [_c_i32] * 5 + [_c_f32, _c_ptr], _c_i32),
    "pa_linear_bf16": ([_c_ptr] * 4 + [_c_i32] * 3 + [_c_ptr], _c_i32),
}


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpackedattn.so (built in-tree by ``packed_varlen_gb300.build``).

    Raises if the library is missing: there is no fallback implementation."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != PA_OK:
        detail = ""
        if status == 4 and _lib is not None:
            detail = _lib.pa_last_cuda_error().decode()
        raise PackedAttnError(fn, status, detail)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtype, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")


def varlen_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                    max_q: int, max_k: int, scale: Optional[float] = None,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Packed varlen attention (pa_varlen_attn_fwd).  q [Tq, H, D], k/v
    [Tk, H, D] bf16; cu_seqlens int32 [B + 1] on the device.  Rows of ``out``
    beyond cu_seqlens_q[B] are not written (a fresh ``out`` is zero-filled)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    Tq, H, D = q.shape
    if k.shape[1:] != (H, D) or v.shape != k.shape:
        raise ValueError("k and v must be [Tk, H, D] with q's H and D")
    if cu_seqlens_k.numel() != cu_seqlens_q.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if out is None:
        out = torch.zeros_like(q)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = lib.pa_varlen_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                cu_seqlens_q.numel() - 1, Tq, k.shape[0], int(max_q),
                                int(max_k), H, D, float(scale), _stream(stream))
    _check("pa_varlen_attn_fwd", st)
    return out


def block_window_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block: int,
                          look_back: int, look_ahead: int, scale: Optional[float] = None,
                          out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Block-window attention (pa_block_window_attn_fwd); q/k/v [batch, n, H, D] bf16."""
    lib = load_library()
    for t, nme in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nme, torch.bfloat16, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same [batch, n, H, D] shape")
    batch, n, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = lib.pa_block_window_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      batch, n, int(block), int(look_back), int(look_ahead),
                                      H, D, float(scale), _stream(stream))
    _check("pa_block_window_attn_fwd", st)
    return out


def block_window_attn_fwd_f32(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block: int,
                              look_back: int, look_ahead: int, scale: Optional[float] = None,
                              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 block-window attention (pa_block_window_attn_fwd_f32); q/k/v
    [batch, n, H, D] float32."""
    lib = load_library()
    for t, nme in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nme, torch.float32, 4)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same [batch, n, H, D] shape")
    batch, n, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float32, 4)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = lib.pa_block_window_attn_fwd_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          out.data_ptr(), batch, n, int(block), int(look_back),
                                          int(look_ahead), H, D, float(scale), _stream(stream))
    _check("pa_block_window_attn_fwd_f32", st)
    return out


def cu_seqlens_from_lengths(lengths: torch.Tensor, out: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """cu[0] = 0, cu[b+1] = cu[b] + lengths[b] (pa_cu_seqlens_from_lengths)."""
    lib = load_library()
    _need(lengths, "lengths", torch.int32, 1)
    if out is None:
        out = torch.empty(lengths.numel() + 1, dtype=torch.int32, device=lengths.device)
    _need(out, "out", torch.int32, 1)
    if out.numel() != lengths.numel() + 1:
        raise ValueError("out must have batch + 1 entries")
    st = lib.pa_cu_seqlens_from_lengths(lengths.data_ptr(), out.data_ptr(), lengths.numel(),
                                        _stream(stream))
    _check("pa_cu_seqlens_from_lengths", st)
    return out


def _row_bytes(t: torch.Tensor, lead: int) -> int:
    n = 1
    for s in t.shape[lead:]:
        n *= s
    return n * t.element_size()


def pack(padded: torch.Tensor, cu_seqlens: torch.Tensor, total: int,
         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """padded [B, S_max, ...] -> flat [total, ...] (pa_pack).  ``total`` must be
    at least cu_seqlens[B] (the caller knows it from the host-side lengths)."""
    lib = load_library()
    _need(padded, "padded", padded.dtype)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    B, s_max = padded.shape[0], padded.shape[1]
    if cu_seqlens.numel() != B + 1:
        raise ValueError("cu_seqlens must have B + 1 entries")
    if out is None:
        out = torch.empty((int(total),) + tuple(padded.shape[2:]), dtype=padded.dtype,
                          device=padded.device)
    _need(out, "out", padded.dtype)
    if out.shape[0] != total or out.shape[1:] != padded.shape[2:]:
        raise ValueError("out must be [total, *padded.shape[2:]]")
    st = lib.pa_pack(padded.data_ptr(), out.data_ptr(), cu_seqlens.data_ptr(), B, s_max,
                     int(total), _row_bytes(padded, 2), _stream(stream))
    _check("pa_pack", st)
    return out


def unpack(flat: torch.Tensor, cu_seqlens: torch.Tensor, padded_out: torch.Tensor,
           stream=None) -> torch.Tensor:
    """flat [total, ...] -> rows [0, L_b) of each slot of padded_out [B, S_max, ...]
    (pa_unpack); padding rows of padded_out are left as they are."""
    lib = load_library()
    _need(flat, "flat", flat.dtype)
    _need(padded_out, "padded_out", flat.dtype)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    B, s_max = padded_out.shape[0], padded_out.shape[1]
    if cu_seqlens.numel() != B + 1 or padded_out.shape[2:] != flat.shape[1:]:
        raise ValueError("shape mismatch between flat, padded_out and cu_seqlens")
    st = lib.pa_unpack(flat.data_ptr(), padded_out.data_ptr(), cu_seqlens.data_ptr(), B, s_max,
                       flat.shape[0], _row_bytes(flat, 1), _stream(stream))
    _check("pa_unpack", st)
    return padded_out


def rope_packed(q: torch.Tensor, k: torch.Tensor, cu_seqlens_q: torch.Tensor,
                cu_seqlens_k: torch.Tensor, pos_offset: Optional[torch.Tensor] = None,
                base: float = 10000.0, stream=None):
    """Rotary embedding with request-local positions, in place on packed q
    [Tq, H, D] and k [Tk, H, D] bf16 (pa_rope_packed).  Returns (q, k)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    if k.shape[1:] != q.shape[1:] or cu_seqlens_k.numel() != cu_seqlens_q.numel():
        raise ValueError("q/k heads, dims or batch differ")
    B = cu_seqlens_q.numel() - 1
    ptr = None
    if pos_offset is not None:
        _need(pos_offset, "pos_offset", torch.int32, 1)
        if pos_offset.numel() != B:
            raise ValueError("pos_offset must have one entry per sequence")
        ptr = pos_offset.data_ptr()
    st = lib.pa_rope_packed(q.data_ptr(), k.data_ptr(), cu_seqlens_q.data_ptr(),
                            cu_seqlens_k.data_ptr(), ptr, B, q.shape[0], k.shape[0], q.shape[1],
                            q.shape[2], float(base), _stream(stream))
    _check("pa_rope_packed", st)
    return q, k


def cfg_combine(flat: torch.Tensor, cu_seqlens: torch.Tensor, img_off: torch.Tensor,
                pos_seq: torch.Tensor, neg_seq: torch.Tensor, cfg_scale: torch.Tensor,
                cfg_normalize: torch.Tensor, img_max: int, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """Per-request image-span unpack with the CFG combine (pa_cfg_combine).
    flat [T, ...] bf16 -> out [R, img_max, ...] bf16; index tensors int32 and
    cfg_scale float32 on the device.  Rows of ``out`` past each request's
    image span are left as they are (a fresh ``out`` is zero-filled)."""
    lib = load_library()
    _need(flat, "flat", torch.bfloat16)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    for t, n in ((img_off, "img_off"), (pos_seq, "pos_seq"), (neg_seq, "neg_seq"),
                 (cfg_normalize, "cfg_normalize")):
        _need(t, n, torch.int32, 1)
    _need(cfg_scale, "cfg_scale", torch.float32, 1)
    B, R = cu_seqlens.numel() - 1, pos_seq.numel()
    if img_off.numel() != B or neg_seq.numel() != R or cfg_scale.numel() != R or \
            cfg_normalize.numel() != R:
        raise ValueError("segment metadata sizes do not match")
    row = _row_bytes(flat, 1) // 2
    if out is None:
        out = torch.zeros((R, int(img_max)) + tuple(flat.shape[1:]), dtype=torch.bfloat16,
                          device=flat.device)
    _need(out, "out", torch.bfloat16)
    if out.shape[0] != R or out.shape[1] != img_max or out.shape[2:] != flat.shape[1:]:
        raise ValueError("out must be [R, img_max, *flat.shape[1:]]")
    st = lib.pa_cfg_combine(flat.data_ptr(), out.data_ptr(), cu_seqlens.data_ptr(),
                            img_off.data_ptr(), pos_seq.data_ptr(), neg_seq.data_ptr(),
                            cfg_scale.data_ptr(), cfg_normalize.data_ptr(), B, R, flat.shape[0],
                            int(img_max), row, _stream(stream))
    _check("pa_cfg_combine", st)
    return out


def varlen_num_work_items(cu_seqlens_q_host, H: int, tile_m: int = VARLEN_TILE_M) -> int:
    """Host-side work item count (pa_varlen_num_work_items); cu on the host."""
    lib = load_library()
    arr = (ctypes.c_int32 * len(cu_seqlens_q_host))(*[int(x) for x in cu_seqlens_q_host])
    n = lib.pa_varlen_num_work_items(ctypes.cast(arr, ctypes.c_void_p),
                                     len(cu_seqlens_q_host) - 1, H, tile_m)
    if n < 0:
        raise PackedAttnError("pa_varlen_num_work_items", 1)
    return int(n)


def varlen_work_order(cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, H: int,
                      capacity: int, tile_m: int = VARLEN_TILE_M, stream=None) -> torch.Tensor:
    """The attention kernel's work list as an int32 [capacity, 3] tensor of
    (sequence, head, q_tile) rows (pa_varlen_work_order)."""
    lib = load_library()
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    items = torch.full((max(1, capacity), 3), -1, dtype=torch.int32, device=cu_seqlens_q.device)
    st = lib.pa_varlen_work_order(cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                  cu_seqlens_q.numel() - 1, H, tile_m, items.data_ptr(),
                                  capacity, _stream(stream))
    _check("pa_varlen_work_order", st)
    return items[:capacity]


def get_device_status() -> int:
    """Synchronize, read and clear the device status word (pa_get_device_status).
    Returns the device error code (0 = none)."""
    lib = load_library()
    code = ctypes.c_int32(0)
    st = lib.pa_get_device_status(ctypes.byref(code))
    if st not in (PA_OK, 5):
        raise PackedAttnError("pa_get_device_status", st)
    return int(code.value)


def selftest_wait_timeout(timeout_us: int = 1000, stream=None) -> None:
    """Launch the bounded-wait self-test (pa_selftest_wait_timeout)."""
    lib = load_library()
    _check("pa_selftest_wait_timeout",
           lib.pa_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def status_string(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


def linear_bf16(x: torch.Tensor, w: torch.Tensor, bias: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = x w^T + bias (pa_linear_bf16); x [M, K], w [N, K], bias [N], bf16."""
    lib = load_library()
    _need(x, "x", torch.bfloat16, 2)
    _need(w, "w", torch.bfloat16, 2)
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError(f"w must be [N, {K}], got {tuple(w.shape)}")
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
        if bias.shape[0] != N:
            raise ValueError("bias must be [N]")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N]")
    st = lib.pa_linear_bf16(x.data_ptr(), w.data_ptr(),
                            bias.data_ptr() if bias is not None else None, out.data_ptr(),
                            M, N, K, _stream(stream))
    _check("pa_linear_bf16", st)
    return out
