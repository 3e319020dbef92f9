"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol the header declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import math
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "packedattn.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:pa_status|const char \*|int64_t)\s*(pa_\w+)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def lib(lib_path):
    import packed_varlen_gb300 as pv
    return pv.load_library(lib_path)


def test_header_declares_expected_entry_points():
    names = _declared()
    for n in ["pa_varlen_attn_fwd", "pa_block_window_attn_fwd", "pa_cu_seqlens_from_lengths",
              "pa_pack", "pa_unpack", "pa_varlen_work_order", "pa_varlen_num_work_items",
              "pa_get_device_status", "pa_status_string", "pa_cfg_combine",
              "pa_last_cuda_error", "pa_selftest_wait_timeout", "pa_rope_packed",
              "pa_block_window_attn_fwd_f32", "pa_linear_bf16"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in packedattn.h but not exported"


def test_status_strings(lib):
    for code, name in [(0, "PA_OK"), (1, "PA_ERR_INVALID_ARG"), (2, "PA_ERR_UNSUPPORTED"),
                       (3, "PA_ERR_MISALIGNED"), (4, "PA_ERR_CUDA"), (5, "PA_ERR_DEVICE"),
                       (99, "PA_ERR_UNKNOWN")]:
        assert lib.pa_status_string(code).decode() == name


# Fake, never-dereferenced addresses: every call below must be rejected by the
# host-side checks before anything touches the device.
A = 0x10000      # 16-byte aligned
MIS = 0x10008    # 8-byte aligned only


def _varlen(lib, **kw):
    args = dict(q=A, k=A, v=A, out=A, cu_q=A, cu_k=A, batch=2, total_q=10, total_k=10,
                max_q=8, max_k=8, H=2, D=64, scale=0.125)
    args.update(kw)
    return lib.pa_varlen_attn_fwd(args["q"], args["k"], args["v"], args["out"], args["cu_q"],
                                  args["cu_k"], args["batch"], args["total_q"], args["total_k"],
                                  args["max_q"], args["max_k"], args["H"], args["D"],
                                  args["scale"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(cu_k=None), 1), (dict(batch=0), 1), (dict(H=0), 1),
    (dict(total_q=-1), 1), (dict(max_k=-2), 1), (dict(scale=math.inf), 1),
    (dict(scale=math.nan), 1), (dict(D=96), 2), (dict(D=256), 2), (dict(batch=1025), 2),
    (dict(q=MIS), 3), (dict(out=MIS), 3), (dict(cu_q=A + 2), 3),
])
def test_varlen_host_checks(lib, kw, code):
    assert _varlen(lib, **kw) == code


def _bw(lib, fn, **kw):
    args = dict(q=A, k=A, v=A, out=A, batch=1, n=2400, block=24, lb=0, la=0, H=16, D=64,
                scale=0.125)
    args.update(kw)
    return getattr(lib, fn)(args["q"], args["k"], args["v"], args["out"], args["batch"],
                            args["n"], args["block"], args["lb"], args["la"], args["H"],
                            args["D"], args["scale"], None)


@pytest.mark.parametrize("fn", ["pa_block_window_attn_fwd", "pa_block_window_attn_fwd_f32"])
@pytest.mark.parametrize("kw,code", [
    (dict(v=None), 1), (dict(n=0), 1), (dict(block=0), 1), (dict(lb=-1), 1), (dict(la=-1), 1),
    (dict(scale=math.inf), 1), (dict(D=32), 2), (dict(k=MIS), 3), (dict(out=A + 4), 3),
    (dict(batch=70000), 2), (dict(H=0), 1),
])
def test_block_window_host_checks(lib, fn, kw, code):
    assert _bw(lib, fn, **kw) == code


def test_pack_and_scan_host_checks(lib):
    assert lib.pa_pack(None, A, A, 2, 8, 10, 6144, None) == 1
    assert lib.pa_pack(A, A, A, 0, 8, 10, 6144, None) == 1
    assert lib.pa_pack(A, A, A, 2, 8, 10, 0, None) == 1
    assert lib.pa_pack(A, A, A, 2, 8, 10, 6145, None) == 3
    assert lib.pa_unpack(A, MIS, A, 2, 8, 10, 6144, None) == 3
    assert lib.pa_cu_seqlens_from_lengths(None, A, 4, None) == 1
    assert lib.pa_cu_seqlens_from_lengths(A, A, 0, None) == 1
    assert lib.pa_varlen_work_order(A, A, 2, 0, 128, A, 10, None) == 1
    assert lib.pa_varlen_work_order(A, A, 2000, 2, 128, A, 10, None) == 2
    code = ctypes.c_int32(0)
    assert lib.pa_get_device_status(None) == 1


def test_num_work_items_matches_oracle(lib):
    import packed_varlen_gb300 as pv
    for L in ([37, 64], [0, 129, 128, 1], [33024], [16640, 4352, 7000, 2500]):
        cu = oracle.cu_seqlens_from_lengths(L).tolist()
        for H in (1, 24):
            for tile in (128, pv.VARLEN_TILE_M):
                assert pv.varlen_num_work_items(cu, H, tile) == len(oracle.work_order(L, L, H, tile))


def test_cfg_combine_host_checks(lib):
    # a template of arguments that is only ever passed with one field broken
    args = [A] * 8 + [4, 2, 100, 50, 64, None]
    bad = list(args); bad[0] = None
    assert lib.pa_cfg_combine(*bad) == 1
    bad = list(args); bad[8] = 0
    assert lib.pa_cfg_combine(*bad) == 1
    bad = list(args); bad[12] = 60   # row_elems not a multiple of 8
    assert lib.pa_cfg_combine(*bad) == 3
    bad = list(args); bad[1] = MIS
    assert lib.pa_cfg_combine(*bad) == 3
    bad = list(args); bad[9] = 70000
    assert lib.pa_cfg_combine(*bad) == 2


def test_rope_host_checks(lib):
    # every call has exactly one broken field, so nothing reaches the device
    ok = [A, A, A, A, None, 2, 10, 10, 2, 64, 1e4, None]
    for i, v, code in [(0, None, 1), (5, 0, 1), (9, 63, 1), (10, -1.0, 1), (10, math.inf, 1),
                       (9, 520, 2), (9, 12, 2), (0, MIS, 3), (2, A + 2, 3), (4, A + 1, 3)]:
        bad = list(ok)
        bad[i] = v
        assert lib.pa_rope_packed(*bad) == code, (i, v)


def test_linear_host_checks(lib):
    # every call has exactly one broken field, so nothing reaches the device
    ok = [A, A, None, A, 300, 512, 3072, None]
    for i, v, code in [(0, None, 1), (1, None, 1), (3, None, 1), (4, -1, 1), (5, 0, 1),
                       (6, 0, 1), (5, 516, 3), (6, 3076, 3), (0, MIS, 3), (3, A + 2, 3),
                       (2, MIS, 3)]:
        bad = list(ok)
        bad[i] = v
        assert lib.pa_linear_bf16(*bad) == code, (i, v)
    # M = 0 is a no-op that touches nothing; x and y may then be NULL
    empty = list(ok)
    empty[4] = 0
    assert lib.pa_linear_bf16(*empty) == 0
    empty[0] = empty[3] = None
    assert lib.pa_linear_bf16(*empty) == 0
