"""Failure handling on the GPU without faulting it: a bounded wait that runs
out records a timeout and returns, and the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close_to_oracle, gpu_varlen

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    import packed_varlen_gb300 as pv
    pv.load_library()
    pv.get_device_status()
    pv.selftest_wait_timeout(2000)          # nothing ever arrives: ~2 ms
    assert pv.get_device_status() == 3      # PA_DEVICE_ERR_TIMEOUT
    assert pv.get_device_status() == 0
    # the context still runs the real path correctly
    w = workloads.random_varlen([200, 77], None, 2, 128, seed=21)
    out, _, _ = gpu_varlen(pv, w)
    cu = oracle.cu_seqlens_from_lengths(w.lengths_q)
    want = oracle.varlen_attention(w.q, w.k, w.v, cu, cu, w.scale)
    assert_close_to_oracle(oracle.to_f64(out), want, "after timeout")
    assert pv.get_device_status() == 0


def test_selftest_rejects_bad_timeout():
    import packed_varlen_gb300 as pv
    with pytest.raises(pv.PackedAttnError):
        pv.selftest_wait_timeout(0)
