"""Failure detection on the GPU without a fault: the bounded wait used by
every kernel gives up after its limit, reports MOE_DEV_TIMEOUT through the
caller's error word, and leaves the context usable."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import dropless_grouped_gemm_gb300 as M
    L = M.lib()
    L.moe_selftest_bounded_wait.restype = ctypes.c_int
    L.moe_selftest_bounded_wait.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.moe_selftest_bounded_wait(20000, ctypes.c_void_p(err.data_ptr()),
                                     ctypes.c_void_p(waited.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == M.DEV_TIMEOUT          # timed out, and the completed wait did not
    assert 20000 <= int(waited.item()) < 1000000
    # the context still runs the grouped MLP correctly
    off = np.array([0, 96, 96, 200])
    x = W.normal((205, 128), (16, W.X, 0), 1.0, "cuda")
    W1 = W.w1_interleaved(16, 3, 128, 64, 0.05, "cuda")
    W2 = W.w2(16, 3, 64, 128, 0.05, "cuda")
    _, _, y, e2 = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, "swiglu")
    torch.cuda.synchronize()
    assert int(e2.item()) == 0
    _, _, Y = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), "swiglu", round_out=False)
    assert_rms_close(f64(y)[:200], Y[:200], "Y after the timeout test")
