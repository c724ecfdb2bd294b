"""The no-allocation routing entry point (moe_route_offsets_noalloc).

Some callers cannot allocate device memory at the point where they route
tokens: a CUDA-graph capture that must not grow a memory pool, an
allocator-free runtime, or a plugin whose host framework owns every
allocation.  For them the library keeps its routing scratch in a fixed
array of its own.  This file checks, through the C ABI, that the entry
point gives exactly what moe_route_offsets gives with a caller-allocated
workspace, on two calls in a row with different routings (so a stale
scratch from the first call cannot hide a fault in the second), and that a
size needing more than the fixed scratch is refused.  It is collected last
so that a failure here leaves every other test already run."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _entry():
    from dropless_grouped_gemm_gb300 import build
    build.build()
    import dropless_grouped_gemm_gb300 as M
    f = M.lib().moe_route_offsets_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.restype = i32
    f.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    return M, f


def _routing(seed, T, k, E):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)) + np.log(1.0 / (np.arange(E) + 1.0) ** 1.2)
    return np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)


def _call_noalloc(f, idx_t, E, align, M_cap):
    T, k = idx_t.shape
    dev = idx_t.device
    o = {"counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
         "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
         "row_of_pair": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
         "pair_of_row": torch.full((M_cap,), -7, dtype=torch.int32, device=dev),
         "true_total": torch.full((1,), -7, dtype=torch.int32, device=dev),
         "err": torch.zeros(1, dtype=torch.int32, device=dev)}
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = f(p(idx_t), T, k, E, align, M_cap, p(o["counts"]), p(o["offsets"]), p(o["row_of_pair"]),
           p(o["pair_of_row"]), p(o["true_total"]), p(o["err"]),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o


def test_noalloc_equals_workspace_version_two_calls_in_a_row():
    M, f = _entry()
    for seed, (T, k, E, align) in [(1, (4096, 8, 256, 1)), (2, (3000, 2, 64, 32))]:
        idx = torch.from_numpy(_routing(seed, T, k, E)).cuda()
        M_cap = T * k + E * (align - 1)
        ref = M.route_offsets(idx, E, align, M_cap)
        rc, got = _call_noalloc(f, idx, E, align, M_cap)
        assert rc == 0
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "row_of_pair", "pair_of_row", "true_total", "err"):
            assert torch.equal(got[name], ref[name]), (seed, name)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    M, f = _entry()
    E, k = 1024, 8
    T = 140000                      # (ceil(T*k/4096) + 1) * E * 4 bytes > 1 MiB
    assert M.route_workspace_size(T, k, E) > (1 << 20)
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    rc, _ = _call_noalloc(f, idx, E, 1, T * k)
    assert rc == -6                 # MOE_E_WORKSPACE
