"""NVFP4 scaling statistics fused into the grouped GEMM epilogues:
max |A| of the forward output (FC1 epilogue, bf16 and MXFP8 paths) and the
amax of the transposed, 16-point Hadamard-rotated dH (FC2-dgrad epilogue,
plain and routed backward).

Each is checked two ways: against the oracle's statistic of the oracle's
own tensor (within the bf16 tolerance, relative), and against the oracle's
statistic of the tensor the kernel itself wrote (the fused reduction must
agree with a separate pass over its own output: bit-exact for max |A|,
float32 rounding of the 16-term sums for the rotated amax)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import cuda_i32, f64

pytestmark = pytest.mark.gpu

COUNTS = [300, 0, 129, 1, 77]      # ragged: blocks start at each expert's first row


def _layer(act, counts, d=256, n=128, seed=70, tail=7):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M_cap = int(off[-1]) + tail
    E = len(counts)
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    W1 = (W.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    dy = W.normal((M_cap, d), (seed, W.DY, 0), 1.0, "cuda")
    return off, x, W1, W2, dy


def _close(got, want, what, rel=2e-2):
    assert abs(got - want) <= rel * abs(want), (what, got, want)


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_forward_amax(act):
    import dropless_grouped_gemm_gb300 as M
    off, x, W1, W2, _ = _layer(act, COUNTS)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    h, a, y, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, act, save_h=True, amax=amax)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = int(off[-1])
    got = float(amax.item())
    assert got == O.amax(f64(a)[:R])                       # its own output, bit-exact
    _, A, _ = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act)
    _close(got, O.amax(A[:R]), f"{act} amax(A)")


def test_forward_amax_mxfp8_path():
    import dropless_grouped_gemm_gb300 as M
    counts = [256, 0, 96, 32]
    off, x, W1, W2, _ = _layer("swiglu", counts, d=256, n=128, tail=32)
    E, n, d = W2.shape
    M_cap = x.shape[0]
    bufs = M.mx_buffers(E, n, d, M_cap, "cuda")
    M.mx_quantize_weights(W2, bufs["w2_q"], bufs["w2_s"])
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    _, a, _, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, "swiglu", mx=bufs, amax=amax)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = int(off[-1])
    assert float(amax.item()) == O.amax(f64(a)[:R])


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_backward_rht_amax(act):
    import dropless_grouped_gemm_gb300 as M
    off, x, W1, W2, dy = _layer(act, COUNTS, seed=71)
    offs = cuda_i32(off)
    h, a, _, _ = M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    dh, _, _, _, err = M.grouped_mlp_bwd(x, h, a, dy, offs, W1, W2, act, amax=amax)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = float(amax.item())
    own = O.amax_rht_transposed(f64(dh), off)
    assert abs(got - own) <= 1e-6 * own, (got, own)
    H, A, _ = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act)
    dH, _, _, _ = O.grouped_mlp_bwd(f64(x), H, A, f64(dy), off, f64(W1), f64(W2), act)
    _close(got, O.amax_rht_transposed(dH, off), f"{act} amax(RHT(dH^T))")


def test_routed_backward_rht_amax():
    import dropless_grouped_gemm_gb300 as M
    E, T, k, d, n = 6, 256, 2, 256, 128
    rng = np.random.default_rng(72)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    probs = torch.from_numpy(rng.random((T, k)).astype(np.float32)).cuda()
    r = M.route_offsets(cuda_i32(idx), E, 1)
    ro = O.route_offsets(idx, E, 1)
    M_cap = len(ro["pair_of_row"])
    x = W.normal((M_cap, d), (72, W.X, 0), 1.0, "cuda")
    W1 = W.w1_interleaved(72, E, d, n, 0.05, "cuda")
    W2 = W.w2(72, E, n, d, 0.05, "cuda")
    dO = W.normal((T, d), (72, W.DO, 0), 1.0, "cuda")
    h, _, _, _ = M.grouped_mlp_fwd(x, r["offsets"], W1, W2, "swiglu", save_h=True)
    do_perm = M.permute(dO, r["pair_of_row"], k)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    dh, _, _, _, _, _, err = M.grouped_mlp_bwd_routed(x, h, do_perm, r["pair_of_row"], probs.view(-1),
                                                      r["offsets"], W1, W2, "swiglu", amax=amax)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = float(amax.item())
    own = O.amax_rht_transposed(f64(dh), ro["offsets"])
    assert abs(got - own) <= 1e-6 * own, (got, own)
