"""The unfused pieces (moe_grouped_gemm, moe_activation, moe_activation_bwd)
vs the oracle, and the unfused chain vs the fused entry points.

Sizes span several 128x256 tiles, ragged tails, an empty expert, a
one-row expert and an output width that ends in a partial tile."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu

COUNTS = [300, 0, 129, 1]


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("K,N", [(128, 192), (256, 320)])
def test_grouped_gemm_matches_oracle(layout, K, N):
    import dropless_grouped_gemm_gb300 as M
    off = _offsets(COUNTS)
    E, R = len(COUNTS), int(off[-1])
    M_cap = R + 7
    a = W.normal((M_cap, K), (71, W.X, 0), 1.0, "cuda")
    B = W.normal((E, K, N) if layout == "kn" else (E, N, K), (71, W.X, 1), 0.05, "cuda")
    sentinel = torch.full((M_cap, N), 7.0, dtype=torch.bfloat16, device="cuda")
    out, err = M.grouped_gemm(a, cuda_i32(off), B, layout, out=sentinel)
    torch.cuda.synchronize()
    # experts below 256 rows on average: those of 256 rows or more (found on
    # the device) run first, in a launch of their own with 2-SM tiles
    split = M_cap < 256 * E and E > 1
    assert int(err.item()) == 0 and M.last_launch_count() == (2 if split else 1)
    ref = O.grouped_gemm(f64(a), off, f64(B), layout, round_out=False)
    assert_rms_close(f64(out)[:R], ref[:R], f"grouped_gemm {layout} K={K} N={N}")
    assert (f64(out)[R:] == 7.0).all()          # rows outside every expert untouched


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_activation_passes_match_oracle(act):
    import dropless_grouped_gemm_gb300 as M
    off = _offsets(COUNTS)
    R = int(off[-1])
    M_cap, n = R + 9, 192
    n1 = n if act == "srelu" else 2 * n
    h = W.normal((M_cap, n1), (72, W.X, 0), 1.5, "cuda")
    da = W.normal((M_cap, n), (72, W.DY, 0), 1.0, "cuda")
    offs = cuda_i32(off)
    a = torch.full((M_cap, n), 7.0, dtype=torch.bfloat16, device="cuda")
    dh = torch.full((M_cap, n1), 7.0, dtype=torch.bfloat16, device="cuda")
    M.activation(h, offs, act, a=a)
    M.activation_bwd(h, da, offs, act, dh=dh)
    torch.cuda.synchronize()
    assert_rms_close(f64(a)[:R], O.act_forward(f64(h)[:R], act), f"{act} A")
    assert_rms_close(f64(dh)[:R], O.act_backward(f64(h)[:R], f64(da)[:R], act),
                     f"{act} dH")
    assert (f64(a)[R:] == 7.0).all() and (f64(dh)[R:] == 7.0).all()


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_unfused_chain_equals_fused(act):
    """GEMM writing H, then the activation pass, gives the fused FC1's H (bit
    for bit) and A; the dgrad GEMM writing dA, then the derivative pass,
    gives the fused FC2-dgrad's dH.  The unfused passes start from the
    bf16-rounded H and dA, whose relative rounding error (2^-9) the
    activation amplifies by its elasticity (2 for max(h,0)^2, about 1 for
    the gated forms away from phi(g) = 0), and each side rounds its output
    once (2^-9 each): so the relative part of the bound is 2^-7 + 2^-8 <=
    2^-6, i.e. two bf16 steps; the absolute part stays 2e-2 RMS."""
    import dropless_grouped_gemm_gb300 as M
    off = _offsets(COUNTS)
    E, R = len(COUNTS), int(off[-1])
    d, n = 256, 128
    M_cap = R + 3
    n1 = n if act == "srelu" else 2 * n
    x = W.normal((M_cap, d), (73, W.X, 0), 1.0, "cuda")
    W1 = (W.w1_plain(73, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(73, E, d, n, 0.05, "cuda"))
    W2 = W.w2(73, E, n, d, 0.05, "cuda")
    dy = W.normal((M_cap, d), (73, W.DY, 0), 1.0, "cuda")
    offs = cuda_i32(off)
    h_f, a_f, _, e0 = M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True)
    dh_f, _, _, _, e1 = M.grouped_mlp_bwd(x, h_f, a_f, dy, offs, W1, W2, act)
    h_u, e2 = M.grouped_gemm(x, offs, W1, "kn")
    a_u = M.activation(h_u, offs, act)
    da_u, e3 = M.grouped_gemm(dy, offs, W2, "nk")
    dh_u = M.activation_bwd(h_f, da_u, offs, act)
    torch.cuda.synchronize()
    assert all(int(e.item()) == 0 for e in (e0, e1, e2, e3))
    assert torch.equal(h_u[:R], h_f[:R])          # same GEMM, same rounding
    rtol = 2.0 ** -6
    assert_rms_close(f64(a_u)[:R], f64(a_f)[:R], f"{act} A unfused vs fused", rtol=rtol)
    assert_rms_close(f64(dh_u)[:R], f64(dh_f)[:R], f"{act} dH unfused vs fused", rtol=rtol)
