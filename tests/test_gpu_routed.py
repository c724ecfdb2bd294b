"""Routed backward (moe_grouped_mlp_bwd_routed + moe_router_grad_rows): the
router gradient taken inside the expert MLP, vs the oracle's
grouped_mlp_bwd_routed, and vs the Y-based router gradient of the plain
path.  Routings are real (GPU routing layout with alignment, so pad rows
and empty experts occur); dS is fp32 (plain tolerance bound)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def _setup(act, E, T, k, d, n, align, seed):
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[idx == E - 1] = 0 if k == 1 else idx[idx == E - 1]   # keep the last expert rare
    probs = rng.random((T, k)).astype(np.float32)
    r = M.route_offsets(cuda_i32(idx), E, align)
    torch.cuda.synchronize()
    ro = O.route_offsets(idx, E, align)
    M_cap = len(ro["pair_of_row"])
    n1 = n if act == "srelu" else 2 * n
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    H = W.normal((M_cap, n1), (seed, W.X, 1), 1.0, "cuda")
    tok_dO = W.normal((T, d), (seed, W.DO, 0), 1.0, "cuda")
    W1 = (W.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    do_perm = M.permute(tok_dO, r["pair_of_row"], k)             # unscaled gather
    return M, idx, probs, r, ro, x, H, tok_dO, do_perm, W1, W2


CASES = [
    ("ragged_align1", 4, 300, 2, 256, 192, 1),
    ("aligned32_empty", 6, 200, 1, 128, 128, 32),
    ("many_experts", 32, 256, 4, 128, 256, 8),
]


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,E,T,k,d,n,align", CASES, ids=[c[0] for c in CASES])
def test_routed_backward_matches_oracle(name, E, T, k, d, n, align, act):
    M, idx, probs, r, ro, x, H, tok_dO, do_perm, W1, W2 = _setup(act, E, T, k, d, n, align, 60)
    pt = torch.from_numpy(probs).cuda()
    dh, ap, dsp, dx, dW1, dW2, err = M.grouped_mlp_bwd_routed(
        x, H, do_perm, r["pair_of_row"], pt.view(-1), r["offsets"], W1, W2, act)
    dprobs = M.router_grad_rows(dsp, r["row_of_pair"], T, k)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    por = ro["pair_of_row"]
    row_prob = np.where(por >= 0, probs.reshape(-1)[np.maximum(por, 0)].astype(np.float64), 0.0)
    off = ro["offsets"]
    dO_perm = O.permute(f64(tok_dO), por, k)
    dH, _, _, _, Ap, dS = O.grouped_mlp_bwd_routed(f64(x), f64(H), dO_perm, row_prob, off,
                                                   f64(W1), f64(W2), act, round_out=False)
    # the three GEMMs after FC2-dgrad, each on its own inputs: dX = dH W1^T
    # and dW1 = X^T dH from the GPU's dH, dW2 = A'^T dO from the GPU's A'
    dX = O.grouped_gemm(f64(dh), off, f64(W1), "nk", round_out=False)
    dW1r = O.grouped_wgrad(f64(x), f64(dh), off, round_out=False)
    dW2r = O.grouped_wgrad(f64(ap), dO_perm, off, round_out=False)
    R = int(off[-1])
    assert_rms_close(f64(dh)[:R], dH[:R], f"{name}/{act} dH")
    assert_rms_close(f64(ap)[:R], Ap[:R], f"{name}/{act} A'")
    assert_rms_close(f64(dx)[:R], dX[:R], f"{name}/{act} dX")
    assert_rms_close(f64(dW1), dW1r, f"{name}/{act} dW1")
    assert_rms_close(f64(dW2), dW2r, f"{name}/{act} dW2")
    rop = ro["row_of_pair"]
    want = np.where(rop >= 0, dS[np.maximum(rop, 0)], 0.0).reshape(T, k)
    assert_rms_close(dprobs.cpu().numpy().astype(np.float64), want, f"{name}/{act} dS", rtol=0)
    for e in range(E):
        if off[e + 1] == off[e]:
            assert float(dW1[e].abs().max()) == 0 and float(dW2[e].abs().max()) == 0


def test_routed_backward_accumulate_dw():
    """MOE_FLAG_ACCUMULATE_DW on the routed backward: the weight gradients
    are added to the given ones; an empty expert's stay bit-identical."""
    act = "swiglu"
    M, idx, probs, r, ro, x, H, tok_dO, do_perm, W1, W2 = _setup(act, 6, 200, 1, 128, 128, 32, 62)
    T, k = idx.shape
    pt = torch.from_numpy(probs).cuda()
    por = ro["pair_of_row"]
    off = ro["offsets"]
    row_prob = np.where(por >= 0, probs.reshape(-1)[np.maximum(por, 0)].astype(np.float64), 0.0)
    _, _, dW1r, dW2r, _, _ = O.grouped_mlp_bwd_routed(f64(x), f64(H), O.permute(f64(tok_dO), por, k),
                                                      row_prob, off, f64(W1), f64(W2), act,
                                                      round_out=False)
    old1 = W.normal(dW1r.shape, (62, W.X, 90), float(np.sqrt((dW1r ** 2).mean())), "cuda")
    old2 = W.normal(dW2r.shape, (62, W.X, 91), float(np.sqrt((dW2r ** 2).mean())), "cuda")
    dW1, dW2 = old1.clone(), old2.clone()
    dh, ap, *_, err = M.grouped_mlp_bwd_routed(x, H, do_perm, r["pair_of_row"], pt.view(-1),
                                               r["offsets"], W1, W2, act, dW1=dW1, dW2=dW2,
                                               accumulate_dw=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # each weight gradient on its own inputs (the GPU's dH and A')
    dW1r = O.grouped_wgrad(f64(x), f64(dh), off, round_out=False)
    dW2r = O.grouped_wgrad(f64(ap), O.permute(f64(tok_dO), por, k), off, round_out=False)
    assert_rms_close(f64(dW1), f64(old1) + dW1r, "routed dW1 accumulated")
    assert_rms_close(f64(dW2), f64(old2) + dW2r, "routed dW2 accumulated")
    empty = [e for e in range(len(off) - 1) if off[e + 1] == off[e]]
    assert empty, "the case should hold an empty expert"
    for e in empty:
        assert torch.equal(dW1[e], old1[e]) and torch.equal(dW2[e], old2[e])


def test_routed_router_gradient_equals_y_based():
    """The rewrite gives the router gradient of the plain path (<dO, Y> from
    the forward's Y) to within the tolerance, and reruns are bitwise equal."""
    act = "swiglu"
    M, idx, probs, r, ro, x, H, tok_dO, do_perm, W1, W2 = _setup(act, 8, 512, 2, 256, 256, 1, 61)
    T, k = idx.shape
    pt = torch.from_numpy(probs).cuda()
    # forward with the same x to obtain H, A and Y
    h, a, y, e0 = M.grouped_mlp_fwd(x, r["offsets"], W1, W2, act, save_h=True)
    outs = []
    for _ in range(2):
        _, _, dsp, _, _, _, err = M.grouped_mlp_bwd_routed(
            x, h, do_perm, r["pair_of_row"], pt.view(-1), r["offsets"], W1, W2, act)
        outs.append(M.router_grad_rows(dsp, r["row_of_pair"], T, k).clone())
    ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
    M.unpermute(y, r["row_of_pair"], T, k, dO=tok_dO, dprobs=ref, combine=False)
    torch.cuda.synchronize()
    assert int(e0.item()) == 0 and int(err.item()) == 0
    assert torch.equal(outs[0], outs[1])
    assert_rms_close(f64(outs[0]), f64(ref), "dS rewrite vs <dO, Y>", rtol=0)
