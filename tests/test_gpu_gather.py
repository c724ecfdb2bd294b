"""Gather fusion (moe_grouped_mlp_fwd_gather): FC1 reads the token rows
through the routing map instead of a permuted copy.  Its H, A and Y equal
the permute-then-GEMM path's bit for bit (the same rows reach the same
MMAs), and match the oracle.  Routings with pad rows (align > 1), empty
experts, experts of one and of several 128-row blocks."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu

CASES = [
    # name, E, T, k, d, n, align
    ("ragged_align1", 4, 300, 2, 256, 192, 1),
    ("aligned32_pad_rows", 6, 500, 2, 128, 128, 32),
    ("many_experts", 32, 256, 4, 192, 128, 8),
    ("long_expert", 2, 700, 1, 128, 128, 1),
]


def _split(M_cap, E):
    """Extra launch of a non-gathered GEMM whose experts average fewer than
    256 rows: those of 256 rows or more run first, with 2-SM tiles."""
    return int(E > 1 and M_cap < 256 * E)


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
@pytest.mark.parametrize("name,E,T,k,d,n,align", CASES, ids=[c[0] for c in CASES])
def test_gather_forward_equals_permuted(name, E, T, k, d, n, align, act):
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(81)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if E > k:
        idx[idx == E - 1] = (E - 2)          # one expert left empty
    r = M.route_offsets(cuda_i32(idx), E, align)
    x = W.normal((T, d), (81, W.X, 0), 1.0, "cuda")
    W1 = (W.w1_plain(81, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(81, E, d, n, 0.05, "cuda"))
    W2 = W.w2(81, E, n, d, 0.05, "cuda")
    xp = M.permute(x, r["pair_of_row"], k)
    h0, a0, y0, e0 = M.grouped_mlp_fwd(xp, r["offsets"], W1, W2, act, save_h=True)
    h1, a1, y1, e1 = M.grouped_mlp_fwd_gather(x, r["pair_of_row"], k, r["offsets"], W1, W2, act,
                                              save_h=True)
    torch.cuda.synchronize()
    # FC2 reads the permuted A: on a layer below 256 rows per expert its hot
    # experts get a launch of their own (_split)
    assert int(e0.item()) == 0 and int(e1.item()) == 0
    assert M.last_launch_count() == 2 + _split(xp.shape[0], E)
    ro = O.route_offsets(idx, E, align)
    off = ro["offsets"]
    R = int(off[-1])
    assert torch.equal(h1[:R], h0[:R]) and torch.equal(a1[:R], a0[:R])
    assert torch.equal(y1[:R], y0[:R])
    H, A, Y = O.grouped_mlp_fwd(O.permute(f64(x), ro["pair_of_row"], k), off, f64(W1), f64(W2), act,
                                round_out=False)
    assert_rms_close(f64(y1)[:R], Y[:R], f"{name}/{act} Y (gathered)")


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,E,T,k,d,n,align", CASES, ids=[c[0] for c in CASES])
def test_gather_routed_backward_equals_permuted(name, E, T, k, d, n, align, act):
    """The gathered routed backward (dO rows for FC2-dgrad and FC2-wgrad, x
    rows for FC1-wgrad, all through the routing map) gives the permuted
    routed backward's dH, A', dS partials, dX and both weight gradients bit
    for bit, and its dW match the oracle."""
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(82)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if E > k:
        idx[idx == E - 1] = (E - 2)          # one expert left empty
    probs = torch.from_numpy(rng.random((T, k)).astype(np.float32)).cuda()
    r = M.route_offsets(cuda_i32(idx), E, align)
    M_cap = r["pair_of_row"].numel()
    n1 = n if act == "srelu" else 2 * n
    x = W.normal((T, d), (82, W.X, 0), 1.0, "cuda")
    dO = W.normal((T, d), (82, W.DO, 0), 1.0, "cuda")
    H = W.normal((M_cap, n1), (82, W.X, 1), 1.0, "cuda")
    W1 = (W.w1_plain(82, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(82, E, d, n, 0.05, "cuda"))
    W2 = W.w2(82, E, n, d, 0.05, "cuda")
    pr, off = r["pair_of_row"], r["offsets"]
    xp, dop = M.permute(x, pr, k), M.permute(dO, pr, k)
    ref = M.grouped_mlp_bwd_routed(xp, H, dop, pr, probs.view(-1), off, W1, W2, act)
    got = M.grouped_mlp_bwd_routed_gather(x, dO, pr, k, H, probs.view(-1), off, W1, W2, act)
    torch.cuda.synchronize()
    assert int(ref[-1].item()) == 0 and int(got[-1].item()) == 0
    assert M.last_launch_count() == 4 + _split(M_cap, E)     # FC1-dgrad reads dH, not gathered
    ro = O.route_offsets(idx, E, align)
    R = int(ro["offsets"][-1])
    for nm, i in (("dh", 0), ("a_scaled", 1), ("ds_part", 2), ("dx_perm", 3)):
        assert torch.equal(got[i][:R], ref[i][:R]), nm
    assert torch.equal(got[4], ref[4]) and torch.equal(got[5], ref[5])     # dW1, dW2
    por = ro["pair_of_row"]
    row_prob = np.where(por >= 0, probs.cpu().numpy().reshape(-1)[np.maximum(por, 0)], 0.0)
    # each weight gradient on its own inputs: dW1 = X^T dH from the GPU's dH,
    # dW2 = A'^T dO from the GPU's A' (both checked against the oracle in
    # test_gpu_routed.py)
    dW1r = O.grouped_wgrad(O.permute(f64(x), por, k), f64(got[0]), ro["offsets"], round_out=False)
    dW2r = O.grouped_wgrad(f64(got[1]), O.permute(f64(dO), por, k), ro["offsets"],
                           round_out=False)
    assert_rms_close(f64(got[4]), dW1r, f"{name}/{act} dW1 (gathered)")
    assert_rms_close(f64(got[5]), dW2r, f"{name}/{act} dW2 (gathered)")


def test_gather_full_size_zipf_layer_equals_permuted():
    """The full-size Zipf layer (T=4096, d=7168, E=256, top-8, n=2048; the
    bench's gathered step) against the permuted step on the same inputs:
    every output of the training step equal bit for bit.  The permuted
    step's own parity with the oracle at this size is checked in
    test_gpu_fullsize.py."""
    import bench as BE
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    base = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu"]
    wg = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu_gather"]
    inp, o = BE.make_inputs(base, "cuda")

    def like(v):
        if isinstance(v, dict):
            return {k_: like(x) for k_, x in v.items()}
        return torch.empty_like(v)
    o2 = {k_: like(v) for k_, v in o.items()}
    o2["err"].zero_()
    o2["route"]["err"] = o2["err"]
    n1 = BE.make_step(base, inp, o)()
    n2 = BE.make_step(wg, inp, o2)()
    torch.cuda.synchronize()
    assert int(o["err"].item()) == 0 and int(o2["err"].item()) == 0
    # the two permutes are gone; each of the six GEMMs splits its hot experts
    # into a launch of their own on this layer, except the four gathered ones
    assert n2 == n1 - 2 - 4 * _split(base.M_cap, base.E)
    R = int(o["route"]["offsets"][-1].item())
    for k_ in ("h", "a", "y_perm", "dh", "a_scaled", "ds_part", "dx_perm"):
        assert torch.equal(o2[k_][:R], o[k_][:R]), k_
    for k_ in ("out", "dx", "dprobs", "dW1", "dW2"):
        assert torch.equal(o2[k_], o[k_]), k_
    del inp, o, o2
    torch.cuda.empty_cache()


def test_gather_routed_backward_accumulates_like_permuted():
    """MOE_FLAG_ACCUMULATE_DW on the gathered routed backward: the weight
    gradients added to the given ones equal the permuted path's, bit for
    bit, and the empty expert's stay untouched."""
    import dropless_grouped_gemm_gb300 as M
    E, T, k, d, n, align = 6, 500, 2, 128, 128, 32
    act = "swiglu"
    rng = np.random.default_rng(83)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[idx == E - 1] = E - 2                     # expert E-1 empty
    probs = torch.from_numpy(rng.random((T, k)).astype(np.float32)).cuda().view(-1)
    r = M.route_offsets(cuda_i32(idx), E, align)
    M_cap = r["pair_of_row"].numel()
    x = W.normal((T, d), (83, W.X, 0), 1.0, "cuda")
    dO = W.normal((T, d), (83, W.DO, 0), 1.0, "cuda")
    H = W.normal((M_cap, 2 * n), (83, W.X, 1), 1.0, "cuda")
    W1 = W.w1_interleaved(83, E, d, n, 0.05, "cuda")
    W2 = W.w2(83, E, n, d, 0.05, "cuda")
    old1 = W.normal(tuple(W1.shape), (83, W.X, 90), 0.5, "cuda")
    old2 = W.normal(tuple(W2.shape), (83, W.X, 91), 0.5, "cuda")
    pr, off = r["pair_of_row"], r["offsets"]
    xp, dop = M.permute(x, pr, k), M.permute(dO, pr, k)
    a1, a2 = old1.clone(), old2.clone()
    b1, b2 = old1.clone(), old2.clone()
    M.grouped_mlp_bwd_routed(xp, H, dop, pr, probs, off, W1, W2, act, dW1=a1, dW2=a2,
                             accumulate_dw=True)
    M.grouped_mlp_bwd_routed_gather(x, dO, pr, k, H, probs, off, W1, W2, act, dW1=b1, dW2=b2,
                                    accumulate_dw=True)
    torch.cuda.synchronize()
    assert torch.equal(a1, b1) and torch.equal(a2, b2)
    assert torch.equal(b1[E - 1], old1[E - 1]) and torch.equal(b2[E - 1], old2[E - 1])
    assert not torch.equal(b1[0], old1[0])
