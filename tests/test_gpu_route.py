"""GPU routing layout (moe_route_offsets) vs the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import cuda_i32

pytestmark = pytest.mark.gpu


def _run(idx, E, align, M_cap=None):
    import dropless_grouped_gemm_gb300 as M
    T, k = idx.shape
    r = M.route_offsets(cuda_i32(idx), E, align, M_cap)
    torch.cuda.synchronize()
    o = O.route_offsets(idx, E, align, M_cap)
    return {k_: v.cpu().numpy() for k_, v in r.items()}, o


def _check(g, o):
    assert g["counts"].tolist() == o["counts"].tolist()
    assert g["offsets"].tolist() == o["offsets"].tolist()
    assert g["row_of_pair"].tolist() == o["row_of_pair"].tolist()
    assert g["pair_of_row"].tolist() == o["pair_of_row"].tolist()
    assert int(g["true_total"][0]) == o["true_total"]
    assert int(g["err"][0]) == o["err"]


def _rand_route(seed, T, k, E):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)


@pytest.mark.parametrize("align", [1, 8, 32, 128])
def test_tiny_workload_routing(align):
    w = W.WORKLOADS["tiny_t512_d128_e4_top2_n256_swiglu_fwd"]
    idx, _ = W.route_inputs(w)
    g, o = _run(idx, w.E, align)
    _check(g, o)
    assert g["counts"][3] == 0


@pytest.mark.parametrize("align", [1, 32])
def test_zipf_256_experts_top8(align):
    w = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu"]
    idx, _ = W.route_inputs(w)
    g, o = _run(idx, w.E, align)
    _check(g, o)


@pytest.mark.parametrize("T,k,E", [(20000, 4, 64), (3, 1, 1), (1000, 8, 1024), (4097, 2, 5)])
def test_random_multi_chunk(T, k, E):
    g, o = _run(_rand_route(T + E, T, k, E), E, 1)
    _check(g, o)


def test_no_route_bad_ids_and_overflow():
    idx = _rand_route(7, 300, 2, 6)
    idx[5, 0] = -1
    idx[9, 1] = 6          # out of range -> flagged, skipped
    idx[11, 0] = -7
    g, o = _run(idx, 6, 1)
    _check(g, o)
    assert int(g["err"][0]) == O.ERR_BAD_EXPERT
    g, o = _run(_rand_route(8, 300, 2, 6), 6, 4, M_cap=500)   # demands up to 600 + pad
    _check(g, o)
    assert int(g["err"][0]) & O.ERR_OVERFLOW


def test_zero_tokens():
    g, o = _run(np.zeros((0, 2), np.int32), 4, 8)
    _check(g, o)


def test_deterministic():
    import dropless_grouped_gemm_gb300 as M
    idx = cuda_i32(_rand_route(9, 5000, 8, 256))
    a = M.route_offsets(idx, 256, 1)
    b = M.route_offsets(idx, 256, 1)
    for k_ in ("offsets", "row_of_pair", "pair_of_row"):
        assert torch.equal(a[k_], b[k_])


@pytest.mark.parametrize("T,E,k", [(4096, 256, 8), (300, 1024, 4), (64, 5, 5), (1000, 3, 1),
                                   (500, 64, 6), (500, 128, 4), (300, 512, 16)])
def test_router_topk(T, E, k):
    """Device top-k: the chosen experts match the oracle exactly (ties to the
    lower index); the softmax weights within float32 rounding."""
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0, :] = 0.25                                   # all tied
    lg[1, [3 % E, (E - 1)]] = 9.0                     # tie at the top
    if E > 4:
        lg[2, 4] = -np.inf
    idx, p = M.router_topk(torch.from_numpy(lg).cuda(), k)
    oi, op = O.router_topk(lg.astype(np.float64), k)
    assert idx.cpu().numpy().tolist() == oi.tolist()
    assert np.abs(p.cpu().numpy() - op).max() < 1e-6


def test_router_signed_zero_ties():
    """+0.0 and -0.0 logits compare equal, as floats do: a tie between them
    goes to the lower expert index, as in the oracle's stable sort."""
    import dropless_grouped_gemm_gb300 as M
    E, k = 40, 3
    lg = np.full((6, E), -1.0, dtype=np.float32)
    lg[0, [7, 3]] = [-0.0, 0.0]          # tie at the top, -0 at the higher index
    lg[1, [3, 7]] = [-0.0, 0.0]          # -0 at the lower index
    lg[2, [1, 33, 38]] = [0.0, -0.0, 0.0]
    lg[3, :] = -0.0                      # all tied
    lg[4, :] = 0.0
    lg[4, 20:] = -0.0
    lg[5, [0, 39]] = [-np.inf, 0.0]
    idx, p = M.router_topk(torch.from_numpy(lg).cuda(), k)
    oi, op = O.router_topk(lg.astype(np.float64), k)
    assert idx.cpu().numpy().tolist() == oi.tolist()
    assert np.abs(p.cpu().numpy() - op).max() < 1e-6
    fused = M.route_logits(torch.from_numpy(lg).cuda(), k, 1)
    assert torch.equal(fused["topk_idx"], idx) and torch.equal(fused["probs"], p)


def test_router_then_layout_on_zipf_logits():
    """Router on the Zipf layer's logits, then the routing layout: equal to
    the oracle's router followed by the oracle's layout."""
    import dropless_grouped_gemm_gb300 as M
    w = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu"]
    lg = W.logits(w.cfg_id, w.T, w.E, w.zipf_s)
    idx, p = M.router_topk(torch.from_numpy(lg).cuda(), w.k)
    r = M.route_offsets(idx, w.E, 1)
    oi, _ = O.router_topk(lg.astype(np.float64), w.k)
    ro = O.route_offsets(oi, w.E, 1)
    assert r["offsets"].cpu().numpy().tolist() == ro["offsets"].tolist()
    assert r["row_of_pair"].cpu().numpy().tolist() == ro["row_of_pair"].tolist()


# T * k not a multiple of the 4,096-pair chunk, with tokens whose k pairs
# straddle a chunk boundary (k = 3), an expert count above 1,024 / 2, a
# one-expert layer, every per-lane slot count of the router (E up to 32,
# 64, 128, 256, 512, 1,024) and k > 512, where a block's eight tokens span
# three chunks
@pytest.mark.parametrize("T,E,k,align", [(4096, 256, 8, 1), (3000, 600, 3, 32), (700, 1, 1, 8),
                                         (0, 16, 2, 1), (2000, 64, 6, 1), (1500, 128, 4, 4),
                                         (1200, 512, 16, 1), (40, 700, 600, 1)])
def test_fused_router_layout_equals_router_then_layout(T, E, k, align):
    """moe_route_logits (top-k fused into the layout's first pass) writes the
    router's topk_idx and probs and the layout's outputs bit for bit as the
    separate router followed by moe_route_offsets, and matches the oracle."""
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if T > 2:
        lg[0, :] = 0.25                               # all tied
        lg[1, [0, E - 1]] = 9.0                       # tie at the top
    lt = torch.from_numpy(lg).cuda()
    fused = M.route_logits(lt, k, align)
    if T > 0:
        assert M.last_launch_count() == 4           # no separate router launch
    idx, p = M.router_topk(lt, k)
    sep = M.route_offsets(idx, E, align)
    torch.cuda.synchronize()
    assert int(fused["err"].item()) == 0
    assert torch.equal(fused["topk_idx"], idx) and torch.equal(fused["probs"], p)
    for k_ in ("counts", "offsets", "row_of_pair", "pair_of_row", "true_total"):
        assert torch.equal(fused[k_], sep[k_]), k_
    if T > 0:
        oi, _ = O.router_topk(lg.astype(np.float64), k)
        ro = O.route_offsets(oi, E, align)
        assert fused["offsets"].cpu().numpy().tolist() == ro["offsets"].tolist()
        assert fused["row_of_pair"].cpu().numpy().tolist() == ro["row_of_pair"].tolist()
