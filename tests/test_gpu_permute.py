"""GPU permute / unpermute / router-score gradient vs the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def _setup(T, k, E, d, align, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    r = O.route_offsets(idx, E, align)
    x = W.normal((T, d), (seed, W.X, 0), 1.0, "cuda")
    p = rng.random((T, k)).astype(np.float32)
    p /= p.sum(1, keepdims=True)
    return idx, r, x, p


@pytest.mark.parametrize("T,k,E,d,align", [(512, 2, 4, 128, 1), (300, 8, 64, 7168, 32),
                                           (77, 1, 3, 64, 8)])
def test_permute_exact(T, k, E, d, align):
    import dropless_grouped_gemm_gb300 as M
    idx, r, x, _ = _setup(T, k, E, d, align, 1)
    xp = M.permute(x, cuda_i32(r["pair_of_row"]), k)
    ref = O.permute(f64(x), r["pair_of_row"], k)
    assert np.array_equal(f64(xp), ref)           # bit-exact copy, zero pad rows


# token-order permute (moe_permute_tokens): the same output as the row-order
# kernel, bit for bit, from the routing layout's two maps - plain and scaled,
# with pad rows (align), with pairs dropped by a too-small M_cap (their rows
# -1, the rows past M_cap never written), k = 1, and T = 0 (pad rows only)
@pytest.mark.parametrize("T,k,E,d,align,cap_cut,scaled", [
    (512, 2, 4, 128, 1, 0, False), (300, 8, 64, 7168, 32, 0, False),
    (300, 8, 64, 7168, 32, 0, True), (77, 1, 3, 64, 8, 0, False),
    (400, 4, 16, 256, 1, 100, False), (400, 4, 16, 256, 16, 100, True),
    (0, 2, 4, 128, 8, 0, False)])
def test_permute_tokens_equals_row_order(T, k, E, d, align, cap_cut, scaled):
    import dropless_grouped_gemm_gb300 as M
    rng = np.random.default_rng(T + k + E + align)
    idx = (np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
           if T > 0 else np.zeros((0, k), np.int32))
    M_cap = T * k - cap_cut if cap_cut else T * k + E * (align - 1)
    r = M.route_offsets(cuda_i32(idx).reshape(T, k), E, align, M_cap)
    x = W.normal((max(T, 1), d), (7, W.X, 0), 1.0, "cuda")[:T]
    sc = torch.from_numpy(rng.random(T * k).astype(np.float32)).cuda() if scaled else None
    a = torch.full((M_cap, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    b = torch.full((M_cap, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.permute(x, r["pair_of_row"], k, scale=sc, out=a)
    M.permute(x, r["pair_of_row"], k, scale=sc, out=b, row_of_pair=r["row_of_pair"])
    torch.cuda.synchronize()
    assert int(r["err"].item()) == (M.DEV_OVERFLOW if cap_cut else 0)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    if T > 0 and not scaled and not cap_cut:
        ref = O.permute(f64(x), r["pair_of_row"].cpu().numpy(), k)
        assert np.array_equal(f64(b), ref)


def test_permute_tokens_full_size_zipf():
    """The bench's routed steps permute x and dO in token order: on the Zipf
    layer's own routing (T = 4096, top-8, E = 256, d = 7168) both orders
    write the same bits, plain and scaled."""
    import dropless_grouped_gemm_gb300 as M
    w = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu"]
    idx, probs = W.route_inputs(w)
    r = M.route_offsets(cuda_i32(idx), w.E, w.align, w.M_cap)
    x = W.normal((w.T, w.d), (w.cfg_id, W.X, 0), w.x_std, "cuda")
    sc = torch.from_numpy(probs.reshape(-1)).cuda()
    for scale in (None, sc):
        a = M.permute(x, r["pair_of_row"], w.k, scale=scale)
        b = M.permute(x, r["pair_of_row"], w.k, scale=scale, row_of_pair=r["row_of_pair"])
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        del a, b
    assert int(r["err"].item()) == 0


def test_permute_scaled():
    import dropless_grouped_gemm_gb300 as M
    T, k, E, d = 257, 4, 16, 512
    idx, r, x, p = _setup(T, k, E, d, 1, 2)
    xp = M.permute(x, cuda_i32(r["pair_of_row"]), k, scale=torch.from_numpy(p.reshape(-1)).cuda())
    ref = O.permute(f64(x), r["pair_of_row"], k, scale=p.reshape(-1))
    got = f64(xp)
    assert_rms_close(got, O.permute(f64(x), r["pair_of_row"], k, scale=p.reshape(-1),
                                    round_out=False), "scaled permute")
    # float32 product then bf16 rounding: at most one bf16 step from the oracle
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - ref) <= ulp).all()


@pytest.mark.parametrize("T,k,E,d", [(512, 2, 4, 128), (200, 8, 256, 7168), (33, 1, 2, 64)])
def test_unpermute_and_router_grad(T, k, E, d):
    import dropless_grouped_gemm_gb300 as M
    idx, r, _, p = _setup(T, k, E, d, 1, 3)
    M_cap = len(r["pair_of_row"])
    y = W.normal((M_cap, d), (3, W.DY, 0), 1.0, "cuda")
    dO = W.normal((T, d), (3, W.DO, 0), 1.0, "cuda")
    rop = cuda_i32(r["row_of_pair"])
    pt = torch.from_numpy(p).cuda()
    out, _ = M.unpermute(y, rop, T, k, probs=pt)
    out1, _ = M.unpermute(y, rop, T, k)
    _, dp = M.unpermute(y, rop, T, k, dO=dO, combine=False)
    assert_rms_close(f64(out), O.unpermute(f64(y), r["row_of_pair"], T, k, p, round_out=False),
                     "combine")
    assert_rms_close(f64(out1), O.unpermute(f64(y), r["row_of_pair"], T, k, round_out=False),
                     "combine (no probs)")
    assert_rms_close(dp.cpu().numpy(), O.router_grad(f64(dO), f64(y), r["row_of_pair"], T, k),
                     "dprobs", rtol=0)


def test_roundtrip_identity():
    import dropless_grouped_gemm_gb300 as M
    T, k, E, d = 1000, 2, 8, 256
    idx, r, x, _ = _setup(T, k, E, d, 8, 4)
    xp = M.permute(x, cuda_i32(r["pair_of_row"]), k)
    back, _ = M.unpermute(xp, cuda_i32(r["row_of_pair"]), T, k)
    assert torch.equal(back.float(), 2 * x.float())     # k = 2: exact
