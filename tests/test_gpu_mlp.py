"""GPU grouped expert MLP (moe_grouped_mlp_fwd / _bwd) vs the oracle.

Sizes span several 128x256 tiles, ragged tails, empty experts and a
one-row expert.  Every output tensor must satisfy
max(|err| - 2^-8 |ref|) <= 2e-2 * RMS(ref), ref being the oracle's exact
value before the storage rounding.  The backward is checked stage by
stage, each GEMM on its own inputs: dH and dW2 from the GPU forward's
stored bf16 H and A, dX and dW1 from the GPU's stored bf16 dH (the forward
and dH are themselves checked against the oracle)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def _offsets(counts, align=1):
    off = [0]
    for c in counts:
        off.append(off[-1] + -(-c // align) * align)
    return np.array(off, np.int64)


def _case(E, d, n, counts, act, seed, tail=5, align=1):
    off = _offsets(counts, align)
    M_cap = int(off[-1]) + tail
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    if act == "srelu":
        W1 = W.w1_plain(seed, E, d, n, 0.05, "cuda")
    else:
        W1 = W.w1_interleaved(seed, E, d, n, 0.05, "cuda")
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    dy = W.normal((M_cap, d), (seed, W.DY, 0), 1.0, "cuda")
    return off, x, W1, W2, dy


def _bwd_refs(x, h, a, dy, dh, off, W1, W2, act):
    """Unrounded oracle references of the backward's four outputs, stage by
    stage: dH = act'(H; dY W2^T) and dW2 = A^T dY from the GPU's H and A;
    dX = dH W1^T (FC1-dgrad) and dW1 = X^T dH from the GPU's dH."""
    dH, _, _, dW2 = O.grouped_mlp_bwd(f64(x), f64(h), f64(a), f64(dy), off, f64(W1), f64(W2),
                                      act, round_out=False)
    gdh = f64(dh)
    dX = O.grouped_gemm(gdh, off, f64(W1), "nk", round_out=False)
    dW1 = O.grouped_wgrad(f64(x), gdh, off, round_out=False)
    return dH, dX, dW1, dW2


def _fwd(off, x, W1, W2, act, save_h=True):
    import dropless_grouped_gemm_gb300 as M
    h, a, y, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, act, save_h=save_h)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return h, a, y


FWD_CASES = [
    # name, E, d, n, counts
    ("one_tile_one_kblock", 1, 64, 128, [128]),
    ("one_tile_k_loop", 1, 512, 128, [128]),
    ("two_n_tiles", 1, 128, 256, [128]),
    ("ragged_rows", 1, 128, 128, [200]),
    ("ragged_empty_one_row", 4, 256, 192, [300, 0, 129, 1]),
    ("many_small_experts", 64, 128, 64, [(i * 7) % 41 for i in range(64)]),
]


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,E,d,n,counts", FWD_CASES, ids=[c[0] for c in FWD_CASES])
def test_fwd(name, E, d, n, counts, act):
    off, x, W1, W2, _ = _case(E, d, n, counts, act, seed=11)
    h, a, y = _fwd(off, x, W1, W2, act)
    H, A, Y = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act, round_out=False)
    R = int(off[-1])
    assert_rms_close(f64(h)[:R], H[:R], f"{name}/{act} H")
    assert_rms_close(f64(a)[:R], A[:R], f"{name}/{act} A")
    assert_rms_close(f64(y)[:R], Y[:R], f"{name}/{act} Y")


BWD_CASES = [
    ("one_tile", 1, 64, 128, [128]),
    ("ragged_tail_k", 1, 128, 128, [200]),
    ("ragged_empty_one_row", 4, 256, 192, [300, 0, 129, 1]),
    ("many_small_experts", 64, 128, 64, [(i * 7) % 41 for i in range(64)]),
    # >= 512 rows per expert on average: the weight gradients take the
    # large-expert configuration (four stages, 32-column staging)
    ("large_experts_ragged", 3, 128, 128, [700, 0, 900]),
]


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,E,d,n,counts", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_bwd(name, E, d, n, counts, act):
    import dropless_grouped_gemm_gb300 as M
    off, x, W1, W2, dy = _case(E, d, n, counts, act, seed=12)
    h, a, y = _fwd(off, x, W1, W2, act)
    dh, dx, dW1, dW2, err = M.grouped_mlp_bwd(x, h, a, dy, cuda_i32(off), W1, W2, act)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    dH, dX, dW1r, dW2r = _bwd_refs(x, h, a, dy, dh, off, W1, W2, act)
    R = int(off[-1])
    assert_rms_close(f64(dh)[:R], dH[:R], f"{name}/{act} dH")
    assert_rms_close(f64(dx)[:R], dX[:R], f"{name}/{act} dX")
    assert_rms_close(f64(dW2), dW2r, f"{name}/{act} dW2")
    assert_rms_close(f64(dW1), dW1r, f"{name}/{act} dW1")
    for e in range(E):
        if off[e + 1] == off[e]:
            assert float(dW1[e].abs().max()) == 0 and float(dW2[e].abs().max()) == 0


ACC_CASES = [c for c in BWD_CASES
             if c[0] in ("ragged_empty_one_row", "many_small_experts", "large_experts_ragged")]


def _prior(shape, ref, key):
    """A seeded earlier weight gradient with the RMS of this step's, so that
    dropping or doubling either term fails the tolerance."""
    rms = float(np.sqrt((ref ** 2).mean())) or 1.0
    return W.normal(shape, key, rms, "cuda")


@pytest.mark.parametrize("name,E,d,n,counts", ACC_CASES, ids=[c[0] for c in ACC_CASES])
def test_bwd_accumulate_dw(name, E, d, n, counts):
    """MOE_FLAG_ACCUMULATE_DW: dW1, dW2 become old + this step's gradient
    (one bf16 rounding of the sum); experts with no rows keep their old
    values bit for bit; dH and dX are unaffected."""
    import dropless_grouped_gemm_gb300 as M
    act = "swiglu"
    off, x, W1, W2, dy = _case(E, d, n, counts, act, seed=13)
    h, a, y = _fwd(off, x, W1, W2, act)
    _, _, dW1r, dW2r = O.grouped_mlp_bwd(f64(x), f64(h), f64(a), f64(dy), off, f64(W1),
                                           f64(W2), act, round_out=False)
    old1 = _prior(dW1r.shape, dW1r, (13, W.X, 90))
    old2 = _prior(dW2r.shape, dW2r, (13, W.X, 91))
    dW1, dW2 = old1.clone(), old2.clone()
    dh, dx, _, _, err = M.grouped_mlp_bwd(x, h, a, dy, cuda_i32(off), W1, W2, act, dW1=dW1,
                                          dW2=dW2, accumulate_dw=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    dH, dX, dW1r, dW2r = _bwd_refs(x, h, a, dy, dh, off, W1, W2, act)
    R = int(off[-1])
    assert_rms_close(f64(dh)[:R], dH[:R], f"{name} dH")
    assert_rms_close(f64(dx)[:R], dX[:R], f"{name} dX")
    assert_rms_close(f64(dW1), f64(old1) + dW1r, f"{name} dW1 accumulated")
    assert_rms_close(f64(dW2), f64(old2) + dW2r, f"{name} dW2 accumulated")
    for e in range(E):
        if off[e + 1] == off[e]:
            assert torch.equal(dW1[e], old1[e]) and torch.equal(dW2[e], old2[e])


def test_aligned_zero_pad_rows():
    """With align > 1 the pad rows permute writes are zero; the GEMMs then
    produce zero rows there and the weight gradients ignore them."""
    import dropless_grouped_gemm_gb300 as M
    E, d, n, T, k, align = 8, 256, 128, 300, 2, 32
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    tok = W.normal((T, d), (5, W.X, 0), 1.0, "cuda")
    r = M.route_offsets(cuda_i32(idx), E, align)
    xp = M.permute(tok, r["pair_of_row"], k)
    W1 = W.w1_interleaved(5, E, d, n, 0.05, "cuda")
    W2 = W.w2(5, E, n, d, 0.05, "cuda")
    h, a, y, err = M.grouped_mlp_fwd(xp, r["offsets"], W1, W2, "swiglu", save_h=True)
    torch.cuda.synchronize()
    ro = O.route_offsets(idx, E, align)
    off = ro["offsets"]
    H, A, Y = O.grouped_mlp_fwd(O.permute(f64(tok), ro["pair_of_row"], k), off, f64(W1), f64(W2),
                                "swiglu", round_out=False)
    R = int(off[-1])
    assert_rms_close(f64(y)[:R], Y[:R], "Y")
    pad = ro["pair_of_row"][:R] < 0
    assert (f64(y)[:R][pad] == 0).all() and (f64(a)[:R][pad] == 0).all()


def test_deterministic_bitwise():
    import dropless_grouped_gemm_gb300 as M
    off, x, W1, W2, dy = _case(4, 256, 128, [300, 0, 129, 70], "swiglu", seed=13)
    outs = []
    for _ in range(2):
        h, a, y = _fwd(off, x, W1, W2, "swiglu")
        dh, dx, dW1, dW2, _ = M.grouped_mlp_bwd(x, h, a, dy, cuda_i32(off), W1, W2, "swiglu")
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (h, a, y, dh, dx, dW1, dW2)])
    R = int(off[-1])
    for p, q in zip(outs[0], outs[1]):
        if p.shape[0] == x.shape[0]:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q)


def test_zero_rows_layer():
    """No rows at all: the forward writes nothing and the weight gradients
    are exactly zero."""
    import dropless_grouped_gemm_gb300 as M
    E, d, n = 4, 128, 64
    W1 = W.w1_interleaved(14, E, d, n, 0.05, "cuda")
    W2 = W.w2(14, E, n, d, 0.05, "cuda")
    x = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    off = cuda_i32(np.zeros(E + 1))
    h, a, y, err = M.grouped_mlp_fwd(x, off, W1, W2, "swiglu", save_h=True)
    dW1 = torch.full_like(W1, 7.0)
    dW2 = torch.full_like(W2, 7.0)
    _, _, dW1, dW2, err = M.grouped_mlp_bwd(x, h, a, torch.empty_like(x), off, W1, W2, "swiglu",
                                            dW1=dW1, dW2=dW2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert float(dW1.abs().max()) == 0 and float(dW2.abs().max()) == 0


def test_maximum_experts():
    """E = 1024 (the library's limit) with a sparse ragged routing."""
    import dropless_grouped_gemm_gb300 as M
    E, d, n = 1024, 64, 64
    counts = [(7 * i) % 23 if i % 5 else 0 for i in range(E)]
    off, x, W1, W2, dy = _case(E, d, n, counts, "swiglu", seed=15)
    h, a, y = _fwd(off, x, W1, W2, "swiglu")
    dh, dx, dW1, dW2, err = M.grouped_mlp_bwd(x, h, a, dy, cuda_i32(off), W1, W2, "swiglu")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    H, A, Y = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), "swiglu", round_out=False)
    dH, dX, dW1r, dW2r = _bwd_refs(x, h, a, dy, dh, off, W1, W2, "swiglu")
    R = int(off[-1])
    assert_rms_close(f64(y)[:R], Y[:R], "E=1024 Y")
    assert_rms_close(f64(dh)[:R], dH[:R], "E=1024 dH")
    assert_rms_close(f64(dx)[:R], dX[:R], "E=1024 dX")
    assert_rms_close(f64(dW1), dW1r, "E=1024 dW1")
    assert_rms_close(f64(dW2), dW2r, "E=1024 dW2")
