"""Pair mode of the grouped GEMM (2-SM MMAs, tcgen05.mma.cta_group::2):
the two CTAs of a cluster compute a 256 x 256 tile, each holding 128 rows
of A, one 128-column half of B and its 128 accumulator rows.

Every case runs the same forward and backward with pair mode forced on and
forced off (moe_set_pair_mma 2 / 0): all seven outputs must be equal bit for
bit, and within the tolerance of the oracle.  The weight gradients' ragged
reductions zero the rows past an expert's last 16-row boundary in both
CTAs' shared memory (the second CTA's through the cluster).  The first case is the smallest one (one expert
of 256 rows, one 256 x 256 output tile), then ragged shapes: an odd number
of 128-row blocks (the second CTA of the last unit has no rows), one-row and
empty experts, an output width that ends in half a tile, 64 experts.  On a
skinny layer the automatic mode's split launches (hot experts with 2-SM
tiles, the rest single-CTA) give the single-CTA outputs bit for bit too."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore_mode():
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    prev = M.set_pair_mma(M.PAIR_AUTO)
    yield
    M.set_pair_mma(prev)


def _case(E, d, n, counts, act, seed, tail=3):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M_cap = int(off[-1]) + tail
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    W1 = (W.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu" else
          W.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    dy = W.normal((M_cap, d), (seed, W.DY, 0), 1.0, "cuda")
    return off, x, W1, W2, dy


def _run(off, x, W1, W2, dy, act, mode):
    import dropless_grouped_gemm_gb300 as M
    M.set_pair_mma(mode)
    offs = cuda_i32(off)
    h, a, y, err = M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True)
    dh, dx, dW1, dW2, err = M.grouped_mlp_bwd(x, h, a, dy, offs, W1, W2, act, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return h, a, y, dh, dx, dW1, dW2


CASES = [
    # name, E, d, n, counts
    ("one_tile", 1, 256, 128, [256]),
    ("odd_row_blocks", 2, 256, 128, [384, 128]),
    ("ragged_empty_one_row", 4, 256, 192, [300, 0, 129, 1]),
    ("half_tile_width", 2, 384, 192, [256, 200]),
    ("many_experts", 64, 128, 64, [(i * 37) % 300 for i in range(64)]),
    # >= 512 rows per expert on average: the weight gradients' large-expert
    # configuration; ragged reductions (700 and 900 rows: tails of 12 and 4
    # rows past a 16-row boundary, zeroed in both CTAs' shared memory)
    ("large_experts_ragged", 3, 128, 128, [700, 0, 900]),
]


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,E,d,n,counts", CASES, ids=[c[0] for c in CASES])
def test_pair_equals_single_and_oracle(name, E, d, n, counts, act):
    if name == "one_tile" and act != "swiglu":
        pytest.skip("the bring-up case runs once")
    off, x, W1, W2, dy = _case(E, d, n, counts, act, seed=41)
    single = _run(off, x, W1, W2, dy, act, 0)
    pair = _run(off, x, W1, W2, dy, act, 2)
    R = int(off[-1])
    names = ("H", "A", "Y", "dH", "dX", "dW1", "dW2")
    for nm, p, q in zip(names, pair, single):
        if p.shape[0] == x.shape[0]:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q), f"{name}/{act} {nm}: pair mode differs from single-CTA tiles"
    h, a, y, dh, dx, dW1, dW2 = pair
    H, A, Y = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act, round_out=False)
    assert_rms_close(f64(h)[:R], H[:R], f"{name}/{act} H (pair)")
    assert_rms_close(f64(a)[:R], A[:R], f"{name}/{act} A (pair)")
    assert_rms_close(f64(y)[:R], Y[:R], f"{name}/{act} Y (pair)")
    dH, _, _, _ = O.grouped_mlp_bwd(f64(x), f64(h), f64(a), f64(dy), off, f64(W1), f64(W2), act,
                                    round_out=False)
    assert_rms_close(f64(dh)[:R], dH[:R], f"{name}/{act} dH (pair)")
    assert_rms_close(f64(dx)[:R], O.grouped_gemm(f64(dh), off, f64(W1), "nk", round_out=False)[:R],
                     f"{name}/{act} dX (pair)")
    assert_rms_close(f64(dW1), O.grouped_wgrad(f64(x), f64(dh), off, round_out=False),
                     f"{name}/{act} dW1 (pair)")
    assert_rms_close(f64(dW2), O.grouped_wgrad(f64(a), f64(dy), off, round_out=False),
                     f"{name}/{act} dW2 (pair)")
    for e in range(E):
        if counts[e] == 0:
            assert float(dW1[e].abs().max()) == 0 and float(dW2[e].abs().max()) == 0


def test_pair_rows_outside_experts_untouched():
    """Rows past the experts (the pair's second CTA computes them when an
    expert ends inside its unit) are never stored."""
    import dropless_grouped_gemm_gb300 as M
    off, x, W1, W2, dy = _case(2, 256, 128, [130, 1], "swiglu", seed=42, tail=200)
    M.set_pair_mma(2)
    R, Mc = int(off[-1]), x.shape[0]
    h = torch.full((Mc, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    a = torch.full((Mc, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((Mc, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    _, _, _, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, "swiglu", save_h=True, h_saved=h,
                                     a=a, y_perm=y)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for t in (h, a, y):
        assert bool(torch.isnan(t[R:].float()).all()) and bool(torch.isfinite(t[:R].float()).all())


def test_pair_mxfp8_fc1_codes_equal_single():
    """The FC1 epilogue with MXFP8 output in pair mode writes the same A,
    codes and scales as with single-CTA tiles (row tiles start at each
    expert's first row plus a multiple of 128 in both)."""
    import dropless_grouped_gemm_gb300 as M
    E, d, n = 3, 256, 128
    counts = [288, 0, 96]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M_cap = int(off[-1]) + 32
    x = W.normal((M_cap, d), (43, W.X, 0), 1.0, "cuda")
    W1 = W.w1_interleaved(43, E, d, n, 0.05, "cuda")
    W2 = W.w2(43, E, n, d, 0.05, "cuda")
    outs = []
    for mode in (0, 2):
        M.set_pair_mma(mode)
        buf = M.mx_buffers(E, n, d, M_cap, "cuda")
        M.mx_quantize_weights(W2, buf["w2_q"], buf["w2_s"])
        h, a, y, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, "swiglu", save_h=True, mx=buf)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((h, a, y, buf))
    R = int(off[-1])
    (h0, a0, y0, b0), (h1, a1, y1, b1) = outs
    assert torch.equal(h0[:R], h1[:R]) and torch.equal(a0[:R], a1[:R]) and torch.equal(y0[:R], y1[:R])
    assert torch.equal(b0["a_q"][:R], b1["a_q"][:R])
    assert torch.equal(b0["a_qT"][:, :R], b1["a_qT"][:, :R])
    assert torch.equal(b0["a_sT"][:, :R // 32], b1["a_sT"][:, :R // 32])
    from test_gpu_mx import decode_a_scales
    assert np.array_equal(decode_a_scales(b0["a_s"], off, M_cap, n)[:R],
                          decode_a_scales(b1["a_s"], off, M_cap, n)[:R])


MX_CASES = [
    # name, counts (multiples of 32), d, n
    ("mx_one_unit", [256], 256, 128),
    ("mx_odd_row_blocks", [384, 0, 96], 384, 128),
    ("mx_ragged_k", [160, 0, 96, 288], 256, 128),
    # reductions of 8 stages (K = 1024) over several units: every one of the
    # six stages' scale columns is live while an epilogue parks accumulator
    # columns in TMEM (the two must not share columns)
    ("mx_long_k", [512, 512, 256], 1024, 256),
]


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
@pytest.mark.parametrize("name,counts,d,n", MX_CASES, ids=[c[0] for c in MX_CASES])
def test_mx_pair_equals_single(name, counts, d, n, act):
    """The block-scaled GEMMs in pair mode (M = 256 MMAs over the CTA pair;
    each CTA's TMEM gets its own A rows' scales and both B halves' scales,
    loaded by TMA) give the single-CTA kernels' outputs bit for bit: the
    forward's block-scaled FC2, and the MXFP8 backward's FC2-dgrad + dAct +
    quantisation, both weight gradients and FC1-dgrad."""
    import dropless_grouped_gemm_gb300 as M
    from test_gpu_mx_bwd import _gpu_bwd, _layer
    off, x, H, A, dy, W1, W2 = _layer(44, counts, d, n, act)
    E = len(counts)
    R = int(off[-1])
    M_cap = x.shape[0]
    outs = []
    for mode in (0, 2):
        M.set_pair_mma(mode)
        buf = M.mx_buffers(E, n, d, M_cap, "cuda")
        M.mx_quantize_weights(W2, buf["w2_q"], buf["w2_s"])
        Wf = (W.w1_plain(44, E, d, n, 0.05, "cuda") if act == "srelu" else
              W.w1_interleaved(44, E, d, n, 0.05, "cuda"))
        h, a, y, err = M.grouped_mlp_fwd(x, cuda_i32(off), Wf, W2, act, save_h=True, mx=buf)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((y[:R].clone(),) + tuple(t.clone() for t in
                                              _gpu_bwd(off, x, H, A, dy, W1, W2, act)))
    for nm, p, q in zip(("Y", "dH", "dX", "dW1", "dW2"), outs[1], outs[0]):
        if p.shape[0] == M_cap:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q), f"{name}/{act} {nm}: MXFP8 pair mode differs from single-CTA tiles"


# A skinny layer (below 256 rows per expert on average) with a few hot
# experts: in automatic mode each GEMM runs its experts of 256 rows or more
# (weight gradients: reduction rows) in a launch of their own with 2-SM
# tiles, then the rest single-CTA.
SPLIT_COUNTS = [600, 0, 40, 300, 1, 0, 5, 270]


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_split_by_expert_size_equals_single(act):
    """Automatic mode on a skinny layer (the split launches) against
    single-CTA tiles throughout: all seven outputs bit for bit, and two
    kernels per GEMM."""
    import dropless_grouped_gemm_gb300 as M
    E, d, n = len(SPLIT_COUNTS), 256, 128
    off, x, W1, W2, dy = _case(E, d, n, SPLIT_COUNTS, act, seed=45)
    assert x.shape[0] < 256 * E and max(SPLIT_COUNTS) >= 256
    single = _run(off, x, W1, W2, dy, act, 0)
    split = _run(off, x, W1, W2, dy, act, 1)
    assert M.last_launch_count() == 2 * 4           # the backward's four GEMMs, split
    R = int(off[-1])
    for nm, p, q in zip(("H", "A", "Y", "dH", "dX", "dW1", "dW2"), split, single):
        if p.shape[0] == x.shape[0]:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q), f"{act} {nm}: split launches differ from single-CTA tiles"


def test_mx_split_weight_gradients_equal_single():
    """The MXFP8 backward on a skinny layer: in automatic mode the block-
    scaled weight gradients split by expert size (and the other GEMMs run
    2-SM); against single-CTA tiles throughout, every output bit for bit."""
    import dropless_grouped_gemm_gb300 as M
    from test_gpu_mx_bwd import _gpu_bwd, _layer
    counts = [608, 0, 64, 320, 32, 0, 0, 288]
    off, x, H, A, dy, W1, W2 = _layer(46, counts, 256, 128, "swiglu")
    assert x.shape[0] < 256 * len(counts)
    R = int(off[-1])
    outs = []
    for mode in (0, 1):
        M.set_pair_mma(mode)
        outs.append(tuple(t.clone() for t in _gpu_bwd(off, x, H, A, dy, W1, W2, "swiglu")))
    for nm, p, q in zip(("dH", "dX", "dW1", "dW2"), outs[1], outs[0]):
        if p.shape[0] == x.shape[0]:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q), f"MXFP8 {nm}: split launches differ from single-CTA tiles"
