"""Full-size parity of the MXFP8 path (forward and backward) on the Zipf
layer (T=4096, d=7168, E=256, top-8, n=2048, align 32), in the launch
configuration bench.py times.

The GPU runs one step of the bench's MXFP8 training workload.  The oracle
(oracle.moe, oracle.mx) recomputes from the same seeded inputs:
  * sampled rows of a hot expert, a small one and the smallest: A and the
    block-scaled FC2 output Y; dH (block-scaled FC2-dgrad + dAct) and dX
    (block-scaled FC1-dgrad);
  * the fused FC1 epilogue's MXFP8 codes and scales (row-wise and the
    group-aware transposed copy) of a hot, a median and the smallest
    expert, bit for bit against the OCP MX quantiser applied to the GPU's
    own bf16 A, on every block;
  * the whole MXFP8 weight gradients of a small expert: element-wise
    against the oracle's block-scaled weight gradient of the GPU's own bf16
    operands (stage-wise), and in aggregate against the oracle's
    independent chain from x; zeros for experts with no rows.
Rows of an expert include its pad rows (zeros) up to the 32-row boundary:
the group-aware blocks of the weight gradients see them."""
import numpy as np
import pytest
import torch

import bench as BE
import oracle as O
from oracle import mx as X
import workloads as WL
from _helpers import assert_rms_close, f64
from test_gpu_mx import decode_a_scales

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WNAME = "zipf_t4096_d7168_e256_top8_n2048_mxfp8_train"


def _expert_weights(w, e):
    d, n = w.d, w.n
    W1 = WL.w1_interleaved(w.cfg_id, 1, d, n, w.w_std, "cuda", experts=[e])[0]
    W2 = WL.w2(w.cfg_id, 1, n, d, w.w_std, "cuda", experts=[e])[0]
    return f64(W1), f64(W2)


def _token_rows(cols, key, std, toks):
    idx = (torch.as_tensor(toks, dtype=torch.int64)[:, None] * cols +
           torch.arange(cols, dtype=torch.int64)[None, :]).cuda()
    return f64(WL.normal_at(idx, key, std))


def dy_exact(w, ro, probs, rows):
    """p * dO of the given rows before the bf16 rounding (pad rows zero)."""
    pairs = ro["pair_of_row"][rows]
    real = pairs >= 0
    out = np.zeros((len(rows), w.d))
    if real.any():
        dO = _token_rows(w.d, (w.cfg_id, WL.DO, 0), w.dy_std, pairs[real] // w.k)
        out[real] = O.permute(dO, np.arange(int(real.sum())), 1,
                              scale=probs.reshape(-1)[pairs[real]], round_out=False)
    return out


def _expert_inputs(w, ro, probs, rows):
    """x_perm and dy_perm rows (pad rows zero), from the generator."""
    pairs = ro["pair_of_row"][rows]
    real = pairs >= 0
    x = np.zeros((len(rows), w.d))
    dy = np.zeros((len(rows), w.d))
    if real.any():
        toks = pairs[real] // w.k
        x[real] = _token_rows(w.d, (w.cfg_id, WL.X, 0), w.x_std, toks)
        dO = _token_rows(w.d, (w.cfg_id, WL.DO, 0), w.dy_std, toks)
        dy[real] = O.bf16_round(probs.reshape(-1)[pairs[real]].astype(np.float64)[:, None] * dO)
    return x, dy


@pytest.fixture(scope="module")
def run():
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    w = WL.WORKLOADS[WNAME]
    inp, o = BE.make_inputs(w, "cuda")
    step = BE.make_step(w, inp, o)
    step()
    torch.cuda.synchronize()
    assert int(o["err"].item()) == 0
    idx, probs = WL.route_inputs(w)
    ro = O.route_offsets(idx, w.E, w.align, w.M_cap)
    yield w, o, ro, probs
    del inp, o
    torch.cuda.empty_cache()


def test_mx_rows_forward_and_data_gradients(run):
    w, o, ro, probs = run
    counts, off = ro["counts"], ro["offsets"]
    nonempty = [int(e) for e in np.argsort(counts) if counts[e] > 0]
    rng = np.random.default_rng(11)
    for e in [int(np.argmax(counts)), nonempty[len(nonempty) // 2], nonempty[0]]:
        W1, W2 = _expert_weights(w, e)
        rr = np.arange(off[e], off[e] + counts[e])          # real rows
        rows = rr if len(rr) <= 6 else np.sort(rng.choice(rr, 6, replace=False))
        x, dy = _expert_inputs(w, ro, probs, rows)
        o1 = np.array([0, len(rows)])
        _, A, _ = O.grouped_mlp_fwd(x, o1, W1[None], W2[None], w.act, round_out=False)
        r = torch.as_tensor(rows).cuda()
        # each block-scaled GEMM on its own inputs, the GPU's stored bf16
        # operands: FC2 from A (row-wise MX, W2 with blocks along n); FC2-dgrad
        # + dAct from dY and H (dY and W2 with blocks along d); FC1-dgrad from
        # dH (dH and W1 with blocks along n1)
        ga, gh = f64(o["a"][r]), f64(o["h"][r])
        gdy, gdh = f64(o["dy_perm"][r]), f64(o["dh"][r])
        qa, sa = X.mx_quantize_rows(ga)
        qw, sw = X.mx_quantize_weights(W2[None])
        Y = X.mx_fc2(qa, sa, qw, sw, o1)
        dyq, dys = X.mx_quantize_rows(gdy)
        w2q, w2s = X.mx_quantize_rows(W2)
        dA = X.mx_dgrad(dyq, dys, w2q[None], w2s[None], o1)
        dH = O.act_backward(gh, dA, w.act)
        dhq, dhs = X.mx_quantize_rows(gdh)
        w1q, w1s = X.mx_quantize_rows(W1)
        dX = X.mx_dgrad(dhq, dhs, w1q[None], w1s[None], o1)
        # the scaled permute's dY against the generator's dO times the probability
        assert_rms_close(gdy, dy_exact(w, ro, probs, rows), f"MX e{e} dY")
        assert_rms_close(f64(o["a"][r]), A, f"MX e{e} A")
        assert_rms_close(f64(o["y_perm"][r]), Y, f"MX e{e} Y")
        assert_rms_close(f64(o["dh"][r]), dH, f"MX e{e} dH")
        assert_rms_close(f64(o["dx_perm"][r]), dX, f"MX e{e} dX")


def test_mx_fc1_codes_and_scales_bit_exact(run):
    """The FC1 epilogue's E4M3 codes and E8M0 scales of A, row-wise (1x32
    along n, MMA-tiled scales) and transposed (32x1 along the rows of one
    expert), equal the OCP MX quantiser applied to the GPU's own bf16 A on
    every block of three experts: the largest, a median one and the
    smallest (pad rows up to the 32-row boundary included)."""
    w, o, ro, probs = run
    counts, off = ro["counts"], ro["offsets"]
    mx = o["mx"]
    n, Mc = w.n, w.M_cap
    nonempty = [int(e) for e in np.argsort(counts) if counts[e] > 0]
    gs_all = decode_a_scales(mx["a_s"], off, Mc, n)
    for e in [int(np.argmax(counts)), nonempty[len(nonempty) // 2], nonempty[0]]:
        r0, r1 = int(off[e]), int(off[e + 1])
        assert r0 % 32 == 0 and r1 % 32 == 0 and r1 > r0
        ga = f64(o["a"][r0:r1])
        qo, so = X.mx_quantize_rows(ga)
        gq = mx["a_q"][r0:r1].cpu().numpy()
        assert np.array_equal(gq, qo), (e, "row-wise codes",
                                        int((gq != qo).sum()), "of", qo.size)
        assert np.array_equal(gs_all[r0:r1], so), (e, "row-wise scales")
        qTo, sTo = X.mx_quantize_cols(ga, np.array([0, r1 - r0]))
        gqT = mx["a_qT"][:, r0:r1].cpu().numpy()
        gsT = mx["a_sT"][:, r0 // 32:r1 // 32].cpu().numpy()
        assert np.array_equal(gqT, qTo), (e, "transposed codes",
                                          int((gqT != qTo).sum()), "of", qTo.size)
        assert np.array_equal(gsT, sTo), (e, "transposed scales")


def test_mx_weight_gradients_small_expert_and_empty(run):
    """Whole dW1/dW2 of a small expert, two ways.
      * Stage-wise, element-wise: the oracle's block-scaled weight gradient
        (group-aware transposed copies, exact products, fp64 sums) of the
        GPU's own bf16 operands - A from its FC1, dY from its scaled
        permute, dH from its FC2-dgrad, x from the generator - against every
        entry of the GPU's dW within the bf16 tolerance.
      * The independent chain: the oracle's MXFP8 backward from x, where
        each side quantises operands it computed itself (a one-step bf16
        difference can flip an E4M3 code, which shows in a sum over a few
        dozen rows): relative Frobenius error <= 2e-2 over the whole dW."""
    w, o, ro, probs = run
    counts, off = ro["counts"], ro["offsets"]
    e = int([e for e in np.argsort(counts) if counts[e] > 40][0])   # two 32-row blocks or more
    W1, W2 = _expert_weights(w, e)
    rows = np.arange(off[e], off[e + 1])                 # padded to a multiple of 32
    x, dy = _expert_inputs(w, ro, probs, rows)
    o1 = np.array([0, len(rows)])
    H, A, _ = O.grouped_mlp_fwd(x, o1, W1[None], W2[None], w.act)
    ref = X.mx_grouped_mlp_bwd(x, H, A, dy, o1, W1[None], W2[None], w.act)
    r = torch.as_tensor(rows).cuda()
    got2, got1 = f64(o["dW2"][e]), f64(o["dW1"][e])
    for name, got, want in (("dW2", got2, ref["dW2"][0]), ("dW1", got1, ref["dW1"][0])):
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel <= 2e-2, (f"MX {name}[{e}] relative error", rel)
    # stage-wise: the oracle's block-scaled wgrad on the GPU's own operands
    ga, gdy, gdh = f64(o["a"][r]), f64(o["dy_perm"][r]), f64(o["dh"][r])
    want2 = X.mx_wgrad(*X.mx_quantize_cols(ga, o1), *X.mx_quantize_cols(gdy, o1), o1)[0]
    want1 = X.mx_wgrad(*X.mx_quantize_cols(x, o1), *X.mx_quantize_cols(gdh, o1), o1)[0]
    assert_rms_close(got2, want2, f"MX dW2[{e}] from the GPU's own A, dY")
    assert_rms_close(got1, want1, f"MX dW1[{e}] from the GPU's own dH")
    for e in [int(e) for e in range(w.E) if counts[e] == 0][:3]:
        assert float(o["dW1"][e].abs().max()) == 0.0
        assert float(o["dW2"][e].abs().max()) == 0.0


BAL = "balanced_e8_m4096_k8192_n4096_mxfp8_train"


@pytest.fixture(scope="module")
def bal_run():
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    w = WL.WORKLOADS[BAL]
    inp, o = BE.make_inputs(w, "cuda")
    step = BE.make_step(w, inp, o)
    step()
    torch.cuda.synchronize()
    assert int(o["err"].item()) == 0
    yield w, inp, o
    del inp, o
    torch.cuda.empty_cache()


def _bal_rows(w, key, std, rows):
    idx = (torch.as_tensor(rows, dtype=torch.int64)[:, None] * w.d +
           torch.arange(w.d, dtype=torch.int64)[None, :]).cuda()
    return f64(WL.normal_at(idx, key, std))


def test_mx_balanced_rows_each_gemm_on_its_inputs(bal_run):
    """The balanced MXFP8 training step (E=8 x 4096 rows, d=8192, 2n=4096;
    pair mode, six-stage reductions of 64 steps): sampled rows of experts 0
    and 5.  A against the oracle from x; each block-scaled GEMM on the
    GPU's own stored operands, quantised by the oracle: Y (FC2 from A), dH
    (FC2-dgrad + dAct from dY and H), dX (FC1-dgrad from dH); the fused
    FC1 epilogue's codes of A and FC2-dgrad's bf16 dH round trip."""
    w, inp, o = bal_run
    m = w.T // w.E
    rng = np.random.default_rng(7)
    for e in (0, 5):
        W1, W2 = _expert_weights(w, e)
        rows = e * m + np.sort(rng.choice(m, 4, replace=False))
        x = _bal_rows(w, (w.cfg_id, WL.X, 0), w.x_std, rows)
        o1 = np.array([0, len(rows)])
        _, A, _ = O.grouped_mlp_fwd(x, o1, W1[None], W2[None], w.act, round_out=False)
        r = torch.as_tensor(rows).cuda()
        ga, gh, gdh = f64(o["a"][r]), f64(o["h"][r]), f64(o["dh"][r])
        gdy = f64(inp["dy_perm"][r])
        qa, sa = X.mx_quantize_rows(ga)
        qw, sw = X.mx_quantize_weights(W2[None])
        Y = X.mx_fc2(qa, sa, qw, sw, o1)
        dyq, dys = X.mx_quantize_rows(gdy)
        w2q, w2s = X.mx_quantize_rows(W2)
        dH = O.act_backward(gh, X.mx_dgrad(dyq, dys, w2q[None], w2s[None], o1), w.act)
        dhq, dhs = X.mx_quantize_rows(gdh)
        w1q, w1s = X.mx_quantize_rows(W1)
        dX = X.mx_dgrad(dhq, dhs, w1q[None], w1s[None], o1)
        assert_rms_close(ga, A, f"balanced MX e{e} A")
        assert_rms_close(f64(o["y_perm"][r]), Y, f"balanced MX e{e} Y")
        assert_rms_close(gdh, dH, f"balanced MX e{e} dH")
        assert_rms_close(f64(o["dx_perm"][r]), dX, f"balanced MX e{e} dX")
        assert np.array_equal(o["mx"]["a_q"][r].cpu().numpy(), qa)


def test_mx_balanced_weight_gradient_entries(bal_run):
    """dW1[e][k, c] = sum over the expert's 4096 rows of deq(x^T)[k] deq(dH^T)[c]
    and dW2[e][j, c] = sum deq(A^T)[j] deq(dY^T)[c], for sampled (k | j, c),
    from the GPU's own bf16 dH and A and the generator's x and dY, each
    column quantised in 32-row blocks of the expert by the oracle."""
    w, inp, o = bal_run
    m = w.T // w.E
    e = 3
    rows = np.arange(e * m, (e + 1) * m)
    r = torch.as_tensor(rows).cuda()
    rng = np.random.default_rng(8)
    ks = np.sort(rng.choice(w.d, 16, replace=False))
    cs = np.sort(rng.choice(w.n1, 16, replace=False))
    js = np.sort(rng.choice(w.n, 16, replace=False))
    cd = np.sort(rng.choice(w.d, 16, replace=False))
    o1 = np.array([0, m])
    x = f64(inp["x_perm"][r][:, torch.as_tensor(ks).cuda()])
    gdh = f64(o["dh"][r][:, torch.as_tensor(cs).cuda()])
    ga = f64(o["a"][r][:, torch.as_tensor(js).cuda()])
    gdy = f64(inp["dy_perm"][r][:, torch.as_tensor(cd).cuda()])
    want1 = X.mx_wgrad(*X.mx_quantize_cols(x, o1), *X.mx_quantize_cols(gdh, o1), o1)[0]
    want2 = X.mx_wgrad(*X.mx_quantize_cols(ga, o1), *X.mx_quantize_cols(gdy, o1), o1)[0]
    got1 = f64(o["dW1"][e][torch.as_tensor(ks).cuda()][:, torch.as_tensor(cs).cuda()])
    got2 = f64(o["dW2"][e][torch.as_tensor(js).cuda()][:, torch.as_tensor(cd).cuda()])
    assert_rms_close(got1, want1, "balanced MX dW1 entries")
    assert_rms_close(got2, want2, "balanced MX dW2 entries")
