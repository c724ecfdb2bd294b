"""Pins for the oracle's MXFP8 backward (oracle/mx.py: mx_dgrad, mx_wgrad,
mx_grouped_mlp_bwd).

* Operands built to be exactly representable in MXFP8 along the right axis
  quantise without loss, so the block-scaled contractions must equal the
  plain products of the bf16 values exactly; the same operands quantised
  along the wrong axis lose bits, so an axis mistake cannot pass.
* MX quantisation, bf16 rounding and the activation derivatives all commute
  with multiplication by a power of two, so scaling one input by 2^k must
  scale exactly the outputs that depend on it linearly and leave the others
  bit-identical; this pins which operand feeds which contraction.
* On ordinary bf16 inputs the result stays within MXFP8's error of the
  plain (unquantised) backward."""
import numpy as np
import pytest

import oracle as O
from oracle import mx as X

BIG = np.array([256.0, 288.0, 320.0, 352.0, 384.0, 416.0, 448.0])


def _codes_values(rng, shape):
    """Random finite E4M3 values (any code but NaN), random sign."""
    c = rng.integers(0, 0x7F, size=shape)
    v = X.e4m3_decode(c.astype(np.uint8))
    return np.where(rng.random(shape) < 0.5, -v, v)


def _exact(rng, exps):
    """Values q * 2^exps[r, c] with q an E4M3 value; on every position with
    r % 32 == c % 32 the magnitude is in [256, 448], so each 32-block along
    either axis that has a constant exponent holds one such value and
    quantises to exactly these codes with scale 2^exps."""
    R, C = exps.shape
    q = _codes_values(rng, (R, C))
    rr, cc = np.meshgrid(np.arange(R), np.arange(C), indexing="ij")
    diag = (rr % 32) == (cc % 32)
    big = rng.choice(BIG, size=(R, C)) * np.where(rng.random((R, C)) < 0.5, -1, 1)
    q = np.where(diag, big, q)
    return q * np.ldexp(1.0, exps)


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def test_mx_dgrad_exact_on_representable_operands():
    rng = np.random.default_rng(40)
    off = _offsets([64, 0, 32, 96])
    M, K, N, E = int(off[-1]), 128, 64, 4
    # G: blocks along K (row-wise): exponent constant on each (row, 32-col) block
    g_exp = rng.integers(-6, 7, size=(M, 1)) + np.repeat(rng.integers(-4, 5, size=(1, K // 32)), 32, 1)
    G = _exact(rng, g_exp)
    # W_e [N, K]: blocks along K; the exponent varies along N so that
    # blocks along N would mix exponents
    W = np.stack([_exact(rng, rng.integers(-6, 7, size=(N, 1)) +
                         np.repeat(rng.integers(-3, 4, size=(1, K // 32)), 32, 1)) for _ in range(E)])
    g_q, g_s = X.mx_quantize_rows(G)
    assert np.array_equal(X.mx_dequantize(g_q, g_s, 1), G)          # lossless
    w_q, w_s = X.mx_quantize_rows(W.reshape(E * N, K))
    w_q, w_s = w_q.reshape(E, N, K), w_s.reshape(E, N, K // 32)
    out = X.mx_dgrad(g_q, g_s, w_q, w_s, off)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        assert np.array_equal(out[r0:r1], G[r0:r1] @ W[e].T)
    # planted mistake: W quantised with blocks along N (its other axis)
    bad_q, bad_s = X.mx_quantize_cols(W.reshape(E * N, K), np.arange(0, E * N + 1, N), E * N)
    bad = X.mx_dequantize(bad_q, bad_s, 1).T.reshape(E, N, K)
    assert not np.array_equal(bad, W)


def test_mx_wgrad_exact_on_representable_operands():
    rng = np.random.default_rng(41)
    off = _offsets([96, 32, 0, 64])
    M, p, q, E = int(off[-1]), 64, 96, 4
    # blocks of 32 rows inside an expert: exponent constant along rows of a
    # block, varying per column (row-wise blocks would mix exponents)
    def col_exact(C):
        exps = np.repeat(rng.integers(-5, 6, size=(M // 32, 1)), 32, 0) + rng.integers(-6, 7, size=(1, C))
        return _exact(rng, exps)
    P, Q = col_exact(p), col_exact(q)
    p_qT, p_sT = X.mx_quantize_cols(P, off, M)
    q_qT, q_sT = X.mx_quantize_cols(Q, off, M)
    assert np.array_equal(X.mx_dequantize(p_qT, p_sT, 1), P.T)
    dW = X.mx_wgrad(p_qT, p_sT, q_qT, q_sT, off)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        assert np.array_equal(dW[e], P[r0:r1].T @ Q[r0:r1])
    assert (dW[2] == 0).all()
    # planted mistake: the same operand with row-wise blocks loses bits
    r_q, r_s = X.mx_quantize_rows(P)
    assert not np.array_equal(X.mx_dequantize(r_q, r_s, 1), P)


def _layer(rng, counts, d, n, act, std=0.05):
    off = _offsets(counts)
    M = int(off[-1]) + 32
    E = len(counts)
    n1 = n if act == "srelu" else 2 * n
    bf = lambda s, sd: O.bf16_round(rng.standard_normal(s) * sd)
    return dict(x=bf((M, d), 1.0), H=bf((M, n1), 1.0), A=bf((M, n), 1.0), dY=bf((M, d), 1.0),
                W1=bf((E, d, n1), std), W2=bf((E, n, d), std), off=off)


def _run(L, act):
    return X.mx_grouped_mlp_bwd(L["x"], L["H"], L["A"], L["dY"], L["off"], L["W1"], L["W2"], act)


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_power_of_two_equivariance(act):
    """Each input reaches exactly the outputs that are linear in it."""
    rng = np.random.default_rng(42)
    L = _layer(rng, [64, 0, 96, 32], 64, 64, act)
    R = int(L["off"][-1])
    base = _run(L, act)
    # which outputs scale (by the input's factor) when each input is scaled
    cases = {"dY": (8.0, {"dH", "dX", "dW1", "dW2"}),
             "W2": (0.25, {"dH", "dX", "dW1"}),
             "W1": (4.0, {"dX"}),
             "x": (2.0, {"dW1"}),
             "A": (0.5, {"dW2"})}
    for name, (f, scaled) in cases.items():
        L2 = dict(L)
        L2[name] = L[name] * f
        got = _run(L2, act)
        for out in ("dH", "dX", "dW1", "dW2"):
            a, b = got[out], base[out]
            if out in ("dH", "dX"):
                a, b = a[:R], b[:R]
            want = b * f if out in scaled else b
            assert np.array_equal(a, want), (name, out)


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_representable_inputs_match_plain_backward(act):
    """dY representable along both axes, W2 along d and A along rows: dH and
    dW2 equal the plain (unquantised) backward exactly."""
    rng = np.random.default_rng(43)
    counts = [64, 0, 32, 96]
    off = _offsets(counts)
    M, E, d, n = int(off[-1]), 4, 64, 64
    n1 = n if act == "srelu" else 2 * n
    tile = lambda R, C, lo, hi: np.kron(rng.integers(lo, hi, size=(R // 32, C // 32)), np.ones((32, 32), int))
    dY = _exact(rng, tile(M, d, -4, 5))
    W2 = np.stack([_exact(rng, rng.integers(-8, -2, size=(n, 1)) +
                          np.repeat(rng.integers(-2, 3, size=(1, d // 32)), 32, 1)) for _ in range(E)])
    A = _exact(rng, np.repeat(rng.integers(-3, 4, size=(M // 32, 1)), 32, 0) + rng.integers(-4, 5, size=(1, n)))
    H = O.bf16_round(rng.standard_normal((M, n1)))
    x = O.bf16_round(rng.standard_normal((M, d)))
    W1 = O.bf16_round(rng.standard_normal((E, d, n1)) * 0.05)
    got = X.mx_grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act)
    dH, _, _, dW2 = O.grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act)
    assert np.array_equal(got["dH"], dH)
    assert np.array_equal(got["dW2"], dW2)


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_close_to_plain_backward(act):
    """Ordinary bf16 inputs: within MXFP8's error of the unquantised result.
    E4M3 keeps 3 mantissa bits (a relative step of 2^-3 inside a binade, so
    about 3% RMS error per quantised operand): dH and dW2 contract two
    quantised operands (about 4% measured), dX and dW1 also quantise the
    already perturbed dH (about 6%)."""
    rng = np.random.default_rng(44)
    L = _layer(rng, [96, 0, 64, 32, 128], 128, 64, act)
    R = int(L["off"][-1])
    got = _run(L, act)
    ref = O.grouped_mlp_bwd(L["x"], L["H"], L["A"], L["dY"], L["off"], L["W1"], L["W2"], act)
    for name, a, b in zip(("dH", "dX", "dW1", "dW2"), (got["dH"], got["dX"], got["dW1"], got["dW2"]), ref):
        if name in ("dH", "dX"):
            a, b = a[:R], b[:R]
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        bound = 0.06 if name in ("dH", "dW2") else 0.09
        assert 0.01 < rel < bound, (name, rel)
    assert (got["dW1"][1] == 0).all() and (got["dW2"][1] == 0).all()
    assert np.isnan(got["dH"][R:]).all()
