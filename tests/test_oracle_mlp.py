"""Pins for the oracle's grouped expert MLP (forward and backward).

Pinned by brute-force scalar loops on tiny inputs, the interleaved-vs-split
weight equivalence, closed forms of the activations, central finite
differences of the activations and of the whole layer, and the empty-group
and zero-token invariants."""
import math

import numpy as np
import pytest

import oracle as O

ACTS = ["swiglu", "geglu", "srelu"]


def _scalar_act(h_row, act):
    """Pure-Python activation of one H row (brute force)."""
    out = []
    if act == "srelu":
        return [max(v, 0.0) ** 2 for v in h_row]
    for j in range(len(h_row) // 2):
        g, u = h_row[2 * j], h_row[2 * j + 1]
        if act == "swiglu":
            ph = g / (1.0 + math.exp(-g))
        else:
            ph = 0.5 * g * (1.0 + math.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)))
        out.append(ph * u)
    return out


def _tiny(act, rng, rows=(2, 0, 3), d=4, n=3):
    E = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)])
    M = int(off[-1])
    n1 = 2 * n if act != "srelu" else n
    x = rng.standard_normal((M, d))
    W1 = rng.standard_normal((E, d, n1)) * 0.5
    W2 = rng.standard_normal((E, n, d)) * 0.5
    return off, x, W1, W2


@pytest.mark.parametrize("act", ACTS)
def test_fwd_brute_force(act):
    rng = np.random.default_rng(10)
    off, x, W1, W2 = _tiny(act, rng)
    H, A, Y = O.grouped_mlp_fwd(x, off, W1, W2, act, round_bf16=False)
    E = len(off) - 1
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            h = [sum(x[r][i] * W1[e][i][c] for i in range(x.shape[1])) for c in range(W1.shape[2])]
            a = _scalar_act(h, act)
            y = [sum(a[j] * W2[e][j][c] for j in range(len(a))) for c in range(W2.shape[2])]
            assert np.allclose(H[r], h, rtol=0, atol=1e-12)
            assert np.allclose(A[r], a, rtol=0, atol=1e-12)
            assert np.allclose(Y[r], y, rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_interleaved_equals_split(act):
    """Interleaving is a column permutation of concatenated [gate | up]
    weights (the TE page's prefused (E, d, 2*mlp) layout): A from the
    interleaved layout equals phi(X Wg) * (X Wu)."""
    rng = np.random.default_rng(11)
    E, d, n = 3, 8, 5
    Wg = rng.standard_normal((E, d, n))
    Wu = rng.standard_normal((E, d, n))
    W1 = O.interleave_gate_up(Wg, Wu)
    g2, u2 = O.split_gate_up(W1)
    assert (g2 == Wg).all() and (u2 == Wu).all()
    assert (W1[..., :: 2] == Wg).all()
    W2 = rng.standard_normal((E, n, d))
    off = np.array([0, 4, 4, 9])
    x = rng.standard_normal((9, d))
    _, A, _ = O.grouped_mlp_fwd(x, off, W1, W2, act, round_bf16=False)
    concat = np.concatenate([Wg, Wu], axis=2)        # [gate | up]
    for e in range(E):
        xe = x[off[e]:off[e + 1]]
        hc = xe @ concat[e]
        g, u = hc[:, :n], hc[:, n:]
        assert np.allclose(A[off[e]:off[e + 1]], O.phi(g, act) * u, rtol=1e-13, atol=1e-13)


def test_activation_closed_forms():
    g = np.linspace(-8, 8, 2001)
    silu = O.phi(g, "swiglu")
    assert O.phi(np.array([0.0]), "swiglu")[0] == 0.0
    assert np.allclose(O.phi(-g, "swiglu"), silu - g, atol=1e-12)   # silu(-x) = silu(x) - x
    assert abs(O.phi(np.array([50.0]), "swiglu")[0] - 50.0) < 1e-18 + 1e-12
    # tanh-GELU against exact erf-GELU x*Phi(x): a wrong constant breaks this
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in g])
    assert np.abs(O.phi(g, "geglu") - exact).max() < 1e-3
    assert O.phi(np.array([0.0]), "geglu")[0] == 0.0
    h = np.array([-2.0, -0.0, 0.0, 0.5, 3.0])
    assert O.act_forward(h, "srelu").tolist() == [0.0, 0.0, 0.0, 0.25, 9.0]


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_dphi_finite_difference(act):
    g = np.linspace(-7, 7, 301)
    eps = 1e-5
    fd = (O.phi(g + eps, act) - O.phi(g - eps, act)) / (2 * eps)
    assert np.abs(fd - O.dphi(g, act)).max() < 1e-8


@pytest.mark.parametrize("act", ACTS)
def test_act_backward_finite_difference(act):
    rng = np.random.default_rng(12)
    h = rng.standard_normal((3, 8)) * 2
    dA = rng.standard_normal((3, 8 if act == "srelu" else 4))
    dH = O.act_backward(h, dA, act)
    eps = 1e-6
    for idx in np.ndindex(h.shape):
        hp, hm = h.copy(), h.copy()
        hp[idx] += eps
        hm[idx] -= eps
        fd = ((O.act_forward(hp, act) - O.act_forward(hm, act)) * dA).sum() / (2 * eps)
        assert abs(fd - dH[idx]) < 1e-6


@pytest.mark.parametrize("act", ACTS)
def test_layer_gradient_finite_difference(act):
    """L = sum(dY * Y) on an unrounded tiny layer with an empty expert:
    dX, dW1, dW2 from grouped_mlp_bwd equal central differences."""
    rng = np.random.default_rng(13)
    off, x, W1, W2 = _tiny(act, rng, rows=(3, 0, 2), d=5, n=3)
    dY = rng.standard_normal((x.shape[0], W2.shape[2]))

    def L(x_, W1_, W2_):
        _, _, Y = O.grouped_mlp_fwd(x_, off, W1_, W2_, act, round_bf16=False)
        return float((dY * Y).sum())

    H, A, _ = O.grouped_mlp_fwd(x, off, W1, W2, act, round_bf16=False)
    dH, dX, dW1, dW2 = O.grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act, round_bf16=False)
    eps = 1e-6
    for arr, grad, name in [(x, dX, "x"), (W1, dW1, "W1"), (W2, dW2, "W2")]:
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = {"x": (p, W1, W2), "W1": (x, p, W2), "W2": (x, W1, p)}[name]
            args_m = {"x": (m, W1, W2), "W1": (x, m, W2), "W2": (x, W1, m)}[name]
            fd = (L(*args_p) - L(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-5, (name, idx)
    # the empty expert's weight gradients are exactly zero
    assert (dW1[1] == 0).all() and (dW2[1] == 0).all()


def test_special_cases_zero_grads():
    h = np.array([[-1.0, 2.0, -0.5, 0.0]])
    dA = np.ones((1, 4))
    assert (O.act_backward(h, dA, "srelu")[0] == [0, 4.0, 0, 0]).all()
    # SwiGLU with up = 0: output 0 and gate gradient 0
    hg = np.array([[1.3, 0.0, -2.0, 0.0]])
    assert (O.act_forward(hg, "swiglu") == 0).all()
    assert (O.act_backward(hg, np.ones((1, 2)), "swiglu")[0, 0::2] == 0).all()


@pytest.mark.parametrize("act", ACTS)
def test_zero_tokens(act):
    rng = np.random.default_rng(14)
    E, d, n = 3, 4, 2
    n1 = n if act == "srelu" else 2 * n
    off = np.zeros(E + 1, np.int64)
    x = np.zeros((0, d))
    W1 = rng.standard_normal((E, d, n1))
    W2 = rng.standard_normal((E, n, d))
    H, A, Y = O.grouped_mlp_fwd(x, off, W1, W2, act)
    assert H.shape == (0, n1) and A.shape == (0, n) and Y.shape == (0, d)
    dH, dX, dW1, dW2 = O.grouped_mlp_bwd(x, H, A, np.zeros((0, d)), off, W1, W2, act)
    assert (dW1 == 0).all() and (dW2 == 0).all() and dX.shape == (0, d)


def test_rounding_points():
    """With round_bf16=True every stored tensor is bf16-representable, and A
    is computed from the unrounded H."""
    rng = np.random.default_rng(15)
    off, x, W1, W2 = _tiny("swiglu", rng, rows=(5, 3, 4), d=16, n=8)
    x = O.bf16_round(x)
    W1 = O.bf16_round(W1)
    W2 = O.bf16_round(W2)
    H, A, Y = O.grouped_mlp_fwd(x, off, W1, W2, "swiglu")
    for t in (H, A, Y):
        assert (O.bf16_round(t) == t).all()
    Hr, Ar, _ = O.grouped_mlp_fwd(x, off, W1, W2, "swiglu", round_bf16=False)
    assert (A == O.bf16_round(Ar)).all()


def _routed_case(act, seed=50):
    rng = np.random.default_rng(seed)
    E, d, n = 3, 16, 8
    n1 = n if act == "srelu" else 2 * n
    off = np.array([0, 5, 5, 12])
    M = 14                                          # two rows past every expert
    x = rng.standard_normal((M, d))
    H = rng.standard_normal((M, n1))
    dO = rng.standard_normal((M, d))
    p = rng.random(M)
    W1 = rng.standard_normal((E, d, n1)) * 0.3
    W2 = rng.standard_normal((E, n, d)) * 0.3
    return x, H, dO, p, off, W1, W2


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_routed_backward_equals_scaled_backward(act):
    """With dY = p * dO the routed backward ([Sonic] rewrite) gives the same
    dH, dX, dW1 and dW2 as the plain backward, and A' = p * act(H)."""
    x, H, dO, p, off, W1, W2 = _routed_case(act)
    dH, dX, dW1, dW2, Ap, dS = O.grouped_mlp_bwd_routed(x, H, dO, p, off, W1, W2, act,
                                                         round_bf16=False)
    A = O.act_forward(H, act)
    ref = O.grouped_mlp_bwd(x, H, A, p[:, None] * dO, off, W1, W2, act, round_bf16=False)
    R = int(off[-1])
    for got, want in zip((dH, dX, dW1, dW2), ref):
        if got.shape[0] == x.shape[0]:
            got, want = got[:R], want[:R]
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(Ap[:R], p[:R, None] * A[:R], rtol=1e-15, atol=0)
    assert np.isnan(dS[R:]).all()


@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_routed_router_gradient_finite_difference(act):
    """dS_r is the derivative, w.r.t. the row's router probability p_r, of
    L(p) = sum_r p_r <dO_r, Y_r> with Y = act(H) W2 computed forward."""
    x, H, dO, p, off, W1, W2 = _routed_case(act, seed=51)
    _, _, _, _, _, dS = O.grouped_mlp_bwd_routed(x, H, dO, p, off, W1, W2, act, round_bf16=False)
    A = O.act_forward(H, act)

    def loss(pv):
        tot = 0.0
        for e in range(len(off) - 1):
            r0, r1 = off[e], off[e + 1]
            tot += float((pv[r0:r1, None] * dO[r0:r1] * (A[r0:r1] @ W2[e])).sum())
        return tot
    eps = 1e-6
    for r in range(int(off[-1])):
        pp, pm = p.copy(), p.copy()
        pp[r] += eps
        pm[r] -= eps
        assert abs((loss(pp) - loss(pm)) / (2 * eps) - dS[r]) < 1e-6


def test_routed_pad_rows_and_empty_expert():
    """A pad row (p = 0, dO = 0) contributes nothing; an empty expert gets
    zero weight gradients."""
    x, H, dO, p, off, W1, W2 = _routed_case("swiglu", seed=52)
    p[3] = 0.0
    dO[3] = 0.0
    dH, _, dW1, dW2, Ap, dS = O.grouped_mlp_bwd_routed(x, H, dO, p, off, W1, W2, "swiglu")
    assert dS[3] == 0 and (Ap[3] == 0).all() and (dH[3] == 0).all()
    assert (dW1[1] == 0).all() and (dW2[1] == 0).all()


def test_amax_is_the_largest_magnitude():
    """Per-tensor amax: the largest |value|, whichever its sign; 0 for an
    empty or all-zero tensor."""
    assert O.amax(np.array([[-3.0, 2.0], [0.5, -0.25]])) == 3.0
    assert O.amax(np.array([1.5, -1.5])) == 1.5
    assert O.amax(np.zeros((0, 4))) == 0.0 and O.amax(np.zeros(3)) == 0.0


def test_hadamard16_pins():
    """Sylvester's recursion H_{2m} = [[H, H], [H, -H]] gives the same matrix;
    it is orthonormal and symmetric."""
    h = np.array([[1.0]])
    for _ in range(4):
        h = np.block([[h, h], [h, -h]])
    assert np.array_equal(O.hadamard16(), h / 4.0)
    assert np.allclose(O.hadamard16() @ O.hadamard16(), np.eye(16), atol=1e-15)


def test_amax_rht_transposed_special_cases():
    """One nonzero v in a block -> |v|/4; a constant block c -> 4|c| (all of
    it in the first coefficient); Parseval: the rotated block keeps its sum of
    squares; blocks start at each expert's first row, the last one padded."""
    G = np.zeros((40, 3))
    G[5, 0] = -8.0
    assert O.amax_rht_transposed(G, [0, 40]) == 2.0
    G = np.zeros((40, 2))
    G[16:32, 1] = 0.5
    assert O.amax_rht_transposed(G, [0, 40]) == 2.0
    # an expert starting at row 3: its first block is rows 3..18, so a
    # constant run on rows 3..18 rotates to 4c, while on rows 0..15 (crossing
    # the block start) it would not
    G = np.zeros((40, 1))
    G[3:19, 0] = 1.0
    assert O.amax_rht_transposed(G, [0, 3, 40]) == 4.0
    assert O.amax_rht_transposed(G, [0, 40]) < 4.0
    rng = np.random.default_rng(53)
    blk = rng.standard_normal((16, 4))
    rot = O.hadamard16() @ blk
    assert np.allclose((rot ** 2).sum(0), (blk ** 2).sum(0))
    assert np.isclose(O.amax_rht_transposed(blk, [0, 16]), np.abs(rot).max())
    assert O.amax(np.array([[-3.0, 2.0]])) == 3.0 and O.amax(np.zeros((0, 4))) == 0.0


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_grouped_gemm_brute_force(layout):
    """The plain grouped GEMM against scalar loops on tiny ragged groups
    (one of them empty; rows past the last expert stay undefined)."""
    rng = np.random.default_rng(14)
    rows = (2, 0, 3)
    off = np.concatenate([[0], np.cumsum(rows)])
    K, N = 5, 4
    a = rng.standard_normal((int(off[-1]) + 1, K))
    B = rng.standard_normal((3, K, N) if layout == "kn" else (3, N, K))
    out = O.grouped_gemm(a, off, B, layout, round_bf16=False)
    for e in range(3):
        for r in range(off[e], off[e + 1]):
            for c in range(N):
                b = [B[e][i][c] if layout == "kn" else B[e][c][i] for i in range(K)]
                assert abs(out[r][c] - sum(a[r][i] * b[i] for i in range(K))) < 1e-12
    assert np.isnan(out[int(off[-1])]).all()


def test_grouped_gemm_is_the_mlp_fc2():
    """FC2 of the grouped MLP is the grouped GEMM of A with W2, and the
    transposed layout of W2 gives the same result (bf16 rounding included)."""
    rng = np.random.default_rng(15)
    off, x, W1, W2 = _tiny("swiglu", rng)
    H, A, Y = O.grouped_mlp_fwd(x, off, W1, W2, "swiglu")
    R = int(off[-1])
    assert np.array_equal(O.grouped_gemm(A, off, W2)[:R], Y[:R])
    assert np.array_equal(O.grouped_gemm(A, off, np.swapaxes(W2, 1, 2).copy(), "nk")[:R], Y[:R])


def test_grouped_wgrad_brute_force():
    """dW_e = P_e^T Q_e against scalar loops over the rows of each expert
    (an empty expert gives exact zeros; rows past the last expert are not
    read)."""
    rng = np.random.default_rng(16)
    rows = (3, 0, 2)
    off = np.concatenate([[0], np.cumsum(rows)])
    P = rng.standard_normal((int(off[-1]) + 2, 4))
    Q = rng.standard_normal((int(off[-1]) + 2, 3))
    P[-2:] = np.nan
    dW = O.grouped_wgrad(P, Q, off, round_out=False)
    assert dW.shape == (3, 4, 3)
    for e in range(3):
        for i in range(4):
            for j in range(3):
                want = sum(P[r][i] * Q[r][j] for r in range(off[e], off[e + 1]))
                assert abs(dW[e][i][j] - want) < 1e-12
    assert (dW[1] == 0).all()


@pytest.mark.parametrize("act", ACTS)
def test_grouped_wgrad_is_the_mlp_weight_gradients(act):
    """grouped_mlp_bwd's dW1 is grouped_wgrad(X, dH) and its dW2 is
    grouped_wgrad(A, dY), bit for bit (bf16 rounding included)."""
    rng = np.random.default_rng(17)
    off, x, W1, W2 = _tiny(act, rng)
    H, A, _ = O.grouped_mlp_fwd(x, off, W1, W2, act)
    dY = rng.standard_normal((int(off[-1]), W2.shape[2]))
    dH, _, dW1, dW2 = O.grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act)
    assert np.array_equal(O.grouped_wgrad(x, dH, off), dW1)
    assert np.array_equal(O.grouped_wgrad(A, dY, off), dW2)


@pytest.mark.parametrize("act", ACTS)
def test_round_out_changes_only_the_final_rounding(act):
    """round_out=False returns each stored result just before its bf16
    rounding, with every step still fed the rounded values: rounding the
    unrounded outputs gives the default outputs bit for bit, and they lie
    within half a bf16 step (2^-8 relative) of them.  Also for the scaled
    permute, the combine, the plain grouped GEMM, the sampled-row helpers
    and the MXFP8 backward."""
    from oracle import mx as X
    rng = np.random.default_rng(7)
    off, x, W1, W2 = _tiny(act, rng, rows=(64, 0, 32, 96), d=64, n=32)
    x, W1, W2 = O.bf16_round(x), O.bf16_round(W1), O.bf16_round(W2)
    M = int(off[-1])
    dY = O.bf16_round(rng.standard_normal((M, x.shape[1])))
    p = rng.uniform(0.1, 1.0, M)

    def same(u, r):
        u, r = np.asarray(u), np.asarray(r)
        fin = np.isfinite(r)
        assert np.array_equal(np.isfinite(u), fin)
        assert np.array_equal(O.bf16_round(u[fin]), r[fin])
        assert (np.abs(u[fin] - r[fin]) <= 2.0 ** -8 * np.abs(u[fin]) + 1e-300).all()
        return not np.array_equal(u[fin], r[fin])

    changed = []
    fr, fu = O.grouped_mlp_fwd(x, off, W1, W2, act), O.grouped_mlp_fwd(x, off, W1, W2, act,
                                                                       round_out=False)
    changed += [same(u, r) for u, r in zip(fu, fr)]
    H, A, _ = fr
    br = O.grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act)
    bu = O.grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act, round_out=False)
    changed += [same(u, r) for u, r in zip(bu, br)]
    rr = O.grouped_mlp_bwd_routed(x, H, dY, p, off, W1, W2, act)
    ru = O.grouped_mlp_bwd_routed(x, H, dY, p, off, W1, W2, act, round_out=False)
    changed += [same(u, r) for u, r in zip(ru[:5], rr[:5])]
    assert np.array_equal(ru[5], rr[5], equal_nan=True)          # dS is float32-stored: unrounded
    changed.append(same(O.grouped_gemm(A, off, W2, round_out=False), O.grouped_gemm(A, off, W2)))
    changed.append(same(O.grouped_wgrad(x, br[0], off, round_out=False),
                        O.grouped_wgrad(x, br[0], off)))
    h1, a1 = O.fc1_rows(x[:5], W1[0], act, round_out=False)
    h0, a0 = O.fc1_rows(x[:5], W1[0], act)
    changed += [same(h1, h0), same(a1, a0)]
    changed.append(same(O.fc2_rows(a0, W2[0], round_out=False), O.fc2_rows(a0, W2[0])))
    T, k = 40, 2
    pair_of_row = np.concatenate([rng.permutation(T * k), -np.ones(8, np.int64)])
    row_of_pair = np.argsort(pair_of_row[:T * k])
    sc = rng.uniform(0.1, 1.0, T * k)
    xt = O.bf16_round(rng.standard_normal((T, 16)))
    changed.append(same(O.permute(xt, pair_of_row, k, scale=sc, round_out=False),
                        O.permute(xt, pair_of_row, k, scale=sc)))
    yp = O.bf16_round(rng.standard_normal((len(pair_of_row), 16)))
    pr = sc.reshape(T, k)
    changed.append(same(O.unpermute(yp, row_of_pair, T, k, probs=pr, round_out=False),
                        O.unpermute(yp, row_of_pair, T, k, probs=pr)))
    mr = X.mx_grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act)
    mu = X.mx_grouped_mlp_bwd(x, H, A, dY, off, W1, W2, act, round_out=False)
    for key in ("dH", "dX", "dW1", "dW2"):
        changed.append(same(mu[key], mr[key]))
    for key in ("dh_q", "dh_s", "dh_qT", "dh_sT"):            # fed the rounded dH either way
        assert np.array_equal(mu[key], mr[key])
    assert all(changed), changed
