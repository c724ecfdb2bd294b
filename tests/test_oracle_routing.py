"""Pins for the oracle's routing layout and permute / unpermute.

Pinned by the pages' worked examples (tests/golden/routing_examples.json),
by an independent sort-based construction enumerated exhaustively on tiny
inputs, and by the permute/unpermute identities."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "routing_examples.json")))


def _idx_from_counts(counts, seed=0):
    """A k=1 routing with the given per-expert counts, tokens shuffled."""
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int64)
    rng = np.random.default_rng(seed)
    rng.shuffle(ids)
    return ids.reshape(-1, 1)


@pytest.mark.parametrize("name", ["ragged_6_4_5_2", "capacity_10_vs_dropless_4_13_6"])
def test_golden_offsets(name):
    g = GOLD[name]
    r = O.route_offsets(_idx_from_counts(g["counts"]), g["E"])
    assert r["counts"].tolist() == g["counts"]
    assert r["offsets"].tolist() == g["offsets"]
    assert r["err"] == 0
    assert r["true_total"] == g["offsets"][-1]


def test_golden_capacity_contrast():
    """The page's capacity numbers (waste, drop) against our dropless layout:
    dropless wastes nothing and drops nothing."""
    g = GOLD["capacity_10_vs_dropless_4_13_6"]
    cap = g["capacity"]
    counts = np.array(g["counts"])
    assert (np.maximum(cap - counts, 0)).tolist() == g["capacity_wasted"]
    assert (np.maximum(counts - cap, 0)).tolist() == g["capacity_dropped"]
    r = O.route_offsets(_idx_from_counts(counts), g["E"])
    assert (r["pair_of_row"] >= 0).all()          # no padding rows
    assert (r["row_of_pair"] >= 0).all()          # nothing dropped


def test_golden_top2_empty_group():
    g = GOLD["top2_empty_group"]
    # tokens 0..3 pick two distinct experts among {0,1,2}; expert 2 gets 3
    idx = np.array([[0, 2], [1, 2], [2, 0], [1, 0]], dtype=np.int64)
    r = O.route_offsets(idx, g["E"])
    for e, c in g["counts_known"].items():
        assert r["counts"][int(e)] == c
    assert r["offsets"][3] == r["offsets"][4]          # empty range for E3
    assert r["offsets"][4] == idx.size


def _sort_based(idx, E, align, M_cap):
    """Independent construction: sort valid pairs by (expert, t, j)."""
    T, k = idx.shape
    pairs = [(int(idx[t, j]), t, j) for t in range(T) for j in range(k)
             if 0 <= idx[t, j] < E]
    pairs.sort()
    row_of_pair = -np.ones(T * k, np.int64)
    pair_of_row = -np.ones(M_cap, np.int64)
    start = 0
    offs = [0]
    for e in range(E):
        mine = [p for p in pairs if p[0] == e]
        for rank, (_, t, j) in enumerate(mine):
            r = start + rank
            if r < M_cap:
                row_of_pair[t * k + j] = r
                pair_of_row[r] = t * k + j
        start += -(-len(mine) // align) * align
        offs.append(min(start, M_cap))
    return np.array(offs), row_of_pair, pair_of_row, start


@pytest.mark.parametrize("align", [1, 2, 4])
def test_exhaustive_tiny(align):
    """All 3^(2*3) expert assignments of T=3 tokens, k=2, E=3 (ids may
    repeat), compared with the sort-based construction."""
    E, T, k = 3, 3, 2
    for combo in itertools.product(range(E), repeat=T * k):
        idx = np.array(combo, dtype=np.int64).reshape(T, k)
        r = O.route_offsets(idx, E, align)
        offs, rop, por, total = _sort_based(idx, E, align, r["pair_of_row"].size)
        assert r["offsets"].tolist() == offs.tolist()
        assert r["row_of_pair"].tolist() == rop.tolist()
        assert r["pair_of_row"].tolist() == por.tolist()
        assert r["true_total"] == total
        assert r["counts"].sum() == T * k


def test_invariants_random():
    rng = np.random.default_rng(3)
    for trial in range(20):
        E = int(rng.integers(1, 9))
        T = int(rng.integers(0, 40))
        k = int(rng.integers(1, min(E, 4) + 1))
        align = int(rng.choice([1, 8, 32]))
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int64)
        r = O.route_offsets(idx, E, align)
        rop, por, off = r["row_of_pair"], r["pair_of_row"], r["offsets"]
        assert r["counts"].sum() == T * k
        assert len(por) == T * k + E * (align - 1)
        assert (off % align == 0).all()
        for p, row in enumerate(rop):                 # pair_of_row o row_of_pair = id
            assert por[row] == p
        for e in range(E):                            # rows of e lie in its range
            rows = sorted(rop[p] for p in range(T * k) if idx[p // k, p % k] == e)
            assert rows == list(range(off[e], off[e] + r["counts"][e]))
        assert (por[off[-1]:] == -1).all()


def test_no_route_and_bad_expert():
    idx = np.array([[0, -1], [5, 1], [1, -3]], dtype=np.int64)
    r = O.route_offsets(idx, 2)
    assert r["err"] == O.ERR_BAD_EXPERT
    assert r["counts"].tolist() == [1, 2]
    assert r["row_of_pair"].tolist() == [0, -1, -1, 1, 2, -1]


def test_overflow_drop_reports_true_total():
    """DROP-style overflow ([TE] section on the real boundary of dropless:
    excess tokens are dropped and the pre-truncation total is reported)."""
    idx = _idx_from_counts([4, 13, 6])
    r = O.route_offsets(idx, 3, align=1, M_cap=20)
    assert r["err"] == O.ERR_OVERFLOW
    assert r["true_total"] == 23
    assert r["offsets"].tolist() == [0, 4, 17, 20]
    assert (r["row_of_pair"] >= 0).sum() == 20
    assert (r["pair_of_row"] >= 0).all()


def test_empty_tokens():
    r = O.route_offsets(np.zeros((0, 2), np.int64), 4, align=8)
    assert r["counts"].tolist() == [0] * 4
    assert r["offsets"].tolist() == [0] * 5
    assert r["true_total"] == 0


def _bf(rng, shape, std=1.0):
    return O.bf16_round(rng.standard_normal(shape) * std)


def test_permute_unpermute_identity():
    rng = np.random.default_rng(1)
    T, k, E, d = 37, 2, 5, 16
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    r = O.route_offsets(idx, E, align=8)
    x = _bf(rng, (T, d))
    xp = O.permute(x, r["pair_of_row"], k)
    # pad rows are zero, real rows are exact copies
    assert (xp[r["pair_of_row"] < 0] == 0).all()
    # unweighted combine of the permuted copies = k * x exactly (k = 2)
    assert (O.unpermute(xp, r["row_of_pair"], T, k) == 2 * x).all()
    # weighted combine with probabilities summing to 1 gives back x
    p = rng.random((T, k))
    p /= p.sum(1, keepdims=True)
    back = O.unpermute(xp, r["row_of_pair"], T, k, probs=p, round_bf16=False)
    assert np.abs(back - x).max() < 1e-12


def test_combine_weights_each_slot_by_its_own_probability():
    """A worked case by hand: token 0 goes to experts (1, 0) with weights
    (0.75, 0.25), token 1 to (0, 1) with (0.5, 0.5) reversed as (1, 0) with
    (0.125, 0.875).  Expert rows hold distinct powers of two, so each output
    names the rows and weights it used exactly."""
    idx = np.array([[1, 0], [1, 0]])
    r = O.route_offsets(idx, 2)
    # rows: expert 0 = pairs (0,1), (1,1); expert 1 = pairs (0,0), (1,0)
    assert r["row_of_pair"].tolist() == [2, 0, 3, 1]
    y = np.array([[1.0, 0.0], [2.0, 0.0], [0.0, 4.0], [0.0, 8.0]])   # rows 0..3
    p = np.array([[0.75, 0.25], [0.125, 0.875]])
    out = O.unpermute(y, r["row_of_pair"], 2, 2, probs=p, round_bf16=False)
    # token 0: 0.75 * row 2 + 0.25 * row 0;  token 1: 0.125 * row 3 + 0.875 * row 1
    assert out.tolist() == [[0.25, 3.0], [1.75, 1.0]]


def test_permute_scale_is_prob_times_row():
    rng = np.random.default_rng(2)
    T, k, E, d = 9, 2, 3, 8
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    r = O.route_offsets(idx, E)
    dO = _bf(rng, (T, d))
    p = rng.random((T, k)).astype(np.float32)
    dyp = O.permute(dO, r["pair_of_row"], k, scale=p)
    for t in range(T):
        for j in range(k):
            row = r["row_of_pair"][t * k + j]
            assert (dyp[row] == O.bf16_round(np.float64(p[t, j]) * dO[t])).all()


def test_router_grad_matches_directional_derivative_and_rewrite():
    """dS from Y equals the derivative of <dO, combine(Y, probs)> w.r.t.
    probs, and equals the rewritten form <dO W2^T, A> ([Sonic] section on
    rewriting the backward graph)."""
    rng = np.random.default_rng(4)
    T, k, E, d, n = 6, 2, 3, 8, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    r = O.route_offsets(idx, E)
    A = rng.standard_normal((T * k, n))
    W2 = rng.standard_normal((E, n, d))
    Y = np.zeros((T * k, d))
    for e in range(E):
        a, b = r["offsets"][e], r["offsets"][e + 1]
        Y[a:b] = A[a:b] @ W2[e]
    dO = rng.standard_normal((T, d))
    dS = O.router_grad(dO, Y, r["row_of_pair"], T, k)
    p0 = rng.random((T, k))
    L = lambda p: float((dO * O.unpermute(Y, r["row_of_pair"], T, k, p, round_bf16=False)).sum())
    eps = 1e-6
    for t in range(T):
        for j in range(k):
            pp, pm = p0.copy(), p0.copy()
            pp[t, j] += eps
            pm[t, j] -= eps
            assert abs((L(pp) - L(pm)) / (2 * eps) - dS[t, j]) < 1e-6
    # rewritten form
    for t in range(T):
        for j in range(k):
            row = r["row_of_pair"][t * k + j]
            e = idx[t, j]
            assert abs(float((dO[t] @ W2[e].T) @ A[row]) - dS[t, j]) < 1e-10


def test_bf16_round_against_float32_truncation_rule():
    """bf16_round agrees with the bit rule 'round the float32 pattern to its
    top 16 bits, ties to even' on values exactly representable in float32."""
    rng = np.random.default_rng(5)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-40, 40, 20000))).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    rounded = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    assert (O.bf16_bits(f.astype(np.float64)) == rounded).all()
    # exact ties
    one = np.float64(1.0)
    assert O.bf16_round(one + 2.0 ** -8) == 1.0                 # tie -> even (1.0)
    assert O.bf16_round(one + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6   # tie -> even


def test_router_topk_pins():
    """Top-k against a full stable sort; ties go to the lower index; the
    probabilities are a softmax (sum to 1, ratios exp(l_i - l_j)); a
    -inf logit is never chosen while finite ones remain."""
    rng = np.random.default_rng(30)
    lg = rng.standard_normal((50, 16))
    lg[3, :] = 0.5                                  # all tied
    lg[7, [2, 9]] = 10.0                            # a tie at the top
    lg[11, 5] = -np.inf
    idx, p = O.router_topk(lg, 4)
    ref = np.argsort(-lg, axis=1, kind="stable")[:, :4]
    assert (idx == ref).all()
    assert idx[3].tolist() == [0, 1, 2, 3]
    assert idx[7, :2].tolist() == [2, 9]
    assert 5 not in idx[11]
    assert np.allclose(p.sum(1), 1.0, atol=1e-15)
    t = 20
    l = lg[t, idx[t]]
    assert np.allclose(p[t, 0] / p[t, 1], np.exp(l[0] - l[1]), rtol=1e-12)
    i1, p1 = O.router_topk(lg[:5], 1)
    assert (p1 == 1.0).all() and (i1[:, 0] == lg[:5].argmax(1)).all()
