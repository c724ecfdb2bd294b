"""Oracle: routing layout, permute/unpermute, grouped expert MLP fwd/bwd.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  float64 numpy.

Notation follows the pages: T tokens, K (here ``k``) experts per token, E
experts, hidden size d, expert intermediate size n; X gathered tokens,
H = X W1 (FC1 output), A = act(H), Y = A W2; dS is the router-score
gradient ([Sonic] section "역전파 계산 그래프 재작성하기").
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "ERR_BAD_EXPERT", "ERR_OVERFLOW", "ERR_TIMEOUT",
    "bf16_round", "bf16_bits", "bf16_from_bits",
    "router_topk", "route_offsets", "permute", "unpermute", "router_grad",
    "interleave_gate_up", "split_gate_up",
    "act_forward", "act_backward", "phi", "dphi",
    "grouped_mlp_fwd", "grouped_mlp_bwd", "grouped_mlp_bwd_routed",
    "hadamard16", "amax", "amax_rht_transposed",
    "fc1_rows", "fc2_rows", "grouped_gemm", "grouped_wgrad",
]

ERR_BAD_EXPERT = 1
ERR_OVERFLOW = 2
ERR_TIMEOUT = 4


# ---------------------------------------------------------------------------
# bf16 (8 significant bits, 8 exponent bits) rounding, written out
# ---------------------------------------------------------------------------

def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    For |v| in [2^(e-1), 2^e) the bf16 spacing is 2^(e-8); below the smallest
    normal (2^-126) the spacing is fixed at 2^-133.  Division and
    multiplication by powers of two are exact, so ``rint`` (ties to even) does
    the rounding.
    Storage format of every activation and weight ([CuTe] "무엇을 해결하려는가": BF16 activation outputs;
    "공개된 근거에서 확인되는 점": the benchmark shape is BF16)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = v != 0
    _, e = np.frexp(v[nz])
    ulp = np.ldexp(1.0, np.maximum(e, -125) - 8)
    q = np.rint(v[nz] / ulp) * ulp
    big = np.abs(q) > 3.3895313892515355e38  # largest finite bf16
    q[big] = np.copysign(np.inf, q[big])
    out[nz] = q
    out[~nz] = v[~nz]  # keeps -0.0
    return out


def bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of float64 values (rounded first).
    Used for bit-exact comparisons ([CuTe] "무엇을 해결하려는가")."""
    q = bf16_round(v).astype(np.float32)  # exact: q is representable
    return (q.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b) -> np.ndarray:
    """Values of BF16 bit patterns ([CuTe] "무엇을 해결하려는가")."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# router: top-k experts per token ([TE] intro: the learned router activates
# the top-K experts of each token; [TE] "Transformer Engine이 제공하는 세 가지
# 구성 요소": gate, top-K selection, then dispatch).  The pages do not fix the
# weighting; the reading taken is the softmax over the K selected logits.
# ---------------------------------------------------------------------------

def router_topk(logits, k: int):
    """For each token, the k largest logits (ties: lower expert index first,
    in decreasing logit order) and the softmax of those k logits.

    Returns (topk_idx int64 [T, k], probs float64 [T, k]).
    Follows [TE] "Transformer Engine이 제공하는 세 가지 구성 요소" (gate, top-K selection, then dispatch)."""
    logits = np.asarray(logits, dtype=np.float64)
    T, E = logits.shape
    idx = np.zeros((T, k), dtype=np.int64)
    probs = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        taken = np.zeros(E, dtype=bool)
        for j in range(k):
            best = -1
            for e in range(E):
                if taken[e]:
                    continue
                if best < 0 or logits[t, e] > logits[t, best]:
                    best = e
            taken[best] = True
            idx[t, j] = best
        sel = logits[t, idx[t]]
        ex = np.exp(sel - sel.max())
        probs[t] = ex / ex.sum()
    return idx, probs


# ---------------------------------------------------------------------------
# routing layout: counts, ragged prefix offsets, pair <-> row maps
# [TE] "MoE 학습이 밀집 모델보다 어려운 이유: 래그드 텐서" (ragged layout, counts
# 6,4,5,2), "용량 기반 MoE와 드롭리스 MoE" (dropless packs 4,13,6 back to back),
# "최적화 1: grouped GEMM" (per-expert blocks aligned to a token unit) and
# ""드롭리스"의 실제 경계" (expert-major output: one slot per (token, expert)
# pair, each expert region padded to the alignment unit; DROP policy reports
# the pre-truncation total).
# ---------------------------------------------------------------------------

def route_offsets(topk_idx, E: int, align: int = 1, M_cap: int | None = None):
    """Routing layout of the expert-major permuted buffer.

    Parameters: ``topk_idx`` int [T, k] (expert id per (token, slot); -1 = no
    route).  Returns a dict with

    * ``counts``  [E]   number of pairs routed to each expert;
    * ``offsets`` [E+1] exclusive prefix sum of counts rounded up to
      ``align``, clamped to ``M_cap`` (rows of expert e are
      [offsets[e], offsets[e+1]));
    * ``row_of_pair`` [T*k] row of pair (t, j) = offsets[e] + rank of (t, j)
      among the pairs of e in row-major (t, j) order; -1 for skipped or
      dropped pairs;
    * ``pair_of_row`` [M_cap] inverse map, -1 for padding / unused rows;
    * ``true_total`` rows demanded before any truncation;
    * ``err`` ERR_BAD_EXPERT if an id is outside [-1, E), ERR_OVERFLOW if
      ``true_total > M_cap`` (rows at or past M_cap are dropped).
    Follows [TE] "MoE 학습이 밀집 모델보다 어려운 이유: 래그드 텐서" and ""드롭리스"의 실제 경계: 래그드 버퍼 계수와 오버플로 검사".
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape if idx.ndim == 2 else (0, 1)
    if M_cap is None:
        M_cap = T * k + E * (align - 1)
    err = 0
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if e == -1:
                continue
            if e < 0 or e >= E:
                err |= ERR_BAD_EXPERT
                continue
            counts[e] += 1
    demanded = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        demanded[e + 1] = demanded[e] + (counts[e] + align - 1) // align * align
    true_total = int(demanded[E])
    if true_total > M_cap:
        err |= ERR_OVERFLOW
    offsets = np.minimum(demanded, M_cap)

    row_of_pair = np.full(T * k, -1, dtype=np.int64)
    pair_of_row = np.full(M_cap, -1, dtype=np.int64)
    fill = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if e < 0 or e >= E:
                continue
            r = int(demanded[e] + fill[e])
            fill[e] += 1
            if r < M_cap:
                row_of_pair[t * k + j] = r
                pair_of_row[r] = t * k + j
    return dict(counts=counts, offsets=offsets, row_of_pair=row_of_pair,
                pair_of_row=pair_of_row, true_total=true_total, err=err)


def permute(x, pair_of_row, k: int, scale=None, round_bf16: bool = True,
            round_out: bool = True):
    """Expert-major gather ([TE] "최적화 2: NCCL EP": dispatch = permute the
    token rows; [Sonic] "Gather Fusion": gather collects each expert's rows).

    ``x_perm[r] = x[pair_of_row[r] // k]`` (optionally times
    ``scale[pair_of_row[r]]``, the backward use with router probabilities);
    rows with ``pair_of_row[r] == -1`` are zero.  The scaled product is
    rounded to bf16 where it is stored; ``round_out=False`` returns it
    before that rounding (the exact value a stored result is compared
    with)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[1]
    M_cap = len(pair_of_row)
    out = np.zeros((M_cap, d), dtype=np.float64)
    for r in range(M_cap):
        p = int(pair_of_row[r])
        if p < 0:
            continue
        row = x[p // k]
        if scale is not None:
            row = np.float64(np.asarray(scale).reshape(-1)[p]) * row
        out[r] = row
    return bf16_round(out) if (round_bf16 and round_out and scale is not None) else out


def unpermute(y_perm, row_of_pair, T: int, k: int, probs=None, round_bf16=True,
              round_out: bool = True):
    """Combine ([TE] "최적화 2: NCCL EP": results return to token order and the
    per-expert outputs are accumulated per token; [Sonic] "scatter" +
    "expert aggregation").  ``out[t] = sum_j probs[t,j] * y_perm[row(t,j)]``,
    with weight 1 when ``probs`` is None; skipped pairs contribute 0.  The
    sum is rounded to bf16 where it is stored; ``round_out=False`` returns it
    before that rounding."""
    y_perm = np.asarray(y_perm, dtype=np.float64)
    d = y_perm.shape[1] if y_perm.ndim == 2 else 0
    out = np.zeros((T, d), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = int(row_of_pair[t * k + j])
            if r < 0:
                continue
            w = 1.0 if probs is None else float(np.asarray(probs)[t, j])
            out[t] += w * y_perm[r]
    return bf16_round(out) if (round_bf16 and round_out) else out


def router_grad(dO, y_perm, row_of_pair, T: int, k: int):
    """Router-score gradient dS_{t,e} = <dO_t, Y_{e,t}> ([Sonic] "역전파 계산
    그래프 재작성하기", first form), indexed by slot: ``dS[t, j]``."""
    dO = np.asarray(dO, dtype=np.float64)
    y_perm = np.asarray(y_perm, dtype=np.float64)
    dS = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = int(row_of_pair[t * k + j])
            if r >= 0:
                dS[t, j] = float(dO[t] @ y_perm[r])
    return dS


# ---------------------------------------------------------------------------
# gate/up interleaving ([CuTe] "핵심 아이디어 / 구조 / 동작 방식": weights are
# repacked so gate and input columns are interleaved and one thread block's
# epilogue sees both halves).  Granularity (one column each) is this
# implementation's reading.
# ---------------------------------------------------------------------------

def interleave_gate_up(w_gate, w_up):
    """[..., d, n] gate and up -> [..., d, 2n] with column 2j = gate_j,
    column 2j+1 = up_j.
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (gate and up columns interleaved)."""
    w_gate = np.asarray(w_gate)
    w_up = np.asarray(w_up)
    out = np.empty(w_gate.shape[:-1] + (2 * w_gate.shape[-1],), dtype=w_gate.dtype)
    out[..., 0::2] = w_gate
    out[..., 1::2] = w_up
    return out


def split_gate_up(w1):
    """Inverse of interleave_gate_up ([CuTe] "핵심 아이디어 / 구조 / 동작 방식")."""
    w1 = np.asarray(w1)
    return w1[..., 0::2], w1[..., 1::2]


# ---------------------------------------------------------------------------
# activations ([CuTe] "무엇을 해결하려는가" names SwiGLU, GeGLU and sReLU;
# "핵심 아이디어": SwiGLU applies Swish to the gate side and multiplies by the
# input side)
# ---------------------------------------------------------------------------

_C = math.sqrt(2.0 / math.pi)
_A = 0.044715


def phi(g, act: str):
    """Gate nonlinearity: SiLU (Swish-1) for SwiGLU, tanh-approximated GELU
    (Hendrycks & Gimpel) for GeGLU.
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (Swish on the gate side)."""
    g = np.asarray(g, dtype=np.float64)
    if act == "swiglu":
        return g / (1.0 + np.exp(-g))
    if act == "geglu":
        return 0.5 * g * (1.0 + np.tanh(_C * (g + _A * g ** 3)))
    raise ValueError(act)


def dphi(g, act: str):
    """Analytic derivative of ``phi``, needed by the dActivation epilogue
    ([CuTe] "무엇을 해결하려는가": the backward GroupGemm + dActivation)."""
    g = np.asarray(g, dtype=np.float64)
    if act == "swiglu":
        s = 1.0 / (1.0 + np.exp(-g))
        return s * (1.0 + g * (1.0 - s))
    if act == "geglu":
        z = _C * (g + _A * g ** 3)
        th = np.tanh(z)
        return 0.5 * (1.0 + th) + 0.5 * g * (1.0 - th * th) * _C * (1.0 + 3.0 * _A * g * g)
    raise ValueError(act)


def act_forward(h, act: str):
    """A = act(H).  Gated: H columns (2j, 2j+1) = (gate, up), A_j = phi(g) u.
    Squared ReLU: A = max(H, 0)^2.
    Follows [CuTe] "무엇을 해결하려는가" (SwiGLU, GeGLU, sReLU) and "핵심 아이디어 / 구조 / 동작 방식"."""
    h = np.asarray(h, dtype=np.float64)
    if act == "srelu":
        return np.maximum(h, 0.0) ** 2
    g, u = h[..., 0::2], h[..., 1::2]
    return phi(g, act) * u


def act_backward(h, dA, act: str):
    """dH from dA and H (chain rule of ``act_forward``).  Gated:
    dg = dA u phi'(g), du = dA phi(g), written back interleaved.
    Follows [CuTe] "무엇을 해결하려는가" (GroupGemm + dActivation) and [Sonic] "역전파 계산 그래프 재작성하기" (the dH
    kernel reloads H)."""
    h = np.asarray(h, dtype=np.float64)
    dA = np.asarray(dA, dtype=np.float64)
    if act == "srelu":
        return 2.0 * np.maximum(h, 0.0) * dA
    g, u = h[..., 0::2], h[..., 1::2]
    dh = np.empty_like(h)
    dh[..., 0::2] = dA * u * dphi(g, act)
    dh[..., 1::2] = dA * phi(g, act)
    return dh


# ---------------------------------------------------------------------------
# grouped expert MLP ([TE] "최적화 1: grouped GEMM": one grouped call over the
# experts' real token counts; [Sonic] "SonicMoE로 이해하는 ...": up-projection,
# SwiGLU, down-projection)
# ---------------------------------------------------------------------------

def _rb(v, on):
    """Rounding to BF16 where a BF16 implementation stores a tensor ([CuTe] "무엇을 해결하려는가")."""
    return bf16_round(v) if on else np.asarray(v, dtype=np.float64)


def grouped_mlp_fwd(x_perm, offsets, W1, W2, act: str, round_bf16: bool = True,
                    round_out: bool = True):
    """Per expert e with rows R_e = [offsets[e], offsets[e+1]):
    H_e = X_e W1_e, A_e = act(H_e), Y_e = A_e W2_e.

    Rounding points mirror what a bf16 implementation stores: H (saved for
    backward) and A are rounded to bf16, A is computed from the unrounded H,
    FC2 reads the rounded A, Y is rounded.  Rows outside every expert are
    NaN (undefined).  With ``round_out=False`` the returned H, A and Y are
    the values just before their storage rounding, while every step still
    consumes the rounded values (a stored bf16 result is then compared with
    the exact value it rounds).
    Follows [TE] "최적화 1: grouped GEMM, 전문가마다 다른 토큰 수를 커널 하나로" and [CuTe] "핵심 아이디어 / 구조 / 동작 방식"."""
    x_perm = np.asarray(x_perm, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    M_cap = x_perm.shape[0]
    E = len(offsets) - 1
    n1, n, d = W1.shape[2], W2.shape[1], W2.shape[2]
    H = np.full((M_cap, n1), np.nan)
    A = np.full((M_cap, n), np.nan)
    Y = np.full((M_cap, d), np.nan)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        h = x_perm[r0:r1] @ W1[e]
        a_exact = act_forward(h, act)
        a = _rb(a_exact, round_bf16)
        H[r0:r1] = _rb(h, round_bf16 and round_out)
        A[r0:r1] = a if round_out else a_exact
        Y[r0:r1] = _rb(a @ W2[e], round_bf16 and round_out)
    return H, A, Y


def grouped_gemm(a, offsets, B, b_layout: str = "kn", round_bf16: bool = True,
                 round_out: bool = True):
    """Plain grouped GEMM ([TE] "최적화 1: grouped GEMM": one call over the
    experts' ragged row groups): out_e = A_e B_e for the rows of expert e,
    with B [E, K, N] ("kn") or B stored transposed as [E, N, K] ("nk", then
    out_e = A_e B_e^T).  Rows outside every expert are NaN (undefined); the
    result is rounded to bf16 once (not with ``round_out=False``)."""
    a = np.asarray(a, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if b_layout == "nk":
        B = np.swapaxes(B, 1, 2)
    elif b_layout != "kn":
        raise ValueError(b_layout)
    E, N = B.shape[0], B.shape[2]
    out = np.full((a.shape[0], N), np.nan)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            out[r0:r1] = _rb(a[r0:r1] @ B[e], round_bf16 and round_out)
    return out


def grouped_wgrad(P, Q, offsets, round_out: bool = True):
    """Weight gradient of a grouped GEMM ([TE] "최적화 1: grouped GEMM": the
    experts' ragged row groups): dW_e = P_e^T Q_e, the sum over the rows
    of expert e, P [M, p], Q [M, q] -> [E, p, q]; an expert with no rows
    gets 0.  The same product as grouped_mlp_bwd's dW1 (P = X, Q = dH) and
    dW2 (P = A, Q = dY), for checking one weight-gradient GEMM on given
    operands.  Rounded to bf16 once (not with ``round_out=False``)."""
    P = np.asarray(P, dtype=np.float64)
    Q = np.asarray(Q, dtype=np.float64)
    E = len(offsets) - 1
    dW = np.zeros((E, P.shape[1], Q.shape[1]))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            dW[e] = P[r0:r1].T @ Q[r0:r1]
    return bf16_round(dW) if round_out else dW


def grouped_mlp_bwd(x_perm, H, A, dY, offsets, W1, W2, act: str,
                    round_bf16: bool = True, round_out: bool = True):
    """Backward of ``grouped_mlp_fwd`` per expert:
    dA_e = dY_e W2_e^T, dH_e = act'(H_e; dA_e), dW2_e = A_e^T dY_e,
    dX_e = dH_e W1_e^T, dW1_e = X_e^T dH_e.  An expert with no rows gets
    dW1_e = dW2_e = 0.  dH is rounded to bf16 before it feeds dX and dW1
    (a bf16 implementation stores it).  With ``round_out=False`` the returned
    dH, dX, dW1, dW2 are the values just before their storage rounding;
    dX and dW1 are still computed from the rounded dH.
    Follows [CuTe] "무엇을 해결하려는가" (GroupGemm + dActivation) and [TE] "최적화 1: grouped GEMM, 전문가마다 다른
    토큰 수를 커널 하나로"."""
    x_perm = np.asarray(x_perm, dtype=np.float64)
    H = np.asarray(H, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    M_cap = x_perm.shape[0]
    E = len(offsets) - 1
    n1 = W1.shape[2]
    dH = np.full((M_cap, n1), np.nan)
    dX = np.full(x_perm.shape, np.nan)
    dW1 = np.zeros(W1.shape)
    dW2 = np.zeros(W2.shape)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        dA = dY[r0:r1] @ W2[e].T
        dh_exact = act_backward(H[r0:r1], dA, act)
        dh = _rb(dh_exact, round_bf16)
        dH[r0:r1] = dh if round_out else dh_exact
        dW2[e] = A[r0:r1].T @ dY[r0:r1]
        dX[r0:r1] = _rb(dh @ W1[e].T, round_bf16 and round_out)
        dW1[e] = x_perm[r0:r1].T @ dh
    ro = round_bf16 and round_out
    return dH, dX, _rb(dW1, ro), _rb(dW2, ro)


def grouped_mlp_bwd_routed(x_perm, H, dO_perm, row_prob, offsets, W1, W2, act: str,
                           round_bf16: bool = True, round_out: bool = True):
    """Backward with the router gradient taken inside the expert MLP
    ([Sonic] "역전파 계산 그래프 재작성하기": dS_{t,e} = <dO_t, Y_{e,t}> =
    <dO_t W2_e^T, A_e>, so Y need not be kept; A is recomputed from H, and
    the dH kernel's epilogue also emits dS and A' = S*A).

    Inputs: dO_perm is the gathered, unscaled output gradient of each row;
    row_prob the router probability of the row's (token, expert) pair (0
    for pad rows).  Per expert e (rows R_e):
      dA'  = dO_e W2_e^T                      (gradient w.r.t. the row's A,
                                               before the probability)
      dS   = <dA'_r, A_r> per row, A = act(H) from the stored H
      dH   = act'(H; p_r dA'_r)
      A'   = p_r A_r                          (rounded to bf16)
      dW2_e = A'_e^T dO_e,  dX_e = dH_e W1_e^T,  dW1_e = X_e^T dH_e.
    Returns dH, dX, dW1, dW2, A', dS (float64 [M], NaN outside every
    expert).  With ``round_out=False`` the returned dH, dX, dW1, dW2 and A'
    are the values just before their storage rounding; later steps still
    consume the rounded dH and A'."""
    x_perm = np.asarray(x_perm, dtype=np.float64)
    H = np.asarray(H, dtype=np.float64)
    dO = np.asarray(dO_perm, dtype=np.float64)
    p = np.asarray(row_prob, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    M_cap = x_perm.shape[0]
    E = len(offsets) - 1
    n1, n = W1.shape[2], W2.shape[1]
    dH = np.full((M_cap, n1), np.nan)
    dX = np.full(x_perm.shape, np.nan)
    Ap = np.full((M_cap, n), np.nan)
    dS = np.full(M_cap, np.nan)
    dW1 = np.zeros(W1.shape)
    dW2 = np.zeros(W2.shape)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        pr = p[r0:r1, None]
        dAp = dO[r0:r1] @ W2[e].T
        A = act_forward(H[r0:r1], act)
        dS[r0:r1] = (dAp * A).sum(axis=1)
        dh_exact = act_backward(H[r0:r1], pr * dAp, act)
        dh = _rb(dh_exact, round_bf16)
        dH[r0:r1] = dh if round_out else dh_exact
        ap = _rb(pr * A, round_bf16)
        Ap[r0:r1] = ap if round_out else pr * A
        dW2[e] = ap.T @ dO[r0:r1]
        dX[r0:r1] = _rb(dh @ W1[e].T, round_bf16 and round_out)
        dW1[e] = x_perm[r0:r1].T @ dh
    ro = round_bf16 and round_out
    return dH, dX, _rb(dW1, ro), _rb(dW2, ro), Ap, dS


# ---------------------------------------------------------------------------
# NVFP4 scaling statistics ([CuTe] "핵심 아이디어": the per-tensor amax of the
# forward output and the amax of the transposed, Hadamard-rotated output in
# the backward are separate memory passes unless fused)
# ---------------------------------------------------------------------------

def hadamard16() -> np.ndarray:
    """16x16 Hadamard matrix of Sylvester's construction, H[i, j] =
    (-1)^popcount(i & j), scaled by 1/4 so that it is orthonormal.  The
    rotation of the backward's NVFP4 statistic ([CuTe] "핵심 아이디어 / 구조 /
    동작 방식": amax of the transposed, Hadamard-rotated output)."""
    i = np.arange(16)
    parity = np.array([[bin(a & b).count("1") & 1 for b in i] for a in i])
    return np.where(parity == 1, -1.0, 1.0) / 4.0


def amax(t) -> float:
    """Per-tensor absolute maximum.
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (the forward output's per-tensor amax)."""
    t = np.asarray(t, dtype=np.float64)
    return float(np.abs(t).max()) if t.size else 0.0


def amax_rht_transposed(G, offsets) -> float:
    """Absolute maximum of the transposed copy of G [M, C] after the
    16-point Hadamard rotation along its rows: per expert, the rows
    [offsets[e], offsets[e+1]) are cut into 16-row blocks from the expert's
    first row (the last block zero-padded), and each column of a block is
    multiplied by hadamard16().  (Reading: the pages name the statistic;
    the rotation is the orthonormal Sylvester one, without random signs.)
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식"."""
    G = np.asarray(G, dtype=np.float64)
    Hm = hadamard16()
    best = 0.0
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        rows = r1 - r0
        nb = -(-rows // 16)
        blk = np.zeros((nb * 16, G.shape[1]))
        blk[:rows] = G[r0:r1]
        rot = np.einsum("ij,bjc->bic", Hm, blk.reshape(nb, 16, G.shape[1]))
        best = max(best, float(np.abs(rot).max()))
    return best


# sampled-row helpers for full-size parity checks (same arithmetic as above,
# restricted to selected rows of one expert and selected output columns)

def fc1_rows(x_rows, W1_e, act: str, cols=None, round_out: bool = True):
    """(H, A) of the given rows of one expert; ``cols`` selects A columns
    (and the matching H column pairs when gated).
    The arithmetic of grouped_mlp_fwd on selected rows ([CuTe] "핵심 아이디어 / 구조 / 동작 방식")."""
    x_rows = np.asarray(x_rows, dtype=np.float64)
    W1_e = np.asarray(W1_e, dtype=np.float64)
    h = x_rows @ W1_e
    a = act_forward(h, act)
    if cols is not None:
        a = a[:, cols]
    return (bf16_round(h), bf16_round(a)) if round_out else (h, a)


def fc2_rows(a_rows, W2_e, round_out: bool = True):
    """The arithmetic of grouped_mlp_fwd's down-projection on selected rows ([TE] "최적화 1: grouped
    GEMM, 전문가마다 다른 토큰 수를 커널 하나로")."""
    y = np.asarray(a_rows, np.float64) @ np.asarray(W2_e, np.float64)
    return bf16_round(y) if round_out else y
