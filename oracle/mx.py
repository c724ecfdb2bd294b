"""Oracle: MXFP8 (E4M3 elements, E8M0 block scales, 32-element blocks).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages ask for an MXFP8 output and its transposed copy written from the
FC1 epilogue ([CuTe] "무엇을 해결하려는가" and "핵심 아이디어": MXFP8 needs the
quantised output and a transposed output), for quantisation that respects
expert-group boundaries and for an MXFP8 grouped GEMM ([TE] "Transformer
Engine이 제공하는 세 가지 구성 요소").  The block rule is the OCP Microscaling
(MX) v1.0 one: per block of 32 values, shared scale X = 2^(floor(log2 amax) -
emax_elem) with emax_elem = 8 for E4M3, element codes E4M3(v / X) with round
to nearest, ties to even, saturating to the largest finite magnitude 448.

E4M3 here is the OCP "fn" variant: 1 sign, 4 exponent (bias 7), 3 mantissa
bits, no infinities, NaN = S.1111.111; subnormals 2^-6 * m/8.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "E4M3_MAX", "e4m3_decode_table", "e4m3_decode", "e4m3_encode", "e4m3_encode_bruteforce",
    "e8m0_exponent", "mx_quantize_blocks", "mx_quantize_rows",
    "mx_quantize_cols", "mx_quantize_weights", "mx_dequantize", "mx_fc2",
    "mx_dgrad", "mx_wgrad", "mx_grouped_mlp_bwd",
]

E4M3_MAX = 448.0


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 codes (NaN for the two NaN codes).
    E4M3 element format of MXFP8 ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소"; OCP MX v1.0)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        ex = (c >> 3) & 0xF
        m = c & 0x7
        if ex == 0xF and m == 0x7:
            vals[c] = np.nan
        elif ex == 0:
            vals[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (ex - 7)
    return vals


_DEC = e4m3_decode_table()
# positive finite codes 0x00..0x7E in increasing value order
_POS_CODES = np.arange(0x7F)
_POS_VALS = _DEC[:0x7F]


def e4m3_decode(codes) -> np.ndarray:
    """Decodes E4M3 codes ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소"; OCP MX v1.0)."""
    return _DEC[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_bruteforce(v) -> np.ndarray:
    """Brute-force nearest finite E4M3 code, ties to the even code (even
    mantissa), magnitudes above 448 saturate to 448; the sign bit is kept
    (so -0 and negative values that round to zero give 0x80).  This is the
    definition; ``e4m3_encode`` computes the same function faster.
    MXFP8 element rounding ([CuTe] "핵심 아이디어 / 구조 / 동작 방식": the MXFP8 output; OCP MX v1.0)."""
    v = np.asarray(v, dtype=np.float64)
    # saturate first: beyond 448 every magnitude maps to 448 (measuring
    # distances from huge values would also lose the codes' spacing)
    a = np.minimum(np.abs(v).reshape(-1), E4M3_MAX)
    dist = np.abs(a[:, None] - _POS_VALS[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among equally near codes prefer the even one (ties-to-even); two
    # adjacent codes always differ in their lowest bit
    even = cand & ((_POS_CODES[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    code = _POS_CODES[pick].astype(np.uint8)
    code = code | np.where(np.signbit(v.reshape(-1)), 0x80, 0).astype(np.uint8)
    return code.reshape(v.shape)


def e4m3_encode(v) -> np.ndarray:
    """Same function as ``e4m3_encode_bruteforce`` (nearest finite code,
    ties to even, saturating, sign kept), found by bisection in the sorted
    table of the 127 non-negative finite values instead of a full scan.
    MXFP8 element rounding ([CuTe] "핵심 아이디어 / 구조 / 동작 방식"; OCP MX v1.0)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v).reshape(-1), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALS, a, side="left"), 0, 0x7E)   # first value >= a
    lo = np.clip(hi - 1, 0, 0x7E)
    dlo = a - _POS_VALS[lo]
    dhi = _POS_VALS[hi] - a
    pick = np.where(dhi < dlo, hi, lo)
    tie = (dhi == dlo) & (hi != lo)
    pick = np.where(tie, np.where((hi & 1) == 0, hi, lo), pick)
    code = pick.astype(np.uint8) | np.where(np.signbit(v.reshape(-1)), 0x80, 0).astype(np.uint8)
    return code.reshape(v.shape)


def e8m0_exponent(amax) -> np.ndarray:
    """Shared-scale exponent e = clamp(floor(log2 amax) - 8, -127, 127);
    amax = 0 gives -127.  floor(log2) is read exactly from frexp.
    The E8M0 shared scale of an MXFP8 block ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소"; OCP MX
    v1.0)."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)          # amax = m 2^ex, m in [0.5, 1)
    e = (ex - 1) - 8
    e = np.where(amax == 0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def mx_quantize_blocks(blocks):
    """``blocks`` [..., 32] float64 -> (codes uint8 [..., 32], scale codes
    uint8 [...]) where the scale code is e + 127.
    One MXFP8 block ([CuTe] "핵심 아이디어 / 구조 / 동작 방식": the MXFP8 output; OCP MX v1.0)."""
    blocks = np.asarray(blocks, dtype=np.float64)
    amax = np.abs(blocks).max(axis=-1)
    e = e8m0_exponent(amax)
    scaled = blocks * np.ldexp(1.0, -e)[..., None]   # exact (power of two)
    return e4m3_encode(scaled), (e + 127).astype(np.uint8)


def mx_quantize_rows(A):
    """Row-wise MX: blocks of 32 consecutive columns of each row.
    A [M, n] (n % 32 == 0) -> codes [M, n], scales [M, n/32].
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (the MXFP8 output)."""
    A = np.asarray(A, dtype=np.float64)
    M, n = A.shape
    q, s = mx_quantize_blocks(A.reshape(M, n // 32, 32))
    return q.reshape(M, n), s


def mx_quantize_cols(A, offsets, M_cap=None):
    """Column-wise MX for the transposed copy: blocks of 32 consecutive rows
    of each column.  Blocks are taken inside each expert's row range
    [offsets[e], offsets[e+1]) (group-aware; with 32-row alignment every
    range starts on a block boundary and no block crosses two experts).

    Returns (codes_T uint8 [n, M_cap], scales_T uint8 [n, M_cap/32]); rows
    outside every expert are left 0.
    Follows [CuTe] "핵심 아이디어 / 구조 / 동작 방식" (the transposed output) and [TE] "Transformer Engine이
    제공하는 세 가지 구성 요소" (group-aware quantisation)."""
    A = np.asarray(A, dtype=np.float64)
    M = A.shape[0] if M_cap is None else M_cap
    n = A.shape[1]
    qT = np.zeros((n, M), dtype=np.uint8)
    sT = np.zeros((n, M // 32), dtype=np.uint8)
    E = len(offsets) - 1
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        assert r0 % 32 == 0 and r1 % 32 == 0, "column blocks need 32-row alignment"
        for b0 in range(r0, r1, 32):
            blk = A[b0:b0 + 32, :].T             # [n, 32]
            q, s = mx_quantize_blocks(blk)
            qT[:, b0:b0 + 32] = q
            sT[:, b0 // 32] = s
    return qT, sT


def mx_quantize_weights(W2):
    """W2 [E, n, d]: blocks of 32 consecutive rows (FC2's reduction index)
    for each column.  Returns codes [E, n, d] and scales [E, n/32, d].
    Follows [TE] "Transformer Engine이 제공하는 세 가지 구성 요소" (MXFP8 expert weights for the MXFP8 grouped
    GEMM)."""
    W2 = np.asarray(W2, dtype=np.float64)
    E, n, d = W2.shape
    blk = W2.reshape(E, n // 32, 32, d).transpose(0, 1, 3, 2)   # [E, n/32, d, 32]
    q, s = mx_quantize_blocks(blk)
    return q.transpose(0, 1, 3, 2).reshape(E, n, d), s


def mx_dequantize(codes, scale_codes, axis_block: int):
    """Decode codes with their block scales; ``axis_block`` is the axis of
    ``codes`` along which 32 consecutive elements share a scale.
    Inverse of the MX block rule ([TE] "Transformer Engine이 제공하는 세 가지 구성 요소"; OCP MX v1.0)."""
    v = e4m3_decode(codes)
    s = np.ldexp(1.0, scale_codes.astype(np.int64) - 127)
    s = np.repeat(s, 32, axis=axis_block)
    return v * s


def mx_fc2(A_q, A_s, W2_q, W2_s, offsets):
    """MXFP8 down-projection Y_e = sum over 32-blocks b of
    (s_A s_W) * sum_{i in b} qA qW, float64; Y rounded to bf16 by the caller.
    Products of dequantised values are exact in float64.
    Follows [TE] "Transformer Engine이 제공하는 세 가지 구성 요소" (the MXFP8 grouped GEMM)."""
    from .moe import bf16_round
    A = mx_dequantize(A_q, A_s, axis_block=1)
    M = A.shape[0]
    E, n, d = W2_q.shape
    Y = np.full((M, d), np.nan)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        W = mx_dequantize(W2_q[e], W2_s[e], axis_block=0)
        Y[r0:r1] = A[r0:r1] @ W
    return bf16_round(Y)


# ---------------------------------------------------------------- backward
# MXFP8 backward of the expert MLP.  The pages name the fused backward kernel
# ([TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩": GroupGemm +
# dActivation + Quantize/Transpose) and the reason a transposed copy is
# written at all ([CuTe] "무엇을 해결하려는가": low-precision output plus a
# transposed output): a weight gradient contracts over the rows of an expert,
# so its operands need blocks that run along the rows.  Reading: every
# backward GEMM takes MXFP8 operands with 32-element blocks along its own
# reduction index -
#   data gradients (reduction over a hidden index): row-wise blocks of the
#     activation gradient and blocks along the same index of the weight;
#   weight gradients (reduction over the rows of one expert): the
#     column-wise, group-aware blocks of the transposed copies.
# Accumulation is exact here (float64 of exactly decoded values); dH is
# rounded to bf16 before it is quantised, as a bf16 store would leave it.

def mx_dgrad(G_q, G_s, W_q, W_s, offsets):
    """Block-scaled data gradient out_e = deq(G)[rows of e] @ deq(W_e)^T.

    G_q [M, K] codes with row-wise scales G_s [M, K/32]; W_q [E, N, K] codes
    with scales W_s [E, N, K/32] (blocks along K, the last axis).  Returns
    float64 [M, N], unrounded; rows outside every expert are NaN.
    Follows [TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩" (the backward grouped GEMMs in MXFP8)."""
    G = mx_dequantize(G_q, G_s, axis_block=1)
    E, N, K = W_q.shape
    out = np.full((G.shape[0], N), np.nan)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 <= r0:
            continue
        W = mx_dequantize(W_q[e], W_s[e], axis_block=1)       # [N, K]
        out[r0:r1] = G[r0:r1] @ W.T
    return out


def mx_wgrad(P_qT, P_sT, Q_qT, Q_sT, offsets):
    """Block-scaled weight gradient dW_e = P_e^T Q_e, summed over the rows of
    expert e, from the transposed copies: P_qT [p, M] with scales P_sT
    [p, M/32] (blocks of 32 rows inside one expert), Q_qT [q, M], Q_sT.
    Returns float64 [E, p, q], unrounded; an expert with no rows gets 0.
    Follows [CuTe] "무엇을 해결하려는가" (the transposed low-precision copy) and [TE] "다음 단계: NVFP4, GEMM 융합
    양자화, A2A 오버랩"."""
    P = mx_dequantize(P_qT, P_sT, axis_block=1)              # [p, M]
    Q = mx_dequantize(Q_qT, Q_sT, axis_block=1)              # [q, M]
    E = len(offsets) - 1
    dW = np.zeros((E, P.shape[0], Q.shape[0]))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            dW[e] = P[:, r0:r1] @ Q[:, r0:r1].T
    return dW


def mx_grouped_mlp_bwd(x_perm, H, A, dY, offsets, W1, W2, act: str, round_out: bool = True):
    """MXFP8 backward of the grouped expert MLP (see the reading above).

    Inputs are the bf16 values of x_perm [M, d], H [M, n1], A [M, n],
    dY [M, d], W1 [E, d, n1], W2 [E, n, d]; offsets multiples of 32.  Steps:
      1. dY -> row-wise blocks (along d) and the group-aware transposed copy;
      2. W2 -> blocks along d, W1 -> blocks along n1 (each weight's own
         reduction index in its data gradient);
      3. dA = deq(dY) deq(W2_e)^T;  dH = act'(H; dA), rounded to bf16;
      4. dW2_e = deq(A^T) deq(dY^T) over the expert's rows (A's transposed
         copy is the forward's);
      5. dH -> row-wise blocks (along n1) and the transposed copy;
      6. dX = deq(dH) deq(W1_e)^T;
      7. x -> transposed copy;  dW1_e = deq(x^T) deq(dH^T).
    Returns a dict with dH, dX, dW1, dW2 (bf16-rounded float64; with
    ``round_out=False`` the values just before that rounding, while steps 5-7
    still quantise the rounded dH) and the quantised intermediates (codes,
    scales) of steps 1, 2, 5 and 7.
    Follows [TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩" (GroupGemm + dActivation +
    Quantize/Transpose) and [CuTe] "무엇을 해결하려는가"."""
    from .moe import act_backward, bf16_round
    x_perm = np.asarray(x_perm, dtype=np.float64)
    H = np.asarray(H, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    W1 = np.asarray(W1, dtype=np.float64)
    W2 = np.asarray(W2, dtype=np.float64)
    M = x_perm.shape[0]
    E, d, n1 = W1.shape
    n = W2.shape[1]
    dy_q, dy_s = mx_quantize_rows(dY)
    dy_qT, dy_sT = mx_quantize_cols(dY, offsets, M)
    w2_q, w2_s = mx_quantize_rows(W2.reshape(E * n, d))
    w1_q, w1_s = mx_quantize_rows(W1.reshape(E * d, n1))
    w2_q, w2_s = w2_q.reshape(E, n, d), w2_s.reshape(E, n, d // 32)
    w1_q, w1_s = w1_q.reshape(E, d, n1), w1_s.reshape(E, d, n1 // 32)
    dA = mx_dgrad(dy_q, dy_s, w2_q, w2_s, offsets)
    dH = np.full((M, n1), np.nan)
    dH_exact = np.full((M, n1), np.nan)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            dH_exact[r0:r1] = act_backward(H[r0:r1], dA[r0:r1], act)
            dH[r0:r1] = bf16_round(dH_exact[r0:r1])
    rnd = bf16_round if round_out else (lambda v: v)
    a_qT, a_sT = mx_quantize_cols(A, offsets, M)
    dW2 = rnd(mx_wgrad(a_qT, a_sT, dy_qT, dy_sT, offsets))
    used = int(offsets[-1])
    dH0 = np.where(np.isnan(dH), 0.0, dH)
    dh_q, dh_s = mx_quantize_rows(dH0)
    dh_qT, dh_sT = mx_quantize_cols(dH0, offsets, M)
    dX = rnd(mx_dgrad(dh_q, dh_s, w1_q, w1_s, offsets))
    x_qT, x_sT = mx_quantize_cols(x_perm, offsets, M)
    dW1 = rnd(mx_wgrad(x_qT, x_sT, dh_qT, dh_sT, offsets))
    return {"dH": dH if round_out else dH_exact, "dX": dX, "dW1": dW1, "dW2": dW2,
            "dy_q": dy_q[:used], "dy_s": dy_s[:used], "dy_qT": dy_qT, "dy_sT": dy_sT,
            "w2_q": w2_q, "w2_s": w2_s, "w1_q": w1_q, "w1_s": w1_s,
            "dh_q": dh_q[:used], "dh_s": dh_s[:used], "dh_qT": dh_qT, "dh_sT": dh_sT,
            "x_qT": x_qT, "x_sT": x_sT}
