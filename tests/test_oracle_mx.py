"""Pins for the oracle's MXFP8 quantiser (OCP MX v1.0 block rule, E4M3).

Pinned by the E4M3 format's own values, exhaustive comparison over every
bf16 magnitude in range with a library cast (torch's float8_e4m3fn, round to
nearest even), saturation and tie edges, power-of-two blocks that round-trip
exactly, amax at 2^k, all-zero blocks and the transposition identity."""
import numpy as np
import pytest
import torch

import oracle as O


def test_e4m3_known_values():
    t = O.e4m3_decode_table()
    assert t[0x38] == 1.0
    assert t[0x7E] == 448.0
    assert t[0x01] == 2.0 ** -9          # smallest subnormal
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x07] == 7 / 8 * 2.0 ** -6
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert t[0xB8] == -1.0


def test_e4m3_decode_matches_library():
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = O.e4m3_decode_table()
    nan = np.isnan(ours)
    assert (np.isnan(lib) == nan).all()
    assert (lib[~nan] == ours[~nan]).all()


def test_e4m3_encode_exhaustive_bf16_vs_library():
    """Every bf16 value with |v| <= 448 (both signs) encodes like torch's
    round-to-nearest-even cast."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        v = (bits << 16).view(np.float32).astype(np.float64)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    ours = O.e4m3_encode(v)
    lib = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # the library maps exact zeros of either sign to their signed zero code;
    # compare all values
    assert (ours == lib).all()


def test_fast_encoder_equals_bruteforce_definition():
    """Every finite bf16 value (both signs, beyond 448 too), random doubles,
    and every exact tie between neighbouring codes."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        v = (bits << 16).view(np.float32).astype(np.float64)
    v = v[np.isfinite(v)]
    assert (O.e4m3_encode(v) == O.e4m3_encode_bruteforce(v)).all()
    rng = np.random.default_rng(24)
    r = rng.standard_normal(200000) * np.exp(rng.uniform(-25, 8, 200000))
    assert (O.e4m3_encode(r) == O.e4m3_encode_bruteforce(r)).all()
    t = O.e4m3_decode_table()[:0x7F]
    mids = np.concatenate([(t[:-1] + t[1:]) / 2, -(t[:-1] + t[1:]) / 2])
    assert (O.e4m3_encode(mids) == O.e4m3_encode_bruteforce(mids)).all()


def test_e4m3_saturation_and_ties():
    enc = lambda x: int(O.e4m3_encode(np.array([x]))[0])
    for v in (448.0, 460.0, 464.0, 480.0, 511.0, 1e6):
        assert enc(v) == 0x7E
        assert enc(-v) == 0xFE
    assert enc(1.0 + 1 / 16) == 0x38          # tie between 1.0 and 1.125 -> even
    assert enc(1.125 + 1 / 16) == 0x3A        # tie between 1.125 and 1.25 -> even
    assert enc(2.0 ** -10) == 0x00            # tie between 0 and 2^-9 -> even (0)
    assert enc(3 * 2.0 ** -10) == 0x02        # tie between 2^-9 and 2^-8 -> even
    assert enc(-0.0) == 0x80
    assert enc(-(2.0 ** -12)) == 0x80


def test_scale_exponent_rule():
    assert O.e8m0_exponent(np.array([1.0]))[0] == -8
    assert O.e8m0_exponent(np.array([448.0]))[0] == 0
    assert O.e8m0_exponent(np.array([256.0]))[0] == 0
    assert O.e8m0_exponent(np.array([255.9]))[0] == -1
    assert O.e8m0_exponent(np.array([0.0]))[0] == -127
    assert O.e8m0_exponent(np.array([2.0 ** -200]))[0] == -127     # clamp
    for k in range(-20, 20):
        assert O.e8m0_exponent(np.array([2.0 ** k]))[0] == k - 8


def test_power_of_two_blocks_roundtrip():
    rng = np.random.default_rng(20)
    for _ in range(50):
        top = int(rng.integers(-30, 30))
        ex = top - rng.integers(0, 14, size=32)        # within the E4M3 range below amax
        ex[0] = top
        sign = rng.choice([-1.0, 1.0], size=32)
        blk = sign * np.ldexp(1.0, ex)
        q, s = O.mx_quantize_blocks(blk[None, :])
        back = O.e4m3_decode(q[0]) * 2.0 ** (int(s[0]) - 127)
        assert (back == blk).all()


def test_all_zero_block():
    q, s = O.mx_quantize_blocks(np.zeros((1, 32)))
    assert s[0] == 0 and (q == 0).all()


def test_amax_at_power_of_two_and_saturation_region():
    blk = np.zeros(32)
    blk[0] = 2.0 ** 5
    blk[1] = 2.0 ** 5 * 1.9       # amax/X = 486 -> saturates to 448
    q, s = O.mx_quantize_blocks(blk[None, :])
    assert s[0] == 127 + 5 - 8
    assert q[0, 0] == 0x78       # 256 = 1.0 * 2^8 -> exponent field 15 (15 << 3)
    assert q[0, 1] == 0x7E       # saturated


def test_transpose_identity():
    rng = np.random.default_rng(21)
    M, n = 96, 64
    A = O.bf16_round(rng.standard_normal((M, n)))
    offsets = np.array([0, 32, 32, 96])
    qT, sT = O.mx_quantize_cols(A, offsets)
    qR, sR = O.mx_quantize_rows(A.T)     # rows of A^T are columns of A
    assert (qT == qR).all() and (sT == sR).all()


def test_weight_blocks_run_along_n():
    """W2's blocks run along n (FC2's reduction index): expert e's codes and
    scales equal the row-wise quantisation of W2[e]^T (rows of W2[e]^T are
    columns of W2[e]).  An all-zero column block and a block holding a
    single large value make blocks along d give different codes."""
    rng = np.random.default_rng(22)
    E, n, d = 2, 64, 96
    W2 = O.bf16_round(rng.standard_normal((E, n, d)) * 0.05)
    W2[0, 0:32, 3] = 0.0
    W2[1, 40, 7] = 300.0
    q, s = O.mx_quantize_weights(W2)
    assert q.shape == (E, n, d) and s.shape == (E, n // 32, d)
    for e in range(E):
        qR, sR = O.mx_quantize_rows(W2[e].T)
        assert (q[e].T == qR).all() and (s[e].T == sR).all()
    # the zero block gets scale code 0; 300 = 1.17 * 2^8 gives exponent 8 - 8 = 0 (code 127)
    assert s[0, 0, 3] == 0 and s[1, 1, 7] == 127


def test_rowwise_dequant_error_bound():
    """Each dequantised element is within half an E4M3 spacing of the value
    (relative 2^-4 for normals) unless it saturates."""
    rng = np.random.default_rng(22)
    A = O.bf16_round(rng.standard_normal((64, 128)))
    q, s = O.mx_quantize_rows(A)
    D = O.mx_dequantize(q, s, axis_block=1)
    X = np.repeat(2.0 ** (s.astype(np.int64) - 127), 32, axis=1)
    sat = np.abs(A) / X >= 448
    err = np.abs(D - A)[~sat]
    bound = np.maximum(np.abs(A) * 2.0 ** -4, 2.0 ** -10 * X)[~sat]
    assert (err <= bound + 1e-300).all()


def test_mx_fc2_matches_dequantised_product():
    rng = np.random.default_rng(23)
    E, n, d = 3, 64, 32
    offsets = np.array([0, 32, 32, 96])
    A = O.bf16_round(rng.standard_normal((96, n)))
    W2 = O.bf16_round(rng.standard_normal((E, n, d)) * 0.02)
    Aq, As = O.mx_quantize_rows(A)
    Wq, Ws = O.mx_quantize_weights(W2)
    Y = O.mx_fc2(Aq, As, Wq, Ws, offsets)
    Ad = O.mx_dequantize(Aq, As, 1)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            Wd = O.mx_dequantize(Wq[e], Ws[e], 0)
            assert (Y[r0:r1] == O.bf16_round(Ad[r0:r1] @ Wd)).all()
            # and near the unquantised product: the floor-based scale
            # saturates block maxima in [1.75, 2) * 2^k, so single elements
            # can be off by ~10%; the relative Frobenius error stays small
            ref = A[r0:r1] @ W2[e]
            rel = np.linalg.norm(Y[r0:r1] - ref) / np.linalg.norm(ref)
            assert rel < 0.05
