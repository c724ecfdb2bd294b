"""MXFP8 path vs the oracle's OCP MX quantiser.

* The weight quantiser and the standalone group-aware quantiser run on
  generator inputs (plus planted edge blocks): codes and scales must be
  bit-exact.
* The fused FC1 epilogue quantises its own bf16 A.  Its codes and scales,
  row-wise and transposed, must equal the OCP MX quantiser applied to that
  bf16 A bit for bit on every block.  Separately, A itself is compared with
  the oracle's independently computed A within the bf16 tolerance.
* The block-scaled FC2 output is compared with the oracle's MX FC2 on the
  oracle's own quantised A and W2, within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def _lib():
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    return M


def decode_w2_scales(s, E, n, d):
    s = s.cpu().numpy()
    e, b, c = np.meshgrid(np.arange(E), np.arange(n // 32), np.arange(d), indexing="ij")
    off = (e * (n // 32) * d + ((b // 4) * (d // 128) + c // 128) * 512 + (c % 32) * 16 +
           ((c % 128) // 32) * 4 + b % 4)
    return s[off]


def decode_a_scales(s, offsets, M_cap, n):
    """[M_cap, n/32] row-wise scales from the MMA-tiled layout (-1 outside
    every expert)."""
    s = s.cpu().numpy()
    out = -np.ones((M_cap, n // 32), np.int64)
    E = len(offsets) - 1
    b = np.arange(n // 32)
    for e in range(E):
        for row0 in range(int(offsets[e]), int(offsets[e + 1]), 128):
            for r in range(row0, min(row0 + 128, int(offsets[e + 1]))):
                rr = r - row0
                off = ((row0 // 32) * (n // 128) + b // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + b % 4
                out[r] = s[off]
    return out


def _plant(v):
    """Edge blocks into a float64 [rows, cols] array (values stay bf16)."""
    v = v.copy()
    v[0, 0:32] = 0.0                                      # all-zero block
    v[1, 0:32] = 2.0 ** np.arange(-10, 22)[:32] * 1e-3    # wide range -> many subnormal codes
    v[1, 0:32] = O.bf16_round(v[1, 0:32])
    v[2, 0:32] = 2.0 ** 5 * np.linspace(-1.9, 1.9, 32)    # saturating maximum
    v[2, 0:32] = O.bf16_round(v[2, 0:32])
    v[3, 32:64] = np.ldexp(1.0, np.arange(32) % 13 - 6) * np.where(np.arange(32) % 2, -1, 1)
    v[4, 32:64] = -0.0
    v[4, 40] = 3.0
    v[5, 0:32] = 1e-30                                    # tiny: code 0 scales
    v[5, 0:32] = O.bf16_round(v[5, 0:32])
    return v


def test_weight_quantiser_bit_exact():
    M = _lib()
    E, n, d = 3, 256, 384
    W2 = WL.w2(21, E, n, d, 0.02, "cuda")
    w = f64(W2)
    w[0] = _plant(w[0])
    w[2, :, 7] = 0.0                                      # an all-zero column
    W2 = torch.from_numpy(w).to(torch.bfloat16).cuda()
    q, s = M.mx_quantize_weights(W2)
    torch.cuda.synchronize()
    qo, so = O.mx_quantize_weights(w)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(decode_w2_scales(s, E, n, d), so)


# (rows, cols, offsets): the second shape has a partial 128-row tile and an
# odd number of 32-column blocks
QUANT_SHAPES = [(256, 256, [0, 64, 64, 192, 256 - 32]), (224, 96, [0, 64, 64, 160, 192])]


@pytest.mark.parametrize("rows,cols,offs", QUANT_SHAPES, ids=["256x256", "224x96"])
def test_group_aware_quantiser_bit_exact(rows, cols, offs):
    M = _lib()
    offsets = np.array(offs)                             # empty expert; last 32 rows unused
    src = f64(WL.normal((rows, cols), (22, WL.X, 0), 1.0, "cuda"))
    src = _plant(src)
    src_t = torch.from_numpy(src).to(torch.bfloat16).cuda()
    q, s, qT, sT, err = M.mx_quantize(src_t, cuda_i32(offsets))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = int(offsets[-1])
    qo, so = O.mx_quantize_rows(src[:R])
    assert np.array_equal(q.cpu().numpy()[:R], qo)
    assert np.array_equal(s.cpu().numpy()[:R], so)
    qTo, sTo = O.mx_quantize_cols(src, offsets, rows)
    assert np.array_equal(qT.cpu().numpy()[:, :R], qTo[:, :R])
    assert np.array_equal(sT.cpu().numpy()[:, :R // 32], sTo[:, :R // 32])


def decode_k_tiles(sT, offsets, rows, cols):
    """[cols, rows/32] column-block scales from the reduction-tile layout
    (-1 outside every expert): the K step starting at row t0 of an expert
    keeps column c's four 32-row blocks in chunk (t0/32)*(cols/128) + c/128,
    at the chunk offset of row c % 128 and block (r - t0)/32."""
    sT = sT.cpu().numpy()
    out = -np.ones((cols, rows // 32), np.int64)
    c = np.arange(cols)
    cr = c % 128
    for e in range(len(offsets) - 1):
        for t0 in range(int(offsets[e]), int(offsets[e + 1]), 128):
            for r32 in range(t0, min(t0 + 128, int(offsets[e + 1])), 32):
                kb = (r32 - t0) // 32
                off = ((t0 // 32) * (cols // 128) + c // 128) * 512 + (cr % 32) * 16 + (cr // 32) * 4 + kb
                out[:, r32 // 32] = sT[off]
    return out


TILED_SHAPES = [(448, 256, [0, 64, 64, 288, 416]), (256, 384, [0, 128, 128, 224])]


@pytest.mark.parametrize("rows,cols,offs", TILED_SHAPES, ids=["448x256", "256x384"])
def test_tiled_quantiser_bit_exact(rows, cols, offs):
    """moe_mx_quantize_tiled (the quantiser the MXFP8 backward runs on dY, x
    and dH): codes and both tiled scale layouts equal the oracle's OCP MX
    quantiser bit for bit on every row of an expert, with experts of 0, 64,
    128 and 224 rows (tiles of 128 and a 96-row tail) and the planted edge
    blocks; the row-only and transposed-only calls give the same bytes, and
    rows past every expert stay untouched."""
    M = _lib()
    offsets = np.array(offs)
    R = int(offsets[-1])
    src = _plant(f64(WL.normal((rows, cols), (25, WL.X, 0), 1.0, "cuda")))
    src[40, 128:160] = -0.0                                # a block of negative zeros
    src_t = torch.from_numpy(src).to(torch.bfloat16).cuda()
    offs_t = cuda_i32(offsets)
    q, s, qT, sT, err = M.mx_quantize_tiled(src_t, offs_t)
    q1, s1, _, _, e1 = M.mx_quantize_tiled(src_t, offs_t, transposed=False)
    _, _, qT2, sT2, e2 = M.mx_quantize_tiled(src_t, offs_t, rowwise=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and int(e1.item()) == 0 and int(e2.item()) == 0
    qo, so = O.mx_quantize_rows(src[:R])
    assert np.array_equal(q.cpu().numpy()[:R], qo)
    assert np.array_equal(decode_a_scales(s, offsets, rows, cols)[:R], so)
    qTo, sTo = O.mx_quantize_cols(src, offsets, rows)
    assert np.array_equal(qT.cpu().numpy()[:, :R], qTo[:, :R])
    assert np.array_equal(decode_k_tiles(sT, offsets, rows, cols)[:, :R // 32], sTo[:, :R // 32])
    assert torch.equal(q1[:R], q[:R]) and torch.equal(qT2[:, :R], qT[:, :R])
    assert np.array_equal(decode_a_scales(s1, offsets, rows, cols)[:R], so)
    assert np.array_equal(decode_k_tiles(sT2, offsets, rows, cols)[:, :R // 32], sTo[:, :R // 32])
    # the plain-layout quantiser emits the same codes
    qp, sp, qTp, sTp, ep = M.mx_quantize(src_t, offs_t)
    torch.cuda.synchronize()
    assert torch.equal(qp[:R], q[:R]) and torch.equal(qTp[:, :R], qT[:, :R])
    # rows past every expert: untouched
    sentinel = torch.full((rows, cols), 0x5A, dtype=torch.uint8, device="cuda")
    M.lib().moe_mx_quantize_tiled(src_t.data_ptr(), rows, cols, offs_t.data_ptr(), len(offs) - 1,
                                  sentinel.data_ptr(), s.data_ptr(), None, None, err.data_ptr(),
                                  None)
    torch.cuda.synchronize()
    assert bool((sentinel[R:] == 0x5A).all()) and torch.equal(sentinel[:R], q[:R])


def test_tiled_quantiser_reports_unaligned_offsets():
    """A 32-row block must lie inside one expert: offsets that are not
    multiples of 32 raise MOE_DEV_BAD_OFFSETS in the error word (reported,
    not repaired), and aligned offsets leave it clear."""
    M = _lib()
    src = WL.normal((256, 128), (26, WL.X, 0), 1.0, "cuda")
    _, _, _, _, bad = M.mx_quantize_tiled(src, cuda_i32(np.array([0, 96, 150, 224])))
    _, _, _, _, good = M.mx_quantize_tiled(src, cuda_i32(np.array([0, 96, 160, 224])))
    torch.cuda.synchronize()
    assert int(bad.item()) & M.DEV_BAD_OFFSETS
    assert int(good.item()) == 0


def _mx_case(act, E=4, d=256, n=256, counts=(96, 0, 160, 32), seed=23):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M_cap = int(off[-1]) + 32
    x = WL.normal((M_cap, d), (seed, WL.X, 0), 1.0, "cuda")
    W1 = (WL.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu" else
          WL.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = WL.w2(seed, E, n, d, 0.05, "cuda")
    return off, M_cap, x, W1, W2


def _check_blocks(gpu_a, gpu_q, gpu_s, what):
    """Codes and scales bit-exact on every block against the OCP MX
    quantiser applied to the GPU's own bf16 A (the quantiser's input is the
    bf16-rounded A).  Blocks are 32 consecutive entries along the last
    axis."""
    ga = gpu_a.reshape(gpu_a.shape[0], -1, 32)
    qo, so = O.mx_quantize_blocks(ga)
    gq = gpu_q.reshape(gpu_q.shape[0], -1, 32)
    bad = ~((gq == qo).all(axis=2) & (gpu_s == so))
    assert not bad.any(), (what, "blocks differing", int(bad.sum()), "of", bad.size,
                           "first at", tuple(int(v) for v in np.argwhere(bad)[0]))


# (d, n, counts): the second shape gives an expert three 128-row blocks (the
# second CTA of its last row pair has no rows) and an output width d that
# ends in a single 128-column half
FWD_SHAPES = [(256, 256, (96, 0, 160, 32)), (384, 256, (288, 0, 96, 64))]


@pytest.mark.parametrize("shape", FWD_SHAPES, ids=["d256", "d384_rows288"])
@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
def test_fused_fc1_mx_epilogue_and_block_scaled_fc2(act, shape):
    M = _lib()
    E = 4
    d, n, counts = shape
    off, M_cap, x, W1, W2 = _mx_case(act, E, d, n, counts)
    buf = M.mx_buffers(E, n, d, M_cap, "cuda")
    M.mx_quantize_weights(W2, buf["w2_q"], buf["w2_s"])
    h, a, y, err = M.grouped_mlp_fwd(x, cuda_i32(off), W1, W2, act, save_h=True, mx=buf)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = int(off[-1])
    H, A, _ = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act, round_out=False)
    ga = f64(a)[:R]
    assert_rms_close(ga, A[:R], f"{act} A (bf16)")
    # row-wise codes / scales (MMA-tiled scales decoded)
    gs = decode_a_scales(buf["a_s"], off, M_cap, n)[:R]
    _check_blocks(ga, buf["a_q"].cpu().numpy()[:R], gs, "rows")
    # transposed copy: column blocks of 32 rows inside each expert (offsets
    # are multiples of 32, so the blocks of A^T's rows never cross experts)
    gT = buf["a_qT"].cpu().numpy()[:, :R]
    gsT = buf["a_sT"].cpu().numpy()[:, :R // 32]
    _check_blocks(ga.T.copy(), gT, gsT, "cols")
    # decoded codes everywhere within the MX error of the oracle's A
    deq = O.mx_dequantize(buf["a_q"].cpu().numpy()[:R], gs.astype(np.uint8), axis_block=1)
    assert np.linalg.norm(deq - A[:R]) <= 0.05 * np.linalg.norm(A[:R])
    # block-scaled FC2 vs the oracle's MX FC2 on the same bf16 A (the GPU's,
    # checked against the oracle above): a one-step bf16 difference in A can
    # flip an E4M3 code, which is A's parity, not FC2's
    qa, sa = O.mx_quantize_rows(ga)
    qw, sw = O.mx_quantize_weights(f64(W2))
    Yo = O.mx_fc2(qa, sa, qw, sw, off)
    assert_rms_close(f64(y)[:R], Yo[:R], f"{act} Y (MXFP8 FC2)")
    # and close to the bf16 product (the MX error is small)
    _, _, Yb = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act)
    assert np.linalg.norm(f64(y)[:R] - Yb[:R]) <= 0.08 * np.linalg.norm(Yb[:R])


def test_mx_forward_max_experts_with_skipped_weights():
    """1024 experts (the library's limit), most of them empty, with W2
    quantised only for the experts that receive rows (the routing offsets
    given to the weight quantiser, as the training step does).  A and the
    block-scaled Y match the oracle on every row; no empty expert's W2
    codes were written."""
    M = _lib()
    act, E, d, n = "swiglu", 1024, 128, 128
    counts = [32 * (1 + (e % 3 == 0)) if e % 7 == 0 else 0 for e in range(E)]
    off, M_cap, x, W1, W2 = _mx_case(act, E, d, n, counts, seed=24)
    offs = cuda_i32(off)
    buf = M.mx_buffers(E, n, d, M_cap, "cuda")
    buf["w2_q"].fill_(0xA5)
    M.mx_quantize_weights(W2, buf["w2_q"], buf["w2_s"], offsets=offs)
    h, a, y, err = M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True, mx=buf)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    R = int(off[-1])
    _, A, _ = O.grouped_mlp_fwd(f64(x), off, f64(W1), f64(W2), act, round_out=False)
    assert_rms_close(f64(a)[:R], A[:R], "E=1024 A (bf16)")
    qa, sa = O.mx_quantize_rows(f64(a)[:R])            # FC2's input: the GPU's bf16 A
    qw, sw = O.mx_quantize_weights(f64(W2))
    assert_rms_close(f64(y)[:R], O.mx_fc2(qa, sa, qw, sw, off)[:R], "E=1024 Y (MXFP8 FC2)")
    empty = torch.tensor([e for e in range(E) if counts[e] == 0], device="cuda")
    assert bool((buf["w2_q"][empty] == 0xA5).all())


def test_mx_requires_32_aligned_offsets():
    M = _lib()
    off, M_cap, x, W1, W2 = _mx_case("swiglu", counts=(96, 0, 150, 32))   # 96+150 not aligned
    Mc = 320                                                             # multiple of 32
    buf = M.mx_buffers(4, 256, 256, Mc, "cuda")
    M.mx_quantize_weights(W2, buf["w2_q"], buf["w2_s"])
    x2 = torch.zeros((Mc, 256), dtype=torch.bfloat16, device="cuda")
    x2[:M_cap] = x
    _, _, _, err = M.grouped_mlp_fwd(x2, cuda_i32(off), W1, W2, "swiglu", mx=buf)
    torch.cuda.synchronize()
    assert int(err.item()) & M.DEV_BAD_OFFSETS


# both tile configurations of the quantising epilogue (2-SM tiles, the
# automatic choice for FC2 and FC1-dgrad, and single-CTA tiles forced), on a
# layer with d = 256 and one with d = 384, whose second 256-column tile has
# one 128-column half past N
@pytest.mark.parametrize("pair_mode", [1, 0])
@pytest.mark.parametrize("E,d,n,counts", [(4, 256, 128, [128, 0, 96, 64]),
                                          (4, 384, 128, [512, 0, 288, 256])])
def test_group_gemm_quantize_outputs(E, d, n, counts, pair_mode):
    """GroupGemm + Quantize: FC2's epilogue (forward) and FC1-dgrad's (MXFP8
    backward) also write the row-wise MXFP8 copy of the bf16 they store.
    The codes and scales equal the OCP MX quantiser applied to that bf16
    output, bit for bit, on every row inside an expert."""
    import dropless_grouped_gemm_gb300 as MM
    prev = MM.set_pair_mma(pair_mode)
    try:
        _group_gemm_quantize(E, d, n, counts)
    finally:
        MM.set_pair_mma(prev)


def _group_gemm_quantize(E, d, n, counts):
    M = _lib()
    import dropless_grouped_gemm_gb300 as MM
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    M_cap = int(off[-1]) + 32
    R = int(off[-1])
    x = WL.normal((M_cap, d), (81, WL.X, 0), 1.0, "cuda")
    W1 = WL.w1_interleaved(81, E, d, n, 0.05, "cuda")
    W2 = WL.w2(81, E, n, d, 0.05, "cuda")
    offs = cuda_i32(off)
    bufs = MM.mx_buffers(E, n, d, M_cap, "cuda", quantize_y=True)
    MM.mx_quantize_weights(W2, bufs["w2_q"], bufs["w2_s"])
    h, a, y, err = MM.grouped_mlp_fwd(x, offs, W1, W2, "swiglu", save_h=True, mx=bufs)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q, s = O.mx_quantize_rows(f64(y)[:R])
    assert np.array_equal(bufs["y_q"][:R].cpu().numpy(), q)
    assert np.array_equal(bufs["y_s"][:R].cpu().numpy(), s)
    # backward: dX of FC1-dgrad
    dy = WL.normal((M_cap, d), (81, WL.DY, 0), 1.0, "cuda")
    w2q, w2s = MM.mx_quantize_weights_rowwise(W2)
    w1q, w1s = MM.mx_quantize_weights_rowwise(W1)
    ops = dict(a_qT=bufs["a_qT"], a_sT=bufs["a_sT"], w2_q=w2q, w2_s=w2s, w1_q=w1q, w1_s=w1s,
               dx_q=torch.empty((M_cap, d), dtype=torch.uint8, device="cuda"),
               dx_s=torch.empty((M_cap, d // 32), dtype=torch.uint8, device="cuda"))
    _, dx, _, _, err = MM.grouped_mlp_bwd_mx(x, h, dy, offs, ops, "swiglu")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q, s = O.mx_quantize_rows(f64(dx)[:R])
    assert np.array_equal(ops["dx_q"][:R].cpu().numpy(), q)
    assert np.array_equal(ops["dx_s"][:R].cpu().numpy(), s)
