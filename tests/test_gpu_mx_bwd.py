"""MXFP8 backward (moe_grouped_mlp_bwd_mx, moe_mx_quantize_weights_rowwise)
vs the oracle's MXFP8 backward.

* The row-wise weight quantiser is bit-exact against the oracle's OCP MX
  quantiser (codes, and scales decoded from the weight tiles).
* The backward's four outputs are compared with oracle.mx.mx_grouped_mlp_bwd
  on the same bf16 inputs, within the bf16 tolerance.  Both sides quantise
  dY, x, A and the weights identically (the quantisers are bit-exact); dH is
  quantised from each side's own bf16 dH, which may differ by one bf16 step
  at a few elements, so dX and dW1 can differ by one E4M3 step there.  dW1
  and dW2 are also compared element-wise with the oracle's block-scaled
  weight gradient of the GPU's own bf16 operands (stage-wise).
* Expert sizes cover several 128-row tiles, ragged last reduction steps
  (32/64/96 rows), empty experts and many small experts."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import mx as X
import workloads as W
from _helpers import assert_rms_close, cuda_i32, f64

pytestmark = pytest.mark.gpu


def _M():
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    return M


def decode_weight_tiles(s, rows, K):
    """[rows, K/32] scales from the weight-tile layout."""
    s = s.cpu().numpy()
    r, b = np.meshgrid(np.arange(rows), np.arange(K // 32), indexing="ij")
    rr = r % 128
    off = ((r // 128) * (K // 128) + b // 4) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + b % 4
    return s[off]


def test_rowwise_weight_quantiser_bit_exact():
    M = _M()
    E, n, d = 3, 256, 384
    W2 = W.w2(21, E, n, d, 0.05, "cuda")
    W2[0, 0, :32] = 0                                      # all-zero block
    W2[1, 5, 32:64] = torch.tensor(2.0 ** np.arange(-20, 12), dtype=torch.bfloat16)
    q, s = M.mx_quantize_weights_rowwise(W2)
    torch.cuda.synchronize()
    rq, rs = X.mx_quantize_rows(f64(W2).reshape(E * n, d))
    assert np.array_equal(q.cpu().numpy().reshape(E * n, d), rq)
    assert np.array_equal(decode_weight_tiles(s, E * n, d), rs)


def test_both_direction_weight_quantiser_bit_exact():
    """moe_mx_quantize_weights2: the forward's copy (blocks along n) equals
    moe_mx_quantize_weights' and the backward's (blocks along d) the
    oracle's row-wise quantiser, both bit for bit, from one pass."""
    M = _M()
    E, n, d = 3, 256, 384
    W2 = W.w2(22, E, n, d, 0.05, "cuda")
    W2[1, 7, 64:96] = 0                                     # all-zero row block
    W2[2, 0:32, 5] = torch.tensor(2.0 ** np.arange(-20, 12), dtype=torch.bfloat16)
    q, s, qr, sr = M.mx_quantize_weights2(W2)
    q1, s1 = M.mx_quantize_weights(W2)
    torch.cuda.synchronize()
    assert torch.equal(q, q1) and torch.equal(s, s1)
    rq, rs = X.mx_quantize_rows(f64(W2).reshape(E * n, d))
    assert np.array_equal(qr.cpu().numpy().reshape(E * n, d), rq)
    assert np.array_equal(decode_weight_tiles(sr, E * n, d), rs)
    cq, cs = X.mx_quantize_weights(f64(W2))
    assert np.array_equal(q.cpu().numpy(), cq)


@pytest.mark.parametrize("E,n,d", [(37, 256, 384), (1024, 128, 128)])
def test_weight_quantisers_skip_empty_experts(E, n, d):
    """With the routing offsets, the three weight quantisers write the used
    experts' codes and scales bit for bit as without them, and leave every
    byte of an expert that has no rows as it was (sentinel 0xA5).  Per
    expert, the codes are its [n, d] (or [d, n1]) slice and the scales a
    contiguous run of n*d/32 bytes in both tile layouts."""
    M = _M()
    # used and empty experts alternate irregularly; the used-expert list
    # spans two ballots (E = 37) or fills the library's limit (E = 1024)
    counts = [32 * (1 + e % 2) if e % 3 == 0 or e == 33 else 0 for e in range(E)]
    counts[E - 1] = 0                                   # the last expert empty
    offs = cuda_i32(np.concatenate([[0], np.cumsum(counts)]))
    used = [e for e in range(E) if counts[e]]
    W2 = W.w2(23, E, n, d, 0.05, "cuda")
    W1 = W.w1_interleaved(23, E, d, n // 2, 0.05, "cuda")   # [E, d, n]: rows per expert d
    fill = lambda t: torch.full_like(t, 0xA5)

    ui = torch.tensor(used, device="cuda")
    ei = torch.tensor([e for e in range(E) if not counts[e]], device="cuda")

    def check(full, part, per_e):
        for f, p in zip(full, part):
            f, p = f.reshape(E, -1), p.reshape(E, -1)
            assert f.shape[1] == per_e or f.shape[1] == per_e // 32
            assert torch.equal(p[ui], f[ui]), "a used expert differs"
            assert bool((p[ei] == 0xA5).all()), "an empty expert was written"

    full2 = M.mx_quantize_weights2(W2)
    part2 = M.mx_quantize_weights2(W2, *[fill(t) for t in full2], offsets=offs)
    full1 = M.mx_quantize_weights(W2)
    part1 = M.mx_quantize_weights(W2, *[fill(t) for t in full1], offsets=offs)
    fullr = M.mx_quantize_weights_rowwise(W1)
    partr = M.mx_quantize_weights_rowwise(W1, *[fill(t) for t in fullr], offsets=offs)
    torch.cuda.synchronize()
    check(full2, part2, n * d)
    check(full1, part1, n * d)
    check(fullr, partr, d * n)
    assert used[:3] == [0, 3, 6] and 33 in used and E - 1 not in used


def _layer(seed, counts, d, n, act, tail=64):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    assert (off % 32 == 0).all()
    M_cap = int(off[-1]) + tail
    n1 = n if act == "srelu" else 2 * n
    E = len(counts)
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    H = W.normal((M_cap, n1), (seed, W.X, 1), 1.0, "cuda")
    A = W.normal((M_cap, n), (seed, W.X, 2), 1.0, "cuda")
    dy = W.normal((M_cap, d), (seed, W.DY, 0), 1.0, "cuda")
    W1 = (W.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    return off, x, H, A, dy, W1, W2


def _gpu_bwd(off, x, H, A, dy, W1, W2, act, dW1=None, dW2=None, accumulate_dw=False,
             separate_dh_quant=False, workspace=None):
    M = _M()
    offs = cuda_i32(off)
    _, _, aT, sT, e0 = M.mx_quantize(A, offs)          # the forward's transposed copy of A
    w2_q, w2_s = M.mx_quantize_weights_rowwise(W2)
    w1_q, w1_s = M.mx_quantize_weights_rowwise(W1)
    mx = dict(a_qT=aT, a_sT=sT, w2_q=w2_q, w2_s=w2_s, w1_q=w1_q, w1_s=w1_s)
    dh, dx, dW1, dW2, err = M.grouped_mlp_bwd_mx(x, H, dy, offs, mx, act, dW1=dW1, dW2=dW2,
                                                  accumulate_dw=accumulate_dw,
                                                  separate_dh_quant=separate_dh_quant,
                                                  workspace=workspace)
    torch.cuda.synchronize()
    assert int(e0.item()) == 0 and int(err.item()) == 0
    # in automatic pair mode each weight gradient of a layer below 256 rows
    # per expert runs its experts of 256 rows or more in a launch of their
    # own (2-SM tiles)
    M_cap, E = x.shape[0], W2.shape[0]
    mode = M.set_pair_mma(M.PAIR_AUTO)
    M.set_pair_mma(mode)
    split = int(mode == M.PAIR_AUTO and E > 1 and M_cap < 256 * E)
    assert M.last_launch_count() == (8 if separate_dh_quant else 7) + 2 * split
    return dh, dx, dW1, dW2


CASES = [
    # name, counts (multiples of 32), d, n
    ("tiles_ragged_empty", [160, 0, 96, 288], 256, 128),
    ("single_expert_long_k", [1024], 256, 128),
    ("many_small", [32 * ((i * 5) % 4) for i in range(40)], 128, 128),
    # three 128-row blocks of d in the weight gradient and of an expert, and
    # d = 384 ending in a single 128-column half
    ("odd_row_blocks", [288, 32, 0, 416], 384, 128),
    # the library's expert limit: 1024 experts, most of them empty
    ("max_experts", [32 * (1 + (e % 3 == 0)) if e % 7 == 0 else 0 for e in range(1024)], 128, 128),
]


def test_mx_bwd_accumulate_dw():
    """MOE_FLAG_ACCUMULATE_DW on the MXFP8 backward: the block-scaled weight
    gradients are added to the given ones (one bf16 rounding of the sum);
    the empty expert's stay bit-identical."""
    act = "swiglu"
    counts = [160, 0, 96, 288]
    off, x, H, A, dy, W1, W2 = _layer(33, counts, 256, 128, act)
    ref = X.mx_grouped_mlp_bwd(f64(x), f64(H), f64(A), f64(dy), off, f64(W1), f64(W2), act,
                               round_out=False)
    old1 = W.normal(ref["dW1"].shape, (33, W.X, 90), float(np.sqrt((ref["dW1"] ** 2).mean())), "cuda")
    old2 = W.normal(ref["dW2"].shape, (33, W.X, 91), float(np.sqrt((ref["dW2"] ** 2).mean())), "cuda")
    dW1, dW2 = old1.clone(), old2.clone()
    dh, _, _, _ = _gpu_bwd(off, x, H, A, dy, W1, W2, act, dW1=dW1, dW2=dW2, accumulate_dw=True)
    s1, _ = _stagewise_wgrads(f64(x), f64(dh), f64(A), f64(dy), off, int(off[-1]))
    assert_rms_close(f64(dW1), f64(old1) + s1, "MX dW1 accumulated")
    assert_rms_close(f64(dW2), f64(old2) + ref["dW2"], "MX dW2 accumulated")
    assert torch.equal(dW1[1], old1[1]) and torch.equal(dW2[1], old2[1])


def _stagewise_wgrads(x, dh_gpu, a, dy, off, R):
    """The oracle's block-scaled weight gradients of the GPU's own bf16
    operands: dW1 = x^T dH from the GPU's dH, dW2 = A^T dY (A, dY and x are
    the generator's on both sides).  Rows past the experts are zeroed (they
    are outside every block)."""
    M = x.shape[0]
    dh0 = np.zeros_like(dh_gpu)
    dh0[:R] = dh_gpu[:R]
    dW1 = X.mx_wgrad(*X.mx_quantize_cols(x, off, M), *X.mx_quantize_cols(dh0, off, M), off)
    dW2 = X.mx_wgrad(*X.mx_quantize_cols(a, off, M), *X.mx_quantize_cols(dy, off, M), off)
    return dW1, dW2


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,counts,d,n", CASES, ids=[c[0] for c in CASES])
def test_mx_bwd_matches_oracle(name, counts, d, n, act):
    off, x, H, A, dy, W1, W2 = _layer(31, counts, d, n, act)
    dh, dx, dW1, dW2 = _gpu_bwd(off, x, H, A, dy, W1, W2, act)
    ref = X.mx_grouped_mlp_bwd(f64(x), f64(H), f64(A), f64(dy), off, f64(W1), f64(W2), act,
                               round_out=False)
    R = int(off[-1])
    assert_rms_close(f64(dh)[:R], ref["dH"][:R], f"{name}/{act} dH")
    assert_rms_close(f64(dW2), ref["dW2"], f"{name}/{act} dW2")
    # dX and dW1 element-wise against the oracle's block-scaled GEMMs of the
    # GPU's own dH (stage-wise); against the independent chain, whose dH may
    # differ by one bf16 step at a few elements and so flip an E4M3 code in
    # a 32-element block, in aggregate
    dh0 = np.zeros_like(f64(dh))
    dh0[:R] = f64(dh)[:R]
    sx = X.mx_dgrad(*X.mx_quantize_rows(dh0), ref["w1_q"], ref["w1_s"], off)
    assert_rms_close(f64(dx)[:R], sx[:R], f"{name}/{act} dX (stage-wise)")
    s1, s2 = _stagewise_wgrads(f64(x), f64(dh), f64(A), f64(dy), off, R)
    assert_rms_close(f64(dW1), s1, f"{name}/{act} dW1 (stage-wise)")
    assert_rms_close(f64(dW2), s2, f"{name}/{act} dW2 (stage-wise)")
    for nm, got, want in (("dX", f64(dx)[:R], ref["dX"][:R]), ("dW1", f64(dW1), ref["dW1"])):
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel <= 2e-2, (f"{name}/{act} {nm} relative error vs the independent chain", rel)
    for e in range(len(counts)):
        if counts[e] == 0:
            assert float(dW1[e].abs().max()) == 0 and float(dW2[e].abs().max()) == 0


def test_mx_bwd_close_to_bf16_backward():
    """The MXFP8 backward stays within MXFP8's error of the bf16 backward of
    the same layer (both on the GPU)."""
    M = _M()
    act = "swiglu"
    off, x, H, A, dy, W1, W2 = _layer(32, [256, 128, 0, 384], 256, 128, act)
    mx_out = _gpu_bwd(off, x, H, A, dy, W1, W2, act)
    bf_out = M.grouped_mlp_bwd(x, H, A, dy, cuda_i32(off), W1, W2, act)[:4]
    torch.cuda.synchronize()
    R = int(off[-1])
    for name, a, b in zip(("dH", "dX", "dW1", "dW2"), mx_out, bf_out):
        a, b = f64(a), f64(b)
        if name in ("dH", "dX"):
            a, b = a[:R], b[:R]
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel < (0.06 if name in ("dH", "dW2") else 0.09), (name, rel)


def test_mx_bwd_deterministic():
    act = "swiglu"
    off, x, H, A, dy, W1, W2 = _layer(33, [96, 224], 128, 128, act)
    a = _gpu_bwd(off, x, H, A, dy, W1, W2, act)
    b = _gpu_bwd(off, x, H, A, dy, W1, W2, act)
    R = int(off[-1])
    for p, q in zip(a, b):
        if p.shape[0] == x.shape[0]:
            p, q = p[:R], q[:R]
        assert torch.equal(p, q)


def _dh_sections(ws, lay, M_cap, n1):
    """dH's MXFP8 copies from the backward's workspace: row-wise codes [M,
    n1] and row-tile scales, transposed codes [n1, M] and K-tile scales."""
    sec = lambda nm, nbytes: ws[lay[nm]:lay[nm] + nbytes]
    return (sec("dh_q", M_cap * n1).view(M_cap, n1), sec("dh_s", M_cap * n1 // 8),
            sec("dh_qT", M_cap * n1).view(n1, M_cap), sec("dh_sT", M_cap * n1 // 8))


FUSE_CASES = [c for c in CASES if c[0] in ("tiles_ragged_empty", "odd_row_blocks", "many_small")]


@pytest.mark.parametrize("act", ["swiglu", "geglu", "srelu"])
@pytest.mark.parametrize("name,counts,d,n", FUSE_CASES, ids=[c[0] for c in FUSE_CASES])
def test_fused_dact_quantize_transpose(name, counts, d, n, act):
    """GroupGemm + dActivation + Quantize/Transpose: FC2-dgrad's epilogue
    writes dH's row-wise MXFP8 codes (row-tile scales) and its group-aware
    transposed copy (K-tile scales).  On every row and column block inside
    the experts they equal, bit for bit, (a) the separate tiled quantiser
    run on the same bf16 dH (the unfused control) and (b) the OCP MX
    quantiser of the oracle applied to the GPU's own bf16 dH; and every
    output of the backward equals the unfused control's bit for bit."""
    from test_gpu_mx import decode_a_scales, decode_k_tiles
    M = _M()
    off, x, H, A, dy, W1, W2 = _layer(35, counts, d, n, act)
    M_cap = x.shape[0]
    n1 = H.shape[1]
    R = int(off[-1])
    lay = M.mx_bwd_workspace_layout(M_cap, d, n, act)
    wf = torch.full((lay["bytes"],), 0x5A, dtype=torch.uint8, device="cuda")
    wu = torch.full((lay["bytes"],), 0xA5, dtype=torch.uint8, device="cuda")
    fused = _gpu_bwd(off, x, H, A, dy, W1, W2, act, workspace=wf)
    unfused = _gpu_bwd(off, x, H, A, dy, W1, W2, act, separate_dh_quant=True, workspace=wu)
    for nm, a, b in zip(("dh", "dx", "dW1", "dW2"), fused, unfused):
        if a.shape[0] == M_cap:
            a, b = a[:R], b[:R]
        assert torch.equal(a, b), nm
    fq, fs, fqT, fsT = _dh_sections(wf, lay, M_cap, n1)
    uq, us, uqT, usT = _dh_sections(wu, lay, M_cap, n1)
    assert torch.equal(fq[:R], uq[:R]) and torch.equal(fqT[:, :R], uqT[:, :R])
    gs_f = decode_a_scales(fs, off, M_cap, n1)[:R]
    gsT_f = decode_k_tiles(fsT, off, M_cap, n1)[:, :R // 32]
    assert np.array_equal(gs_f, decode_a_scales(us, off, M_cap, n1)[:R])
    assert np.array_equal(gsT_f, decode_k_tiles(usT, off, M_cap, n1)[:, :R // 32])
    gdh = f64(fused[0])[:R]
    qo, so = X.mx_quantize_rows(gdh)
    assert np.array_equal(fq[:R].cpu().numpy(), qo)
    assert np.array_equal(gs_f, so)
    qTo, sTo = X.mx_quantize_cols(gdh, off)
    assert np.array_equal(fqT[:, :R].cpu().numpy(), qTo[:, :R])
    assert np.array_equal(gsT_f, sTo[:, :R // 32])
