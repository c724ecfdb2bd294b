"""Write coverage with NaN-poisoned outputs: every output buffer starts as
NaN; afterwards every row inside an expert is finite and equal, bit for bit,
to the run on unpoisoned buffers (nothing read an output before writing
it), and every row outside all experts is still NaN (nothing wrote there).
Expert sizes 0, 1, 127, 128, 129 and 255 rows straddle the 128-row tiles
(multiples of 32 on the MXFP8 path); a second layer adds hot experts of 300
and 600 rows, which run in the 2-SM launch of the split GEMMs."""
import numpy as np
import pytest
import torch

import workloads as W
from _helpers import cuda_i32

pytestmark = pytest.mark.gpu


def _poisoned(shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def _check(name, got, ref, R):
    g, r = got.float(), ref.float()
    assert torch.isfinite(g[:R]).all(), f"{name}: unwritten or non-finite rows inside the experts"
    assert torch.equal(got[:R], ref[:R]), f"{name}: differs from the unpoisoned run"
    assert torch.isnan(g[R:]).all(), f"{name}: rows past every expert were written"


def _layer(counts, d, n, act, tail, seed):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    E, R = len(counts), int(off[-1])
    M_cap = R + tail
    n1 = n if act == "srelu" else 2 * n
    x = W.normal((M_cap, d), (seed, W.X, 0), 1.0, "cuda")
    dy = W.normal((M_cap, d), (seed, W.DY, 0), 1.0, "cuda")
    W1 = (W.w1_plain(seed, E, d, n, 0.05, "cuda") if act == "srelu"
          else W.w1_interleaved(seed, E, d, n, 0.05, "cuda"))
    W2 = W.w2(seed, E, n, d, 0.05, "cuda")
    return off, E, R, M_cap, n1, x, dy, W1, W2


# the second layer has hot experts (300 and 600 rows, ragged 32-row ends):
# on this skinny layer they run in the GEMMs' 2-SM launch, the rest in the
# single-CTA one
BF16_COUNTS = {"small": [127, 0, 1, 129, 128, 255], "hot": [300, 0, 1, 129, 600, 255]}


@pytest.mark.parametrize("layer", sorted(BF16_COUNTS))
@pytest.mark.parametrize("act", ["swiglu", "srelu"])
def test_bf16_layer_writes_exactly_the_expert_rows(act, layer):
    import dropless_grouped_gemm_gb300 as M
    off, E, R, M_cap, n1, x, dy, W1, W2 = _layer(BF16_COUNTS[layer], 256, 128, act, 37, 91)
    d, n = x.shape[1], W2.shape[1]
    offs = cuda_i32(off)

    def run(poison):
        mk = _poisoned if poison else (lambda s: torch.zeros(s, dtype=torch.bfloat16, device="cuda"))
        h, a, y = mk((M_cap, n1)), mk((M_cap, n)), mk((M_cap, d))
        M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True, h_saved=h, a=a, y_perm=y)
        dh, dx, dW1, dW2 = mk((M_cap, n1)), mk((M_cap, d)), mk(tuple(W1.shape)), mk(tuple(W2.shape))
        _, _, _, _, err = M.grouped_mlp_bwd(x, h, a, dy, offs, W1, W2, act, dh=dh, dx_perm=dx,
                                            dW1=dW1, dW2=dW2)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return dict(h=h, a=a, y=y, dh=dh, dx=dx), dict(dW1=dW1, dW2=dW2)

    rows_p, w_p = run(True)
    rows_z, w_z = run(False)
    for k_ in rows_p:
        _check(k_, rows_p[k_], rows_z[k_], R)
    for k_ in w_p:                   # every expert's weight gradient is written (zeros if empty)
        assert torch.equal(w_p[k_], w_z[k_]), k_
    assert float(w_p["dW1"][1].float().abs().max()) == 0.0


@pytest.mark.parametrize("hot", [False, True], ids=["spread", "hot"])
def test_routed_backward_writes_exactly_the_expert_rows(hot):
    import dropless_grouped_gemm_gb300 as M
    act = "swiglu"
    E, T, k = 6, 300, 2
    rng = np.random.default_rng(92)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[idx == E - 1] = 0                    # expert E-1 empty
    if hot:
        # expert 0 takes every token (300 rows: the GEMMs' 2-SM launch)
        idx[:, 0] = 0
        idx[:, 1] = rng.integers(1, E - 1, T)
    probs = torch.from_numpy(rng.random((T, k)).astype(np.float32)).cuda().view(-1)
    r = M.route_offsets(cuda_i32(idx), E, 8)             # pad rows inside the experts
    M_cap = r["pair_of_row"].numel()
    R = int(r["offsets"][-1].item())
    d, n = 128, 128
    x = W.normal((T, d), (92, W.X, 0), 1.0, "cuda")
    dO = W.normal((T, d), (92, W.DO, 0), 1.0, "cuda")
    H = W.normal((M_cap, 2 * n), (92, W.X, 1), 1.0, "cuda")
    W1 = W.w1_interleaved(92, E, d, n, 0.05, "cuda")
    W2 = W.w2(92, E, n, d, 0.05, "cuda")
    xp, dop = M.permute(x, r["pair_of_row"], k), M.permute(dO, r["pair_of_row"], k)

    def run(poison):
        mk = _poisoned if poison else (lambda s: torch.zeros(s, dtype=torch.bfloat16, device="cuda"))
        dh, ap, dx = mk((M_cap, 2 * n)), mk((M_cap, n)), mk((M_cap, d))
        dsp = torch.full((M_cap, 1), float("nan") if poison else 0.0, device="cuda")
        out = M.grouped_mlp_bwd_routed(xp, H, dop, r["pair_of_row"], probs, r["offsets"], W1, W2,
                                       act, dh=dh, a_scaled=ap, ds_part=dsp, dx_perm=dx)
        torch.cuda.synchronize()
        assert int(out[-1].item()) == 0
        return dict(dh=dh, a_scaled=ap, dx=dx, ds_part=dsp)

    p, z = run(True), run(False)
    for k_ in p:
        _check(k_, p[k_], z[k_], R)


@pytest.mark.parametrize("counts", [[96, 0, 32, 160, 128, 224], [320, 0, 32, 160, 608, 224]],
                         ids=["small", "hot"])
def test_mxfp8_layer_writes_exactly_the_expert_rows(counts):
    import dropless_grouped_gemm_gb300 as M
    act = "swiglu"
    off, E, R, M_cap, n1, x, dy, W1, W2 = _layer(counts, 256, 128, act, 64, 93)
    d, n = x.shape[1], W2.shape[1]
    offs = cuda_i32(off)

    def run(poison):
        mk = _poisoned if poison else (lambda s: torch.zeros(s, dtype=torch.bfloat16, device="cuda"))
        bufs = M.mx_buffers(E, n, d, M_cap, "cuda")
        M.mx_quantize_weights(W2, bufs["w2_q"], bufs["w2_s"])
        h, a, y = mk((M_cap, n1)), mk((M_cap, n)), mk((M_cap, d))
        M.grouped_mlp_fwd(x, offs, W1, W2, act, save_h=True, h_saved=h, a=a, y_perm=y, mx=bufs)
        w2q, w2s = M.mx_quantize_weights_rowwise(W2)
        w1q, w1s = M.mx_quantize_weights_rowwise(W1)
        ops = dict(a_qT=bufs["a_qT"], a_sT=bufs["a_sT"], w2_q=w2q, w2_s=w2s, w1_q=w1q, w1_s=w1s)
        dh, dx, dW1, dW2 = mk((M_cap, n1)), mk((M_cap, d)), mk(tuple(W1.shape)), mk(tuple(W2.shape))
        _, _, _, _, err = M.grouped_mlp_bwd_mx(x, h, dy, offs, ops, act, dh=dh, dx_perm=dx,
                                               dW1=dW1, dW2=dW2)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        return dict(h=h, a=a, y=y, dh=dh, dx=dx), dict(dW1=dW1, dW2=dW2)

    rows_p, w_p = run(True)
    rows_z, w_z = run(False)
    for k_ in rows_p:
        _check(k_, rows_p[k_], rows_z[k_], R)
    for k_ in w_p:
        assert torch.equal(w_p[k_], w_z[k_]), k_
