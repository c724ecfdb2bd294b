"""The whole layer (routing layout, permute, grouped MLP fwd/bwd, combine,
router-score gradient) captures into one CUDA graph: no call reads a count
back to the host.  Replaying the graph after writing a different routing
into the captured input buffer gives bit-identical results to eager calls
on that routing ([CuTe] "무엇을 해결하려는가" and [TE] "Transformer Engine이
제공하는 세 가지 구성 요소": counts unknown to the host, graph capture)."""
import numpy as np
import pytest
import torch

import bench as BE
import workloads as WL

pytestmark = pytest.mark.gpu


def _routing(seed, T, k, E):
    rng = np.random.default_rng(seed)
    # skewed: expert 0 popular, some experts empty
    logits = rng.standard_normal((T, E)) + np.log(1.0 / (np.arange(E) + 1.0) ** 1.5)
    idx = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    p = rng.random((T, k)).astype(np.float32)
    return idx, p / p.sum(1, keepdims=True)


@pytest.mark.parametrize("wname", ["zipf_t4096_d7168_e256_top8_n2048_swiglu",
                                   "zipf_t4096_d7168_e256_top8_n2048_swiglu_gather",
                                   "zipf_t4096_d7168_e256_top8_n2048_mxfp8_train"],
                         ids=["permuted", "gathered", "mxfp8_train"])
def test_layer_graph_capture_and_replay_with_new_routing(wname):
    """Each form of the layer step: with the permutes, with the GEMMs reading
    token rows through the routing map, and the MXFP8 training step (weight
    and activation quantisers, block-scaled GEMMs)."""
    import dropless_grouped_gemm_gb300 as M
    M.lib()
    # MXFP8 needs M_cap = T k + E (align - 1) to be a multiple of 32: E = 32
    w = WL.scaled(WL.WORKLOADS[wname], T=384, d=256, n=128, E=32 if "mxfp8" in wname else 16, k=4)
    inp, o = BE.make_inputs(w, "cuda")
    step = BE.make_step(w, inp, o)
    keys = ["h", "a", "y_perm", "out", "dprobs", "dh", "dx_perm", "dW1", "dW2", "dx"]
    if not w.gather:
        keys.append("x_perm")

    def snapshot():
        torch.cuda.synchronize()
        snap = {k_: o[k_].clone() for k_ in keys}
        snap["_rows"] = int(o["route"]["offsets"][-1].item())
        return snap

    def set_routing(seed):
        idx, p = _routing(seed, w.T, w.k, w.E)
        inp["topk_idx"].copy_(torch.from_numpy(idx))
        inp["probs"].copy_(torch.from_numpy(p))

    set_routing(1)
    step()                      # eager warm-up (also sets kernel attributes)
    eager1 = snapshot()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    rep1 = snapshot()
    set_routing(2)
    step()
    eager2 = snapshot()
    set_routing(2)
    g.replay()
    rep2 = snapshot()
    assert rep1["_rows"] == eager1["_rows"] and rep2["_rows"] == eager2["_rows"]
    for k_ in keys:
        a1, b1, a2, b2 = eager1[k_], rep1[k_], eager2[k_], rep2[k_]
        if a1.shape[0] == w.M_cap:     # rows past the used range are not written
            r1, r2 = eager1["_rows"], eager2["_rows"]
            a1, b1, a2, b2 = a1[:r1], b1[:r1], a2[:r2], b2[:r2]
        assert torch.equal(a1, b1), k_
        assert torch.equal(a2, b2), k_
    assert not torch.equal(eager1["out"], eager2["out"])
    assert int(o["err"].item()) == 0
