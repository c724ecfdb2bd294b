"""The seeded input generator: layout and distribution checks."""
import numpy as np
import torch

import oracle as O
import workloads as W


def test_interleaved_w1_matches_oracle_repack():
    g, u = W.w_split(7, 2, 16, 8, 0.02)
    w1 = W.w1_interleaved(7, 2, 16, 8, 0.02)
    ref = O.interleave_gate_up(g.float().numpy(), u.float().numpy())
    assert (w1.float().numpy() == ref).all()


def test_sampled_elements_equal_whole_tensor():
    full = W.normal((33, 17), (3, W.X, 0), 1.0)
    idx = torch.tensor([0, 5, 17 * 3 + 2, 33 * 17 - 1])
    assert torch.equal(W.normal_at(idx, (3, W.X, 0), 1.0), full.reshape(-1)[idx])


def test_distribution():
    v = W.normal((1 << 18,), (9, W.X, 0), 1.0).float().numpy()
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01
    w = W.normal((1 << 18,), (9, W.W2, 0), 0.02).float().numpy()
    assert abs(w.std() - 0.02) < 0.0005
    # different keys give different streams
    assert not np.array_equal(v[:64], W.normal((64,), (9, W.X, 1), 1.0).float().numpy())


def test_routing_inputs():
    w = W.WORKLOADS["tiny_t512_d128_e4_top2_n256_swiglu_fwd"]
    idx, p = W.route_inputs(w)
    assert idx.shape == (512, 2) and (idx != 3).all()          # forced-empty expert
    assert (idx[:, 0] != idx[:, 1]).all()
    assert np.allclose(p.sum(1), 1.0, atol=1e-6)
    z = W.WORKLOADS["zipf_t4096_d7168_e256_top8_n2048_swiglu"]
    zi, _ = W.route_inputs(z)
    counts = np.bincount(zi.reshape(-1), minlength=256)
    assert (counts == 0).sum() >= 3        # several empty experts
    assert counts.max() > 30 * np.median(counts[counts > 0])   # skewed
