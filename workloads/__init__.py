"""Seeded synthetic workloads for the dropless MoE expert MLP.

This module only *synthesises inputs*.  It holds none of the method's
arithmetic (no routing, no GEMM, no activation), so both the CPU oracle and
the CUDA path may draw their inputs from it.

Generator
---------
Every tensor element is a pure function of ``(tensor key, flat index)``:

* ``h = fmix32(fmix32(index_lo ^ k0) ^ index_hi ^ k1)``, where ``fmix32`` is
  the public MurmurHash3 32-bit finaliser (Appleby), ``k0/k1`` are derived
  from the key by the same finaliser, and ``index_lo/hi`` are the two 32-bit
  halves of the flat index;
* the top 16 bits of ``h`` index a 65,536-entry quantile table
  ``q[i] = std * Phi^-1((i + 1/2) / 65536)`` (computed in float64 with
  ``statistics.NormalDist``), rounded to bf16 (or float32 for logits).

Only integer operations and one table gather are involved, so the same
element has the same bits on the CPU and on a GPU, and an oracle can
regenerate just the elements it samples (``*_at`` functions).

Workloads follow the pages' benchmark shapes: the cuDNN-Frontend grouped
GEMM benchmark shape (E=8, 4096 tokens per expert, K=8192, N=4096, BF16) from
"NVIDIA CuTe DSL 융합 커널은 MoE 학습의 CPU·메모리 병목을 지운다", section
"공개된 근거에서 확인되는 점"; and a fine-grained, skewed dropless layer
(DeepSeek-V3-like d=7168, 256 experts, top-8) for the ragged case discussed in
"NVIDIA Transformer Engine JAX dropless MoE", section on ragged tensors.
"""
from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np
import torch

_M32 = 0xFFFFFFFF

# tensor ids used in keys
X, W_GATE, W_UP, W2, DY, LOGITS, DO, W1_PLAIN = 1, 2, 3, 4, 5, 6, 7, 8


def _fmix32_int(h: int) -> int:
    h &= _M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    h ^= h >> 16
    return h


def _fmix32_t(h: torch.Tensor) -> torch.Tensor:
    # h holds values in [0, 2^32) as int64; products wrap in two's complement
    # and the mask keeps the exact low 32 bits.
    h = h ^ (h >> 16)
    h = (h * 0x85EBCA6B) & _M32
    h = h ^ (h >> 13)
    h = (h * 0xC2B2AE35) & _M32
    h = h ^ (h >> 16)
    return h


def key_words(*key: int) -> tuple[int, int]:
    """Two 32-bit seed words for a tensor key (config, tensor id, expert...)."""
    a, b = 0x9E3779B9, 0x7F4A7C15
    for v in key:
        a = _fmix32_int(a ^ (v & _M32))
        b = _fmix32_int(b ^ a ^ ((v >> 32) & _M32))
    return a, b


def hash_index(idx: torch.Tensor, key: tuple[int, ...]) -> torch.Tensor:
    """32-bit hash of int64 flat indices under ``key``."""
    k0, k1 = key_words(*key)
    lo = idx & _M32
    hi = (idx >> 32) & _M32
    return _fmix32_t(_fmix32_t(lo ^ k0) ^ hi ^ k1)


_TABLES: dict[tuple, torch.Tensor] = {}


def _quantile_table_f64() -> np.ndarray:
    nd = statistics.NormalDist()
    return np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)],
                    dtype=np.float64)


_Q64: np.ndarray | None = None


def quantiles_f64() -> np.ndarray:
    global _Q64
    if _Q64 is None:
        _Q64 = _quantile_table_f64()
    return _Q64


def _table(std: float, dtype: torch.dtype, device) -> torch.Tensor:
    k = (float(std), dtype, str(device))
    t = _TABLES.get(k)
    if t is None:
        q = torch.from_numpy(quantiles_f64() * std)  # float64, exact scale
        if dtype == torch.bfloat16:
            # float64 -> float32 (RNE) -> bf16 (RNE)
            t = q.to(torch.float32).to(torch.bfloat16)
        else:
            t = q.to(dtype)
        t = t.to(device)
        _TABLES[k] = t
    return t


def normal_at(idx: torch.Tensor, key: tuple[int, ...], std: float,
              dtype=torch.bfloat16) -> torch.Tensor:
    """Elements at flat indices ``idx`` of the tensor named by ``key``."""
    h = hash_index(idx, key)
    tab = _table(std, dtype, idx.device)
    return tab[h >> 16]


def normal(shape, key: tuple[int, ...], std: float, device="cpu",
           dtype=torch.bfloat16, chunk: int = 1 << 26) -> torch.Tensor:
    """Whole tensor of ``shape`` (row-major flat indices)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        out[s:e] = normal_at(idx, key, std, dtype)
    return out.view(*shape)


# --------------------------------------------------------------------------
# expert weights: gate / up halves generated separately, then laid out
# --------------------------------------------------------------------------

def w_gate_up_at(cfg_id: int, e: int, rows: torch.Tensor, cols: torch.Tensor,
                 n: int, which: int, std: float) -> torch.Tensor:
    """W_gate (which=W_GATE) or W_up (which=W_UP) of expert e, [d, n] row-major."""
    return normal_at(rows * n + cols, (cfg_id, which, e), std)


def w1_interleaved(cfg_id: int, E: int, d: int, n: int, std: float,
                   device="cpu", experts=None) -> torch.Tensor:
    """W1 [E, d, 2n]: column 2j is gate_j, column 2j+1 is up_j.

    The values are the same elements as ``w_gate``/``w_up`` below; only the
    storage order differs.  Building it here (instead of by a repack kernel)
    keeps the product path free of test-only layout work."""
    experts = range(E) if experts is None else experts
    out = torch.empty((len(experts), d, 2 * n), dtype=torch.bfloat16, device=device)
    for i, e in enumerate(experts):
        g = normal((d, n), (cfg_id, W_GATE, e), std, device)
        u = normal((d, n), (cfg_id, W_UP, e), std, device)
        v = out[i].view(d, n, 2)
        v[:, :, 0] = g
        v[:, :, 1] = u
    return out


def w_split(cfg_id: int, E: int, d: int, n: int, std: float, device="cpu"):
    g = torch.stack([normal((d, n), (cfg_id, W_GATE, e), std, device) for e in range(E)])
    u = torch.stack([normal((d, n), (cfg_id, W_UP, e), std, device) for e in range(E)])
    return g, u


def w1_plain(cfg_id: int, E: int, d: int, n: int, std: float, device="cpu",
             experts=None) -> torch.Tensor:
    """Non-gated W1 [E, d, n] (squared-ReLU)."""
    experts = range(E) if experts is None else experts
    return torch.stack([normal((d, n), (cfg_id, W1_PLAIN, e), std, device)
                        for e in experts])


def w2(cfg_id: int, E: int, n: int, d: int, std: float, device="cpu",
       experts=None) -> torch.Tensor:
    experts = range(E) if experts is None else experts
    return torch.stack([normal((n, d), (cfg_id, W2, e), std, device) for e in experts])


# --------------------------------------------------------------------------
# routing inputs (the router itself is outside the expert-MLP path; its
# outputs, top-k indices and probabilities, are synthetic inputs here)
# --------------------------------------------------------------------------

def zipf_bias(E: int, s: float) -> np.ndarray:
    """b_e = ln p_e with p_e proportional to (e+1)^-s (float64)."""
    p = np.array([(e + 1.0) ** (-s) for e in range(E)], dtype=np.float64)
    p /= p.sum()
    return np.log(p)


def logits(cfg_id: int, T: int, E: int, zipf_s: float | None = None,
           empty_expert: int | None = None) -> np.ndarray:
    """Router logits [T, E] float32: N(0,1) (+ Zipf bias), optional -inf column."""
    lg = normal((T, E), (cfg_id, LOGITS, 0), 1.0, "cpu", torch.float64).numpy()
    if zipf_s is not None:
        lg = lg + zipf_bias(E, zipf_s)[None, :]
    lg = lg.astype(np.float32)
    if empty_expert is not None:
        lg[:, empty_expert] = -np.inf
    return lg


def topk_route(lg: np.ndarray, k: int):
    """Top-k experts per token (ties -> lower expert index) and the softmax of
    the k selected logits, float32.  Returns (topk_idx int32 [T,k], probs f32)."""
    T = lg.shape[0]
    if T == 0:
        return np.zeros((0, k), np.int32), np.zeros((0, k), np.float32)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(lg, order, axis=1).astype(np.float32)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m).astype(np.float32)
    probs = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
    return order.astype(np.int32), probs


def identity_route(E: int, m: int):
    """k=1 routing with token t -> expert t // m (balanced, m tokens each)."""
    T = E * m
    idx = (np.arange(T, dtype=np.int64) // m).astype(np.int32).reshape(T, 1)
    return idx, np.ones((T, 1), np.float32)


# --------------------------------------------------------------------------
# workload table
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int
    T: int
    d: int
    E: int
    k: int
    n: int
    act: str                 # "swiglu" | "geglu" | "srelu"
    backward: bool
    routing: str             # "logits" | "identity"
    zipf_s: float | None = None
    empty_expert: int | None = None
    align: int = 1
    mxfp8: bool = False
    gather: bool = False     # GEMMs read token rows through the routing map
    x_std: float = 1.0
    w_std: float = 0.02
    dy_std: float = 1.0
    notes: str = ""

    @property
    def gated(self) -> bool:
        return self.act in ("swiglu", "geglu")

    @property
    def n1(self) -> int:
        """FC1 output width (2n when gated)."""
        return 2 * self.n if self.gated else self.n

    @property
    def M_cap(self) -> int:
        return self.T * self.k + self.E * (self.align - 1)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_t512_d128_e4_top2_n256_swiglu_fwd", 0, 512, 128, 4, 2, 256,
                 "swiglu", False, "logits", empty_expert=3,
                 notes="expert 3 forced empty (logit -inf)"),
        Workload("balanced_e8_m4096_k8192_n4096_swiglu", 1, 8 * 4096, 8192, 8, 1, 2048,
                 "swiglu", True, "identity",
                 notes="cuDNN-FE benchmark shape; counts fixed, equal"),
        Workload("zipf_t4096_d7168_e256_top8_n2048_swiglu", 2, 4096, 7168, 256, 8, 2048,
                 "swiglu", True, "logits", zipf_s=1.2),
        # the same layer with the permutes fused into the GEMMs' loads
        Workload("zipf_t4096_d7168_e256_top8_n2048_swiglu_gather", 2, 4096, 7168, 256, 8, 2048,
                 "swiglu", True, "logits", zipf_s=1.2, gather=True),
        Workload("balanced_e8_m4096_k8192_n4096_geglu", 3, 8 * 4096, 8192, 8, 1, 2048,
                 "geglu", True, "identity"),
        Workload("balanced_e8_m4096_k8192_n2048_srelu", 5, 8 * 4096, 8192, 8, 1, 2048,
                 "srelu", True, "identity"),
        Workload("zipf_t4096_d7168_e256_top8_n2048_mxfp8", 4, 4096, 7168, 256, 8, 2048,
                 "swiglu", False, "logits", zipf_s=1.2, align=32, mxfp8=True),
        # MXFP8 training: the forward above plus the MXFP8 backward
        Workload("zipf_t4096_d7168_e256_top8_n2048_mxfp8_train", 4, 4096, 7168, 256, 8, 2048,
                 "swiglu", True, "logits", zipf_s=1.2, align=32, mxfp8=True),
        Workload("balanced_e8_m4096_k8192_n4096_mxfp8_train", 1, 8 * 4096, 8192, 8, 1, 2048,
                 "swiglu", True, "identity", mxfp8=True,
                 notes="same tensors as the balanced bf16 layer; MXFP8 forward and backward"),
    ]
}


def route_inputs(w: Workload):
    """(topk_idx int32 [T,k], probs float32 [T,k]) for a workload."""
    if w.routing == "identity":
        return identity_route(w.E, w.T // w.E)
    lg = logits(w.cfg_id, w.T, w.E, w.zipf_s, w.empty_expert)
    return topk_route(lg, w.k)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of ``w`` with some sizes changed (for small parity cases)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(changes)
    return Workload(**d)
