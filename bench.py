#!/usr/bin/env python
"""Benchmark of the dropless MoE expert-MLP path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Metric: grouped MoE MLP forward + backward useful TFLOP/s (FLOPs of real
rows only: 18 M d n for gated activations, 12 M d n for squared ReLU, M =
routed (token, expert) pairs), and the fraction of GB300 dense BF16 peak.

Default workload: the pages' grouped-GEMM benchmark shape (E=8 experts, 4096
tokens each, K=d=8192, N=2n=4096, SwiGLU forward + dSwiGLU backward, BF16;
counts fixed, equal and device-resident).  A step is one
moe_grouped_mlp_fwd (FC1+SwiGLU, FC2) plus one moe_grouped_mlp_bwd
(FC2-dgrad+dSwiGLU, FC2-wgrad, FC1-dgrad, FC1-wgrad).  Workloads with
routing (zipf_*) time the whole layer: routing layout, permute, forward,
combine, and their backward with the router-score gradient.

Inputs are seeded and synthetic (``workloads``), resident in HBM before the
timed region, and larger than L2 (no flush needed).  Timing: W warm-up
steps, then K steps between CUDA events on the launching stream, bracketed
by a synchronize on both sides.

The path runs on one GPU.  Its grouped GEMMs load shared weight tiles with
cluster-multicast TMA, which is kept to single-GPU processes: with
WORLD_SIZE > 1 (torchrun) or --gpus > 1 the bench prints one
``{"unavailable": ...}`` line and exits with status 2, before any CUDA or
process-group call.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "grouped MoE MLP fwd+bwd useful TFLOP/s and % of GB300 dense BF16/FP8 peak"
DEFAULT_WORKLOAD = "balanced_e8_m4096_k8192_n4096_swiglu"
KERNELS_FWD = ["fc1_act", "fc2"]
KERNELS_BWD = ["fc2_dgrad_dact", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad"]
# launch order of the MXFP8 backward (weight quantiser, then moe_grouped_mlp_bwd_mx,
# whose FC2-dgrad epilogue also quantises dH both ways)
KERNELS_MX_BWD = ["mx_quantize_w1_rows", "mx_quantize_dy", "mx_quantize_x", "mx_retile_a",
                  "fc2_dgrad_dact", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad"]


# ---------------------------------------------------------------- accounting
def useful_flops(w, M):
    """fwd + bwd FLOPs of real rows (the pages' arithmetic-intensity model
    counts the same terms: [Sonic] section on MoE arithmetic intensity).
    Forward-only workloads (the MXFP8 forward) have no backward term."""
    n1 = w.n1
    fwd = 2 * M * w.d * n1 + 2 * M * w.n * w.d
    bwd = 2 * M * w.d * w.n + 2 * M * w.n * w.d + 2 * M * n1 * w.d + 2 * M * w.d * n1
    return fwd, (bwd if w.backward else 0)


def kernel_work(w, M, E_ne):
    """Algorithmic FLOPs and bytes per launch of each grouped GEMM (bf16 =
    2 B; weights of non-empty experts only, also in the weight quantisers,
    which skip the empty experts; weight gradients of all experts, written
    as zeros for empty ones)."""
    d, n, n1, E = w.d, w.n, w.n1, w.E
    B = 2
    if w.mxfp8:
        # FC1 (bf16 MMA) writes bf16 A (+ H when training) and MX codes
        # (row-wise and transposed, 1 B each) and scales; the block-scaled
        # GEMMs stream E4M3 codes (1 B) plus one scale byte per 32 codes
        mxb = lambda elems: elems + elems // 32
        work = {
            "mx_quantize_weights": (0, E_ne * n * d * 2 + mxb(E_ne * n * d)),
            "fc1_act": (2 * M * d * n1, B * (M * d + E_ne * d * n1 + M * n) + 2 * mxb(M * n) +
                        (B * M * n1 if w.backward else 0)),
            "fc2": (2 * M * n * d, mxb(M * n) + mxb(E_ne * n * d) + B * M * d),
        }
        if w.backward:
            work.update({
                # W2 read once, both MXFP8 copies written
                "mx_quantize_weights2": (0, E_ne * n * d * 2 + 2 * mxb(E_ne * n * d)),
                "mx_quantize_w1_rows": (0, E_ne * d * n1 * 2 + mxb(E_ne * d * n1)),
                "mx_quantize_dy": (0, B * M * d + 2 * mxb(M * d)),
                "mx_quantize_x": (0, B * M * d + mxb(M * d)),
                "mx_retile_a": (0, 2 * (M * n // 32)),
                # reads dY codes, W2 codes, H; writes dH (bf16) and its two MXFP8 copies
                "fc2_dgrad_dact": (2 * M * d * n, mxb(M * d) + mxb(E_ne * n * d) + 2 * B * M * n1 +
                                   2 * mxb(M * n1)),
                "fc2_wgrad": (2 * M * n * d, mxb(M * n) + mxb(M * d) + B * E * n * d),
                "fc1_dgrad": (2 * M * n1 * d, mxb(M * n1) + mxb(E_ne * d * n1) + B * M * d),
                "fc1_wgrad": (2 * M * d * n1, mxb(M * d) + mxb(M * n1) + B * E * d * n1),
            })
        return work
    # routed workloads: the FC2-dgrad epilogue also writes A' (bf16) and the dS partials
    routed = w.routing != "identity"
    # gathered operands read the token tensor itself (T rows), not its
    # K-times larger permuted copy
    tok = w.T * d if w.gather else M * d
    return {
        "fc1_act": (2 * M * d * n1, B * (tok + E_ne * d * n1 + M * n + M * n1)),
        "fc2": (2 * M * n * d, B * (M * n + E_ne * n * d + M * d)),
        "fc2_dgrad_dact": (2 * M * d * n, B * (tok + E_ne * n * d + 2 * M * n1) +
                           ((B * M * n + 4 * M * ((n + 127) // 128)) if routed else 0)),
        "fc2_wgrad": (2 * M * n * d, B * (M * n + tok + E * n * d)),
        "fc1_dgrad": (2 * M * n1 * d, B * (M * n1 + E_ne * d * n1 + M * d)),
        "fc1_wgrad": (2 * M * d * n1, B * (tok + M * n1 + E * d * n1)),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# source files of each kernel family; a traffic figure is reported only while
# the files of the kernel it was measured on are unchanged
KERNEL_SOURCES = {
    "bf16": ("gemm.cu", "gemm.cuh", "ptx.cuh", "act.cuh", "mx.cuh"),
    "mx": ("mx.cu", "mx.cuh", "mxgemm.cuh", "ptx.cuh", "act.cuh"),
}


def kernel_family(w, kernel):
    """The block-scaled GEMMs of the MXFP8 workloads live in mx.cu; FC1 (and
    every GEMM of the bf16 workloads) in gemm.cu."""
    return "mx" if (w.mxfp8 and kernel != "fc1_act") else "bf16"


def kernel_src_hash(family="bf16"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        h.update(open(os.path.join(ROOT, "dropless_grouped_gemm_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, w):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current source of that kernel's family; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    j = json.load(open(p))
    rec = j.get(w.name, {}).get(kernel)
    if not rec or rec.get("src_hash") != kernel_src_hash(kernel_family(w, kernel)):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.p = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- inputs
def make_inputs(w, dev):
    import torch
    import dropless_grouped_gemm_gb300 as M
    d, n, E = w.d, w.n, w.E
    inp = {}
    if w.gated:
        inp["W1"] = WL.w1_interleaved(w.cfg_id, E, d, n, w.w_std, dev)
    else:
        inp["W1"] = WL.w1_plain(w.cfg_id, E, d, n, w.w_std, dev)
    inp["W2"] = WL.w2(w.cfg_id, E, n, d, w.w_std, dev)
    if w.routing == "identity":
        m = w.T // E
        inp["offsets"] = torch.arange(0, w.T + 1, m, dtype=torch.int32, device=dev)
        inp["x_perm"] = WL.normal((w.M_cap, d), (w.cfg_id, WL.X, 0), w.x_std, dev)
        inp["dy_perm"] = WL.normal((w.M_cap, d), (w.cfg_id, WL.DY, 0), w.dy_std, dev)
        inp["M"] = w.T
        inp["E_ne"] = E
    else:
        idx, probs = WL.route_inputs(w)
        inp["topk_idx"] = torch.from_numpy(idx).to(dev)
        inp["probs"] = torch.from_numpy(probs).to(dev)
        inp["x"] = WL.normal((w.T, d), (w.cfg_id, WL.X, 0), w.x_std, dev)
        inp["dO"] = WL.normal((w.T, d), (w.cfg_id, WL.DO, 0), w.dy_std, dev)
        counts = np.bincount(idx.reshape(-1), minlength=E)
        inp["M"] = int(counts.sum())
        inp["E_ne"] = int((counts > 0).sum())
    # outputs / intermediates, allocated once
    Mc, n1 = w.M_cap, w.n1
    bf = torch.bfloat16
    o = {k: torch.empty(s, dtype=bf, device=dev) for k, s in [
        ("h", (Mc, n1)), ("a", (Mc, n)), ("y_perm", (Mc, d)), ("dh", (Mc, n1)),
        ("dx_perm", (Mc, d)), ("dW1", tuple(inp["W1"].shape)), ("dW2", tuple(inp["W2"].shape))]}
    o["err"] = torch.zeros(1, dtype=torch.int32, device=dev)
    if w.routing != "identity":
        o["x_perm"] = torch.empty((Mc, d), dtype=bf, device=dev)
        o["dy_perm"] = torch.empty((Mc, d), dtype=bf, device=dev)
        o["out"] = torch.empty((w.T, d), dtype=bf, device=dev)
        o["dx"] = torch.empty((w.T, d), dtype=bf, device=dev)
        o["dprobs"] = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        if w.backward and not w.mxfp8:
            o["a_scaled"] = torch.empty((Mc, n), dtype=bf, device=dev)
            o["ds_part"] = torch.empty((Mc, (n + 127) // 128), dtype=torch.float32, device=dev)
        o["ws"] = torch.empty(max(16, M.route_workspace_size(w.T, w.k, E)), dtype=torch.uint8,
                              device=dev)
        o["route"] = {
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "row_of_pair": torch.empty(w.T * w.k, dtype=torch.int32, device=dev),
            "pair_of_row": torch.empty(Mc, dtype=torch.int32, device=dev),
            "true_total": torch.empty(1, dtype=torch.int32, device=dev),
            "err": o["err"],
        }
    if w.mxfp8:
        o["mx"] = M.mx_buffers(E, n, d, Mc, dev)
        if w.backward:
            u8 = torch.uint8
            o["mxb"] = {"w2_q": torch.empty((E, n, d), dtype=u8, device=dev),
                        "w2_s": torch.empty(E * n * d // 32, dtype=u8, device=dev),
                        "w1_q": torch.empty((E, d, n1), dtype=u8, device=dev),
                        "w1_s": torch.empty(E * d * n1 // 32, dtype=u8, device=dev),
                        "ws": torch.empty(M.mx_bwd_workspace_size(Mc, d, n, w.act), dtype=u8,
                                          device=dev)}
    return inp, o


def make_step(w, inp, o):
    """One pass of the path; returns the number of libmoe kernel launches."""
    import dropless_grouped_gemm_gb300 as M
    act = w.act

    def mx_backward(x_perm, dy_perm, offsets):
        """MXFP8 backward: weights quantised along their data-gradient
        reduction index, then the eight launches of grouped_mlp_bwd_mx."""
        mx, mb = o["mx"], o["mxb"]
        M.mx_quantize_weights_rowwise(inp["W1"], mb["w1_q"], mb["w1_s"], offsets=offsets)
        ops = dict(a_qT=mx["a_qT"], a_sT=mx["a_sT"], w2_q=mb["w2_q"], w2_s=mb["w2_s"],
                   w1_q=mb["w1_q"], w1_s=mb["w1_s"])
        M.grouped_mlp_bwd_mx(x_perm, o["h"], dy_perm, offsets, ops, act, dh=o["dh"],
                             dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"], err=o["err"],
                             workspace=mb["ws"])
        return 1 + M.last_launch_count()

    if w.routing == "identity" and w.mxfp8:
        def step_mx_id():
            M.mx_quantize_weights2(inp["W2"], o["mx"]["w2_q"], o["mx"]["w2_s"], o["mxb"]["w2_q"],
                                   o["mxb"]["w2_s"], offsets=inp["offsets"])
            n = M.last_launch_count()
            M.grouped_mlp_fwd(inp["x_perm"], inp["offsets"], inp["W1"], inp["W2"], act,
                              save_h=True, h_saved=o["h"], a=o["a"], y_perm=o["y_perm"],
                              err=o["err"], mx=o["mx"])
            n += M.last_launch_count()
            return n + mx_backward(inp["x_perm"], inp["dy_perm"], inp["offsets"])
        return step_mx_id

    if w.routing == "identity":
        def step():
            M.grouped_mlp_fwd(inp["x_perm"], inp["offsets"], inp["W1"], inp["W2"], act,
                              save_h=True, h_saved=o["h"], a=o["a"], y_perm=o["y_perm"],
                              err=o["err"])
            n = M.last_launch_count()
            M.grouped_mlp_bwd(inp["x_perm"], o["h"], o["a"], inp["dy_perm"], inp["offsets"],
                              inp["W1"], inp["W2"], act, dh=o["dh"], dx_perm=o["dx_perm"],
                              dW1=o["dW1"], dW2=o["dW2"], err=o["err"])
            return n + M.last_launch_count()
        return step

    T, k = w.T, w.k

    if w.mxfp8 and w.backward:
        def step_mx_train():
            n = 0
            r = M.route_offsets(inp["topk_idx"], w.E, w.align, w.M_cap, out=o["route"],
                                workspace=o["ws"])
            n += M.last_launch_count()
            M.permute(inp["x"], r["pair_of_row"], k, out=o["x_perm"], row_of_pair=r["row_of_pair"])
            n += M.last_launch_count()
            M.mx_quantize_weights2(inp["W2"], o["mx"]["w2_q"], o["mx"]["w2_s"], o["mxb"]["w2_q"],
                                   o["mxb"]["w2_s"], offsets=r["offsets"])
            n += M.last_launch_count()
            M.grouped_mlp_fwd(o["x_perm"], r["offsets"], inp["W1"], inp["W2"], act, save_h=True,
                              h_saved=o["h"], a=o["a"], y_perm=o["y_perm"], err=o["err"],
                              mx=o["mx"])
            n += M.last_launch_count()
            M.unpermute(o["y_perm"], r["row_of_pair"], T, k, probs=inp["probs"], out=o["out"])
            n += M.last_launch_count()
            M.permute(inp["dO"], r["pair_of_row"], k, scale=inp["probs"].view(-1),
                      out=o["dy_perm"], row_of_pair=r["row_of_pair"])
            n += M.last_launch_count()
            M.unpermute(o["y_perm"], r["row_of_pair"], T, k, dO=inp["dO"], dprobs=o["dprobs"],
                        combine=False)
            n += M.last_launch_count()
            n += mx_backward(o["x_perm"], o["dy_perm"], r["offsets"])
            M.unpermute(o["dx_perm"], r["row_of_pair"], T, k, out=o["dx"])
            n += M.last_launch_count()
            return n
        return step_mx_train

    if w.mxfp8:
        def step_mx():
            n = 0
            r = M.route_offsets(inp["topk_idx"], w.E, w.align, w.M_cap, out=o["route"],
                                workspace=o["ws"])
            n += M.last_launch_count()
            M.permute(inp["x"], r["pair_of_row"], k, out=o["x_perm"], row_of_pair=r["row_of_pair"])
            n += M.last_launch_count()
            M.mx_quantize_weights(inp["W2"], o["mx"]["w2_q"], o["mx"]["w2_s"], offsets=r["offsets"])
            n += M.last_launch_count()
            M.grouped_mlp_fwd(o["x_perm"], r["offsets"], inp["W1"], inp["W2"], act, a=o["a"],
                              y_perm=o["y_perm"], err=o["err"], mx=o["mx"])
            n += M.last_launch_count()
            M.unpermute(o["y_perm"], r["row_of_pair"], T, k, probs=inp["probs"], out=o["out"])
            n += M.last_launch_count()
            return n
        return step_mx

    if not w.backward:
        def step_fwd():
            # forward-only layer: routing layout, permute, expert MLP, combine
            n = 0
            r = M.route_offsets(inp["topk_idx"], w.E, w.align, w.M_cap, out=o["route"],
                                workspace=o["ws"])
            n += M.last_launch_count()
            M.permute(inp["x"], r["pair_of_row"], k, out=o["x_perm"], row_of_pair=r["row_of_pair"])
            n += M.last_launch_count()
            M.grouped_mlp_fwd(o["x_perm"], r["offsets"], inp["W1"], inp["W2"], act, a=o["a"],
                              y_perm=o["y_perm"], err=o["err"])
            n += M.last_launch_count()
            M.unpermute(o["y_perm"], r["row_of_pair"], T, k, probs=inp["probs"], out=o["out"])
            n += M.last_launch_count()
            return n
        return step_fwd

    if w.gather:
        def step_gather():
            # the permutes fused into the GEMMs' loads ([Sonic] "Gather
            # Fusion"): FC1, FC2-dgrad and both weight gradients read the
            # token rows of x and dO through the routing map
            n = 0
            r = M.route_offsets(inp["topk_idx"], w.E, w.align, w.M_cap, out=o["route"],
                                workspace=o["ws"])
            n += M.last_launch_count()
            M.grouped_mlp_fwd_gather(inp["x"], r["pair_of_row"], k, r["offsets"], inp["W1"],
                                     inp["W2"], act, save_h=True, h_saved=o["h"], a=o["a"],
                                     y_perm=o["y_perm"], err=o["err"])
            n += M.last_launch_count()
            M.unpermute(o["y_perm"], r["row_of_pair"], T, k, probs=inp["probs"], out=o["out"])
            n += M.last_launch_count()
            M.grouped_mlp_bwd_routed_gather(inp["x"], inp["dO"], r["pair_of_row"], k, o["h"],
                                            inp["probs"].view(-1), r["offsets"], inp["W1"],
                                            inp["W2"], act, dh=o["dh"], a_scaled=o["a_scaled"],
                                            ds_part=o["ds_part"], dx_perm=o["dx_perm"],
                                            dW1=o["dW1"], dW2=o["dW2"], err=o["err"])
            n += M.last_launch_count()
            M.router_grad_rows(o["ds_part"], r["row_of_pair"], T, k, dprobs=o["dprobs"])
            n += M.last_launch_count()
            M.unpermute(o["dx_perm"], r["row_of_pair"], T, k, out=o["dx"])
            n += M.last_launch_count()
            return n
        return step_gather

    def step():
        n = 0
        r = M.route_offsets(inp["topk_idx"], w.E, w.align, w.M_cap, out=o["route"],
                            workspace=o["ws"])
        n += M.last_launch_count()
        M.permute(inp["x"], r["pair_of_row"], k, out=o["x_perm"], row_of_pair=r["row_of_pair"])
        n += M.last_launch_count()
        M.grouped_mlp_fwd(o["x_perm"], r["offsets"], inp["W1"], inp["W2"], act, save_h=True,
                          h_saved=o["h"], a=o["a"], y_perm=o["y_perm"], err=o["err"])
        n += M.last_launch_count()
        M.unpermute(o["y_perm"], r["row_of_pair"], T, k, probs=inp["probs"], out=o["out"])
        n += M.last_launch_count()
        # backward: combine -> (scaled permute of dO, router-score gradient)
        # backward with the router gradient inside the expert MLP ([Sonic]
        # rewrite): dO gathered without the probability; FC2-dgrad applies it
        # and emits dS partials and A' = S*A; FC2-wgrad contracts A' with dO
        M.permute(inp["dO"], r["pair_of_row"], k, out=o["dy_perm"], row_of_pair=r["row_of_pair"])
        n += M.last_launch_count()
        M.grouped_mlp_bwd_routed(o["x_perm"], o["h"], o["dy_perm"], r["pair_of_row"],
                                 inp["probs"].view(-1), r["offsets"], inp["W1"], inp["W2"], act,
                                 dh=o["dh"], a_scaled=o["a_scaled"], ds_part=o["ds_part"],
                                 dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"], err=o["err"])
        n += M.last_launch_count()
        M.router_grad_rows(o["ds_part"], r["row_of_pair"], T, k, dprobs=o["dprobs"])
        n += M.last_launch_count()
        M.unpermute(o["dx_perm"], r["row_of_pair"], T, k, out=o["dx"])
        n += M.last_launch_count()
        return n
    return step


def event_names(w):
    if w.mxfp8 and w.backward:
        if w.routing == "identity":
            return ["mx_quantize_weights2"] + KERNELS_FWD + KERNELS_MX_BWD
        return (["route", "permute", "mx_quantize_weights2"] + KERNELS_FWD +
                ["combine", "permute_bwd", "router_grad"] + KERNELS_MX_BWD + ["unpermute_bwd"])
    if w.routing == "identity":
        return KERNELS_FWD + KERNELS_BWD
    if w.mxfp8:
        return ["route", "permute", "mx_quantize_weights"] + KERNELS_FWD + ["combine"]
    if not w.backward:
        return ["route", "permute"] + KERNELS_FWD + ["combine"]
    if w.gather:
        return (["route"] + KERNELS_FWD + ["combine"] + KERNELS_BWD +
                ["router_grad_rows", "unpermute_bwd"])
    return (["route", "permute"] + KERNELS_FWD + ["combine", "permute_bwd"] +
            KERNELS_BWD + ["router_grad_rows", "unpermute_bwd"])


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w, rows):
    """A bounded sample of the workload for the oracle: ``rows`` routed rows
    of expert 0 with that expert's weights (regenerated on the CPU)."""
    import torch
    d, n = w.d, w.n
    cpu = "cpu"
    f = lambda t: t.to(torch.float64).numpy()
    x = f(WL.normal((rows, d), (w.cfg_id, WL.X, 0), w.x_std, cpu))
    dy = f(WL.normal((rows, d), (w.cfg_id, WL.DY, 0), w.dy_std, cpu))
    W1 = f(WL.w1_interleaved(w.cfg_id, 1, d, n, w.w_std, cpu) if w.gated else
           WL.w1_plain(w.cfg_id, 1, d, n, w.w_std, cpu))
    W2 = f(WL.w2(w.cfg_id, 1, n, d, w.w_std, cpu))
    return x, dy, W1, W2


def oracle_step(w, x, dy, W1, W2, off):
    """One oracle pass over the sample: fwd+bwd; for the MXFP8 workloads the
    forward with the MX quantiser and the MXFP8 FC2 (and, when training, the
    MXFP8 backward)."""
    import oracle as O
    from oracle import mx as OX
    H, A, _ = O.grouped_mlp_fwd(x, off, W1, W2, w.act)
    if w.mxfp8:
        qa, sa = O.mx_quantize_rows(A)
        qw, sw = O.mx_quantize_weights(W2)
        O.mx_fc2(qa, sa, qw, sw, off)
        if w.backward:
            OX.mx_grouped_mlp_bwd(x, H, A, dy, off, W1, W2, w.act)
    elif w.backward:
        O.grouped_mlp_bwd(x, H, A, dy, off, W1, W2, w.act)


def time_oracle(w, rows, reps=1):
    x, dy, W1, W2 = oracle_sample(w, rows)
    off = np.array([0, rows])
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(w, x, dy, W1, W2, off)
    dt = (time.perf_counter() - t0) / reps
    fwd, bwd = useful_flops(w, rows)
    return (fwd + bwd) / dt / 1e12, dt


def cpu_cores():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


# ---------------------------------------------------------------- roofline
SUSTAINED_AFTER_S = 2.0


def roofline(kernel, flops, nbytes, t_s, peaks, fp8, region_s):
    """Roofline record of one kernel: achieved = algorithmic FLOPs (or
    bytes) per launch / its average live duration.  The tensor peak is the
    measured burst bf16 rate when the timed region is shorter than
    SUSTAINED_AFTER_S (the GPU has not settled at its power cap yet), the
    sustained rate otherwise; the other one is reported beside it.  FP8
    peaks are 2x the bf16 figure (the nominal dense ratio, not a
    measurement)."""
    mult = 2.0 if fp8 else 1.0
    burst = peaks["bf16_tflops"] * mult
    sust = peaks["bf16_tflops_sustained"] * mult
    use_sust = region_s >= SUSTAINED_AFTER_S
    tpeak = sust if use_sust else burst
    tag = "bf16_tflops_sustained" if use_sust else "bf16_tflops"
    if flops / (tpeak * 1e12) >= nbytes / (peaks["hbm_gbs"] * 1e9):
        ach = flops / t_s / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": round(ach, 1),
                "peak": round(tpeak, 1), "unit": "TFLOP/s",
                "peak_kind": (f"2 x {tag} (fp8 nominal ratio, {peaks['source']})" if fp8 else
                              f"{tag} ({peaks['source']})"),
                "frac": round(ach / tpeak, 4),
                "frac_burst": round(ach / burst, 4), "frac_sustained": round(ach / sust, 4),
                "algorithmic_per_launch": flops}
    ach = nbytes / t_s / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": round(ach, 1),
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "peak_kind": f"hbm_gbs ({peaks['source']})",
            "frac": round(ach / peaks["hbm_gbs"], 4), "algorithmic_per_launch": nbytes}


# ---------------------------------------------------------------- main
SINGLE_GPU_ONLY = ("single-GPU path: the grouped GEMMs use cluster-multicast TMA loads, which "
                   "run only in single-GPU processes; run one process per GPU as independent "
                   "replicas")


def world_size():
    return int(os.environ.get("WORLD_SIZE", "1"))


def run_reference(args, w):
    ws = world_size()
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    rows = args.ref_rows
    x, dy, W1, W2 = oracle_sample(w, rows)
    off = np.array([0, rows])

    def step():
        oracle_step(w, x, dy, W1, W2, off)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    fwd, bwd = useful_flops(w, rows)
    v = (fwd + bwd) / dt / 1e12
    sample = (f"{rows} rows of expert 0 ({w.d}x{w.n1} W1, {w.n}x{w.d} W2), oracle float64 "
              f"{('fwd (MXFP8 FC2)' if w.mxfp8 else 'fwd') if not w.backward else 'fwd+bwd'}"
              f"{' MXFP8' if w.mxfp8 and w.backward else ''} per step")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="steps of the pipelined end-to-end leg (default: --steps, at least "
                         "30; its first input copy is not overlapped, so more steps approach "
                         "the steady state)")
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="rows of the oracle's cpu_baseline sample")
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="rows per step of the --impl reference sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the timings of the rows built after the hot path (NVFP4 "
                         "statistics, GroupGemm + Quantize, device router)")
    ap.add_argument("--no-fusion-control", action="store_true",
                    help="skip the fused-against-unfused epilogue comparison")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WL.WORKLOADS[args.workload]

    if args.impl == "reference":
        return run_reference(args, w)

    if world_size() > 1 or args.gpus > 1:
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"unavailable": SINGLE_GPU_ONLY, "n_gpus": max(world_size(),
                                                                              args.gpus)}),
                  flush=True)
        return 2

    import torch
    lrank = 0
    dev = "cuda:0"
    torch.cuda.set_device(lrank)
    from dropless_grouped_gemm_gb300 import build as B
    B.build()
    import dropless_grouped_gemm_gb300 as M
    M.lib()

    inp, o = make_inputs(w, dev)
    step = make_step(w, inp, o)
    names = event_names(w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(o["err"].item()) != 0:
        raise SystemExit(f"device error bits {int(o['err'].item())}")

    # per-launch events for the timed region
    import ctypes
    per = len(names)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * per * args.steps)]
    for e in evs:          # torch creates the CUDA event on its first record
        e.record(stream)
    torch.cuda.synchronize()
    handles = (ctypes.c_void_p * len(evs))(*[e.cuda_event for e in evs])
    try:
        uuid = str(torch.cuda.get_device_properties(lrank).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        gpu_id = lrank
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    launches = 0
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    M.lib().moe_set_launch_events(handles, len(evs))
    t_start.record(stream)
    for _ in range(args.steps):
        launches += step()
    t_end.record(stream)
    torch.cuda.synchronize()
    used = M.lib().moe_launch_events_used()
    M.lib().moe_set_launch_events(None, 0)
    clocks = sampler.stop()
    if int(o["err"].item()) != 0:   # a timed region with device errors measures nothing
        raise SystemExit(f"device error bits {int(o['err'].item())} in the timed region")
    ms = t_start.elapsed_time(t_end) / args.steps

    Mrows = inp["M"]
    fwd_f, bwd_f = useful_flops(w, Mrows)
    value = (fwd_f + bwd_f) / (ms * 1e-3) / 1e12
    peaks = load_peaks()
    region_s = ms * args.steps * 1e-3

    # per-kernel durations
    dur = {nm: [] for nm in names}
    for i in range(used // 2):
        dur[names[i % per]].append(evs[2 * i].elapsed_time(evs[2 * i + 1]))
    work = kernel_work(w, Mrows, inp["E_ne"])
    kern = {}
    for nm in names:
        if not dur[nm]:
            continue
        avg = sum(dur[nm]) / len(dur[nm])
        rec = {"ms": round(avg, 4), "share": None}
        if nm in work:
            fl, by = work[nm]
            rec["tflops"] = round(fl / (avg * 1e-3) / 1e12, 1)
            rec["gbs"] = round(by / (avg * 1e-3) / 1e9, 1)
        kern[nm] = rec
    tot = sum(r["ms"] for r in kern.values())
    for r in kern.values():
        r["share"] = round(r["ms"] / tot, 4) if tot else None
    gemms = [nm for nm in kern if nm in work]
    dom = max(gemms, key=lambda nm: kern[nm]["ms"])
    fl, by = work[dom]
    t_dom = kern[dom]["ms"] * 1e-3
    fp8 = w.mxfp8 and (dom == "fc2" or (w.backward and dom in KERNELS_BWD))
    roof = roofline(dom, fl, by, t_dom, peaks, fp8, region_s)
    roof["traffic"] = ncu_traffic(dom, w)

    # the same step captured once as a CUDA graph and replayed (the pages'
    # benchmark times graph replays); the whole path is capturable
    graph = time_graph(step, max(args.steps, 20), fwd_f + bwd_f)

    # end to end through the public API with host buffers
    e2e_steps = args.e2e_steps if args.e2e_steps else max(args.steps, 30)
    e2e = run_e2e(w, inp, o, step, e2e_steps, fwd_f + bwd_f)

    if int(o["err"].item()) != 0:   # the graph and end-to-end legs share the error word
        raise SystemExit(f"device error bits {int(o['err'].item())} after the graph / e2e legs")

    # fused against unfused epilogues, and the rows built after the hot path
    # (outside the timed region; a side leg that fails is reported in the
    # line instead of costing it)
    def side(f, *a):
        try:
            return f(*a)
        except Exception as e:  # noqa: BLE001
            return {"error": f"{type(e).__name__}: {e}"[:300]}
    fusion = None
    if w.routing == "identity" and not w.mxfp8 and w.backward and not args.no_fusion_control:
        fusion = side(fusion_control, w, inp, o)
    if w.mxfp8 and w.backward and not args.no_fusion_control:
        fusion = side(mx_fusion_control, w, inp, o)
    extra = None if args.no_next_rows else side(next_rows, w, inp, o, peaks)

    cpu = None
    if not args.no_cpu_baseline:
        v, dt = time_oracle(w, args.cpu_rows)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{args.cpu_rows} rows of expert 0, float64 "
                         f"{('fwd (MXFP8 FC2)' if w.mxfp8 else 'fwd') if not w.backward else 'fwd+bwd'}"
                         f"{' MXFP8' if w.mxfp8 and w.backward else ''} ({dt:.1f} s)"}

    side_err = int(o["err"].item())
    if side_err != 0:
        # a side leg raised a device error bit: its numbers are dropped
        bad = {"error": f"device error bits {side_err} in a side leg"}
        fusion = bad if fusion is not None else None
        extra = bad if extra is not None else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3/e8m0 block-scaled (FC1 bf16)" if w.mxfp8 else "bf16",
        "data": "synthetic",
        "pct_of_bf16_peak": round(100 * value / peaks["bf16_tflops"], 2),
        "config": {"workload": w.name, "E": w.E, "T": w.T, "top_k": w.k, "d": w.d, "n": w.n,
                   "act": w.act, "rows": Mrows, "nonempty_experts": inp["E_ne"],
                   "step": step_description(w),
                   "l2": "inputs larger than L2 (no flush)", "parallelism": "none (1 GPU)",
                   "timed_region_s": round(region_s, 3)},
        "roofline": roof, "kernels": kern, "graph": graph, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks, "gpu_launches": launches,
    }
    if fusion is not None:
        line["fusion_control"] = fusion
    if extra is not None:
        line["next_rows"] = extra
    print(json.dumps(line), flush=True)
    return 0


def fusion_control(w, inp, o, reps=20):
    """Fused against unfused on the same GEMM kernels: FC1 + activation in
    one launch (writing H and A) against the plain grouped GEMM writing H
    and a separate activation pass; FC2-dgrad + dActivation against the
    plain dgrad GEMM writing dA and a separate derivative pass.  The pages
    compare their fused kernels with an unfused path the same way ([CuTe]
    "공개된 근거에서 확인되는 점": forward GLU about 1.2-1.3x, dSwiGLU 2.09x and
    dGeGLU 2.22x on GB300, E=8, 4096 tokens per expert, K=8192, N=4096, CUDA
    graph replay); their unfused baseline also uses other GEMM kernels, so
    only the fusion itself is compared here.  Each launch is timed with its
    own events, interleaved over ``reps`` rounds."""
    import torch
    import dropless_grouped_gemm_gb300 as M
    act, Mc = w.act, w.M_cap
    bf = torch.bfloat16
    dev = inp["x_perm"].device
    h_u = torch.empty((Mc, w.n1), dtype=bf, device=dev)
    a_u = torch.empty((Mc, w.n), dtype=bf, device=dev)
    da_u = torch.empty((Mc, w.n), dtype=bf, device=dev)
    dh_u = torch.empty((Mc, w.n1), dtype=bf, device=dev)
    x, dy, off, W1, W2 = inp["x_perm"], inp["dy_perm"], inp["offsets"], inp["W1"], inp["W2"]

    def round_():
        M.grouped_mlp_fwd(x, off, W1, W2, act, save_h=True, h_saved=o["h"], a=o["a"],
                          y_perm=o["y_perm"], err=o["err"])                       # 2 launches
        M.grouped_gemm(x, off, W1, "kn", out=h_u, err=o["err"])                   # 1
        M.activation(h_u, off, act, a=a_u)                                       # 1
        M.grouped_mlp_bwd(x, o["h"], o["a"], dy, off, W1, W2, act, dh=o["dh"],
                          dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"], err=o["err"])  # 4
        M.grouped_gemm(dy, off, W2, "nk", out=da_u, err=o["err"])                 # 1
        M.activation_bwd(o["h"], da_u, off, act, dh=dh_u)                        # 1
    avg = _launch_rounds(round_, 10, reps)
    if avg is None or int(o["err"].item()) != 0:
        return None
    fused_f, unf_f = avg[0], avg[2] + avg[3]
    fused_b, unf_b = avg[4], avg[8] + avg[9]
    return {"fwd": {"fused_ms": round(fused_f, 4), "unfused_ms": round(unf_f, 4),
                    "gemm_ms": round(avg[2], 4), "act_ms": round(avg[3], 4),
                    "speedup": round(unf_f / fused_f, 3)},
            "bwd": {"fused_ms": round(fused_b, 4), "unfused_ms": round(unf_b, 4),
                    "gemm_ms": round(avg[8], 4), "dact_ms": round(avg[9], 4),
                    "speedup": round(unf_b / fused_b, 3)},
            "reps": reps,
            "what": "same GEMM kernels; unfused = GEMM storing H (dA) + separate "
                    "activation (derivative) pass"}


def mx_fusion_control(w, inp, o, reps=20):
    """GroupGemm + dActivation + Quantize/Transpose against its unfused
    control: the MXFP8 backward with dH quantised in FC2-dgrad's epilogue
    (7 launches) and with FC2-dgrad storing dH alone and a separate tiled
    quantiser pass (8 launches), interleaved over ``reps`` rounds on the
    step's own operands, each launch timed by its own events; the results
    of the two are identical (tested)."""
    import dropless_grouped_gemm_gb300 as M
    if w.routing == "identity":
        x, dy, off = inp["x_perm"], inp["dy_perm"], inp["offsets"]
    else:
        x, dy, off = o["x_perm"], o["dy_perm"], o["route"]["offsets"]
    mx, mb = o["mx"], o["mxb"]
    ops = dict(a_qT=mx["a_qT"], a_sT=mx["a_sT"], w2_q=mb["w2_q"], w2_s=mb["w2_s"],
               w1_q=mb["w1_q"], w1_s=mb["w1_s"])

    def call(sep):
        M.grouped_mlp_bwd_mx(x, o["h"], dy, off, ops, w.act, dh=o["dh"], dx_perm=o["dx_perm"],
                             dW1=o["dW1"], dW2=o["dW2"], err=o["err"], workspace=mb["ws"],
                             separate_dh_quant=sep)
    def round_():
        call(False)
        call(True)
    avg = _launch_rounds(round_, 15, reps)
    if avg is None or int(o["err"].item()) != 0:
        return None
    fused = avg[3]                       # FC2-dgrad + dAct + Quantize/Transpose
    unf_gemm, unf_q = avg[7 + 3], avg[7 + 4]
    return {"bwd_dh": {"fused_ms": round(fused, 4), "unfused_ms": round(unf_gemm + unf_q, 4),
                       "gemm_ms": round(unf_gemm, 4), "quantize_ms": round(unf_q, 4),
                       "speedup": round((unf_gemm + unf_q) / fused, 3)},
            "fused_backward_ms": round(sum(avg[:7]), 4),
            "unfused_backward_ms": round(sum(avg[7:]), 4),
            "reps": reps,
            "what": "MXFP8 backward: FC2-dgrad + dAct with dH's MXFP8 copies written by its "
                    "epilogue, against FC2-dgrad + dAct storing dH and a separate tiled quantiser"}


def _launch_rounds(round_, per, reps):
    """Average duration (ms) of each of the ``per`` library launches (or
    calls) that ``round_`` makes, from the events the library records
    around them, over ``reps`` rounds after two untimed ones; None when the
    events do not add up or the error word is set."""
    import ctypes
    import torch
    import dropless_grouped_gemm_gb300 as M
    stream = torch.cuda.current_stream()
    for _ in range(2):
        round_()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * per * reps)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    handles = (ctypes.c_void_p * len(evs))(*[e.cuda_event for e in evs])
    M.lib().moe_set_launch_events(handles, len(evs))
    for _ in range(reps):
        round_()
    torch.cuda.synchronize()
    used = M.lib().moe_launch_events_used()
    M.lib().moe_set_launch_events(None, 0)
    if used != len(evs):
        return None
    t = [[evs[2 * (r * per + i)].elapsed_time(evs[2 * (r * per + i) + 1]) for r in range(reps)]
         for i in range(per)]
    return [sum(v) / len(v) for v in t]


def next_rows(w, inp, o, peaks, reps=20):
    """The rows built after the hot path, timed on the step's own operands
    outside the timed region, each launch between its own events:
    - bf16 training layers (identity routing): the NVFP4 statistics fused
      into the epilogues ([TE] "다음 단계: NVFP4, GEMM 융합 양자화, A2A 오버랩"):
      FC1 raising max|A| and FC2-dgrad raising the amax of the transposed
      16-point Hadamard-rotated dH, against the same launches without them;
    - MXFP8 training layers (identity routing): GroupGemm + Quantize, the
      block-scaled FC2 and FC1-dgrad also writing the MXFP8 copy of their
      bf16 output, against the same launches without it;
    - routed layers: the device router (top-k and softmax of the logits),
      the routing layout from its indices, and the router fused into the
      layout's first pass, from the workload's logits; the fused and the
      separate results are compared for identity."""
    import torch
    import dropless_grouped_gemm_gb300 as M
    act = w.act
    dev = o["err"].device
    if w.routing == "identity" and w.backward and not w.mxfp8:
        x, dy, off, W1, W2 = inp["x_perm"], inp["dy_perm"], inp["offsets"], inp["W1"], inp["W2"]
        amax_a = torch.zeros(1, dtype=torch.float32, device=dev)
        amax_dh = torch.zeros(1, dtype=torch.float32, device=dev)

        def round_():
            for am in (None, amax_a):                                           # 2 + 2
                M.grouped_mlp_fwd(x, off, W1, W2, act, save_h=True, h_saved=o["h"], a=o["a"],
                                  y_perm=o["y_perm"], err=o["err"], amax=am)
            for am in (None, amax_dh):                                          # 4 + 4
                M.grouped_mlp_bwd(x, o["h"], o["a"], dy, off, W1, W2, act, dh=o["dh"],
                                  dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"], err=o["err"],
                                  amax=am)
        avg = _launch_rounds(round_, 12, reps)
        if avg is None or int(o["err"].item()) != 0:
            return None
        fc1, fc1_s, dg, dg_s = avg[0], avg[2], avg[4], avg[8]
        return {"nvfp4_statistics": {
            "fc1_ms": round(fc1, 4), "fc1_with_amax_a_ms": round(fc1_s, 4),
            "fc1_overhead": round(fc1_s / fc1 - 1, 4),
            "fc2_dgrad_dact_ms": round(dg, 4), "fc2_dgrad_dact_with_amax_dh_ms": round(dg_s, 4),
            "fc2_dgrad_dact_overhead": round(dg_s / dg - 1, 4),
            "amax_a": float(amax_a.item()), "amax_dh": float(amax_dh.item()),
            "what": "max|A| in FC1's epilogue; amax of the transposed 16-point Hadamard-rotated "
                    "dH in FC2-dgrad's epilogue (one atomic maximum per warp)"},
            "reps": reps}
    if w.routing == "identity" and w.backward and w.mxfp8:
        x, dy, off, W1, W2 = inp["x_perm"], inp["dy_perm"], inp["offsets"], inp["W1"], inp["W2"]
        Mc, d = w.M_cap, w.d
        u8 = torch.uint8
        mx, mb = o["mx"], o["mxb"]
        mxq = dict(mx, y_q=torch.empty((Mc, d), dtype=u8, device=dev),
                   y_s=torch.empty((Mc, d // 32), dtype=u8, device=dev))
        ops = dict(a_qT=mx["a_qT"], a_sT=mx["a_sT"], w2_q=mb["w2_q"], w2_s=mb["w2_s"],
                   w1_q=mb["w1_q"], w1_s=mb["w1_s"])
        opsq = dict(ops, dx_q=torch.empty((Mc, d), dtype=u8, device=dev),
                    dx_s=torch.empty((Mc, d // 32), dtype=u8, device=dev))

        def round_():
            for m_ in (mx, mxq):                                                # 2 + 2
                M.grouped_mlp_fwd(x, off, W1, W2, act, save_h=True, h_saved=o["h"], a=o["a"],
                                  y_perm=o["y_perm"], err=o["err"], mx=m_)
            for p_ in (ops, opsq):                                              # 7 + 7
                M.grouped_mlp_bwd_mx(x, o["h"], dy, off, p_, act, dh=o["dh"],
                                     dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"],
                                     err=o["err"], workspace=mb["ws"])
        avg = _launch_rounds(round_, 18, reps)
        if avg is None or int(o["err"].item()) != 0:
            return None
        fc2, fc2_q, dgr, dgr_q = avg[1], avg[3], avg[4 + 5], avg[11 + 5]
        return {"group_gemm_quantize": {
            "fc2_ms": round(fc2, 4), "fc2_with_y_mxfp8_ms": round(fc2_q, 4),
            "fc2_overhead": round(fc2_q / fc2 - 1, 4),
            "fc1_dgrad_ms": round(dgr, 4), "fc1_dgrad_with_dx_mxfp8_ms": round(dgr_q, 4),
            "fc1_dgrad_overhead": round(dgr_q / dgr - 1, 4),
            "what": "block-scaled FC2 (FC1-dgrad) writing Y (dX) as bf16 and as row-wise "
                    "E4M3 codes with E8M0 scales from the same epilogue"},
            "reps": reps}
    if w.routing != "identity":
        T, k, E = w.T, w.k, w.E
        lg = torch.from_numpy(WL.logits(w.cfg_id, T, E, w.zipf_s, w.empty_expert)).to(dev)
        ws = o["ws"]

        def lay():
            return {nm: torch.empty_like(v) for nm, v in o["route"].items() if nm != "err"}
        out_sep, out_fused = lay(), lay()
        out_fused["topk_idx"] = torch.empty((T, k), dtype=torch.int32, device=dev)
        out_fused["probs"] = torch.empty((T, k), dtype=torch.float32, device=dev)
        calls = {
            "router_topk": lambda: M.router_topk(lg, k),
            "route_offsets": lambda: M.route_offsets(inp["topk_idx"], E, w.align, w.M_cap,
                                                     err=o["err"], out=out_sep, workspace=ws),
            "router_then_layout": lambda: M.route_offsets(M.router_topk(lg, k)[0], E, w.align,
                                                          w.M_cap, err=o["err"], out=out_sep,
                                                          workspace=ws),
            "route_logits_fused": lambda: M.route_logits(lg, k, w.align, w.M_cap, err=o["err"],
                                                         out=out_fused, workspace=ws),
        }
        # each captured as a CUDA graph and replayed: GPU time, without the
        # host's cost of issuing the calls
        ms = {nm: time_graph(f, reps, 0.0)["ms_per_step"] for nm, f in calls.items()}
        idx, probs = M.router_topk(lg, k)
        sep = M.route_offsets(idx, E, w.align, w.M_cap, workspace=ws)
        fused = M.route_logits(lg, k, w.align, w.M_cap, workspace=ws)
        torch.cuda.synchronize()
        same = all(torch.equal(fused[nm], sep[nm]) for nm in
                   ("counts", "offsets", "row_of_pair", "pair_of_row")) and \
            torch.equal(fused["topk_idx"], idx) and torch.equal(fused["probs"], probs) and \
            torch.equal(idx, inp["topk_idx"])
        lg_bytes = T * E * 4
        return {"router": {
            "router_topk_ms": ms["router_topk"],
            "route_offsets_ms": ms["route_offsets"],
            "router_then_layout_ms": ms["router_then_layout"],
            "route_logits_fused_ms": ms["route_logits_fused"],
            "fused_speedup": round(ms["router_then_layout"] / ms["route_logits_fused"], 3),
            "router_logits_gbs": round(lg_bytes / ms["router_topk"] / 1e6, 1),
            "router_frac_of_hbm": round(lg_bytes / ms["router_topk"] / 1e6 / peaks["hbm_gbs"], 4),
            "identical": bool(same),
            "what": "T x E float32 logits -> top-k indices and softmax weights (router_topk); "
                    "the routing layout from given indices (route_offsets); the two in sequence; "
                    "the router fused into the layout's first pass (route_logits); each call "
                    "captured as a CUDA graph, median of the replays"},
            "reps": reps}
    return None


def step_description(w):
    if w.mxfp8 and w.backward:
        core = ("W2 MXFP8 quantise + fwd (FC1 + MX epilogue, block-scaled FC2) + weight "
                "quantise + MXFP8 bwd (grouped_mlp_bwd_mx)")
        return core if w.routing == "identity" else (
            "route + permute + " + core.replace(" + weight", " + combine + weight") +
            " (+ router grad)")
    if w.routing == "identity":
        return "grouped_mlp_fwd + grouped_mlp_bwd"
    if w.mxfp8:
        return ("route + permute + W2 MXFP8 quantise + fwd (FC1 + MX epilogue, block-scaled FC2) "
                "+ combine")
    if not w.backward:
        return "route + permute + fwd + combine"
    if w.gather:
        return ("route + fwd reading x through the routing map (grouped_mlp_fwd_gather) + "
                "combine + bwd with the router gradient inside the expert MLP, reading x and dO "
                "through the routing map (grouped_mlp_bwd_routed_gather + router_grad_rows) + "
                "combine backward")
    return ("route + permute + fwd + combine + bwd with the router gradient inside the expert "
            "MLP (grouped_mlp_bwd_routed + router_grad_rows) + combine backward")


def time_graph(step, replays, flops):
    """One step captured as a CUDA graph and replayed: each of ``replays``
    (at least 20) replays timed by its own pair of CUDA events; the median
    replay is reported (the pages time graph replays)."""
    import torch
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    cur.wait_stream(side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(replays)]
    for s, e in evs:
        s.record()
        g.replay()
        e.record()
    torch.cuda.synchronize()
    t = sorted(s.elapsed_time(e) for s, e in evs)
    ms = statistics.median(t)
    del g
    return {"ms_per_step": round(ms, 4), "value": round(flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "replays": replays, "statistic": "median",
            "min_ms": round(t[0], 4), "max_ms": round(t[-1], 4)}


def run_e2e(w, inp, o, step, steps, flops):
    """Same metric through the public API from pinned host buffers.  Every
    step copies its inputs host->device and reads its results back to the
    host, as an input pipeline would: the inputs of step i+1 are copied on
    one stream while step i computes, and step i's results are read back on
    another, with three device input sets and three result sets (with two,
    step i+1 waited for step i-1's results to be read back).  A training
    step's results are the input gradient and both weight gradients; a
    forward step's is the layer output.  The timed region runs from the
    first input copy to the last result read."""
    import torch
    if w.routing == "identity":
        names_in = ["x_perm", "dy_perm", "offsets"]
        out_names = ["dx_perm", "dW1", "dW2"]
    elif not w.backward:
        names_in = ["x", "topk_idx", "probs"]
        out_names = ["out"]
    else:
        names_in = ["x", "dO", "topk_idx", "probs"]
        out_names = ["dx", "dW1", "dW2", "dprobs"]
    host = {nm: torch.empty(inp[nm].shape, dtype=inp[nm].dtype, pin_memory=True)
            for nm in names_in}
    for nm in names_in:
        host[nm].copy_(inp[nm])
    out_host = {nm: torch.empty(o[nm].shape, dtype=o[nm].dtype, pin_memory=True)
                for nm in out_names}
    h2d = sum(host[nm].numel() * host[nm].element_size() for nm in names_in)
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    # NSET input sets / result buffers; weights and intermediates shared
    NSET = 3
    sets, outs, steps_fn = [], [], []
    for i in range(NSET):
        ins = dict(inp)
        if i > 0:
            for nm in names_in:
                ins[nm] = torch.empty_like(inp[nm])
        oo = dict(o)
        if i > 0:
            for nm in out_names:
                oo[nm] = torch.empty_like(o[nm])
        sets.append(ins)
        outs.append(oo)
        steps_fn.append(make_step(w, ins, oo))
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event() for _ in range(NSET)]
    freed = [torch.cuda.Event() for _ in range(NSET)]   # compute done with the set / result
    read = [torch.cuda.Event() for _ in range(NSET)]    # result copied out

    def h2d_copy(i):
        k = i % NSET
        with torch.cuda.stream(up):
            if i >= NSET:
                up.wait_event(freed[k])
            for nm in names_in:
                sets[k][nm].copy_(host[nm], non_blocking=True)
            ready[k].record(up)

    def run(n):
        h2d_copy(0)
        for i in range(n):
            k = i % NSET
            if i + 1 < n:
                h2d_copy(i + 1)
            comp.wait_event(ready[k])
            if i >= NSET:
                comp.wait_event(read[k])            # result buffer k copied out
            steps_fn[k]()
            freed[k].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(freed[k])
                for nm in out_names:
                    out_host[nm].copy_(outs[k][nm], non_blocking=True)
                read[k].record(down)

    run(NSET)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(up)
    run(steps)
    down.wait_stream(comp)
    down.wait_stream(up)
    e.record(down)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "read_back": out_names,
            "pipelined": "inputs of step i+1 copied during step i; three input and result sets"}


if __name__ == "__main__":
    sys.exit(main())
