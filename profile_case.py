"""Run one seeded case of the path a fixed number of times (for profilers).

    python profile_case.py --workload NAME
        [--rows-per-expert R | --tokens T] [--what fwd|bwd|step] [--reps N]

Inputs come from the ``workloads`` generator; shapes other than the row /
token count are the workload's.  ``fwd`` launches FC1+act and FC2 per rep,
``bwd`` one forward then the four backward GEMMs per rep, ``step`` the whole
pass that bench.py times.  Prints the launch order it used.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch
    import workloads as WL
    import bench as BE
    from dropless_grouped_gemm_gb300 import build as B
    import dropless_grouped_gemm_gb300 as M

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=BE.DEFAULT_WORKLOAD, choices=sorted(WL.WORKLOADS))
    ap.add_argument("--rows-per-expert", type=int, default=None)
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None,
                    help="fewer experts, for captures that must stay small (routed workloads: "
                         "the same tokens over fewer experts; identity-routed ones: the first "
                         "E experts with their rows, every launch's work scaled by E / E_full)")
    ap.add_argument("--what", choices=["fwd", "bwd", "step"], default="step")
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    B.build()
    M.lib()
    w = WL.WORKLOADS[a.workload]
    if a.rows_per_expert is not None and w.routing == "identity":
        w = WL.scaled(w, T=w.E * a.rows_per_expert)
    if a.tokens is not None and w.routing != "identity":
        w = WL.scaled(w, T=a.tokens)
    if a.experts is not None and w.routing != "identity":
        w = WL.scaled(w, E=a.experts, k=min(w.k, a.experts))
    if a.experts is not None and w.routing == "identity":
        w = WL.scaled(w, E=a.experts, T=a.experts * (w.T // w.E))
    inp, o = BE.make_inputs(w, "cuda")
    step = BE.make_step(w, inp, o)
    if a.what == "step":
        order = BE.event_names(w)
        for _ in range(a.reps):
            step()
    else:
        if w.routing != "identity":
            raise SystemExit("fwd/bwd cases use identity-routed workloads")
        x, off = inp["x_perm"], inp["offsets"]

        def fwd():
            M.grouped_mlp_fwd(x, off, inp["W1"], inp["W2"], w.act, save_h=True, h_saved=o["h"],
                              a=o["a"], y_perm=o["y_perm"], err=o["err"])

        def bwd():
            M.grouped_mlp_bwd(x, o["h"], o["a"], inp["dy_perm"], off, inp["W1"], inp["W2"], w.act,
                              dh=o["dh"], dx_perm=o["dx_perm"], dW1=o["dW1"], dW2=o["dW2"],
                              err=o["err"])
        if a.what == "fwd":
            order = BE.KERNELS_FWD
            for _ in range(a.reps):
                fwd()
        else:
            fwd()
            order = BE.KERNELS_FWD + BE.KERNELS_BWD * a.reps
            for _ in range(a.reps):
                bwd()
    torch.cuda.synchronize()
    e = int(o["err"].item())
    print(f"workload={w.name} T={w.T} what={a.what} reps={a.reps} err={e} launch order per rep: "
          f"{' '.join(order)}")
    return 1 if e else 0


if __name__ == "__main__":
    sys.exit(main())
