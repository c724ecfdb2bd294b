"""Shared test helpers (no method arithmetic here)."""
import numpy as np
import torch

# Tolerance for floating-point results: max|err| <= TOL * RMS(ref) per output
# tensor, where ref is the oracle's exact value (float64) before the storage
# rounding (the oracle's round_out=False).  A bf16 output adds the cost of its
# one storage rounding: round-to-nearest moves a value by at most half a bf16
# step, 2^-8 of its magnitude, so the check is
#     max_i (|got_i - ref_i| - HALF_STEP |ref_i|) <= TOL * RMS(ref).
# float32 outputs pass rtol=0.
TOL = 2e-2
HALF_STEP = 2.0 ** -8

# (name, max|err|/RMS, max excess/RMS) of every comparison in this process,
# printed in the session's terminal summary
RECORDS = []


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_rms_close(got, ref, name, tol=TOL, rtol=HALF_STEP):
    """max_i (|got_i - ref_i| - rtol |ref_i|) <= tol * RMS(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert np.isfinite(ref).all(), f"{name}: non-finite reference values"
    rms = float(np.sqrt((ref ** 2).mean()))
    diff = np.abs(got - ref)
    excess = diff - rtol * np.abs(ref)
    i = int(np.argmax(excess))
    err = float(excess.reshape(-1)[i])
    plain = float(diff.max()) / rms if rms > 0 else float(diff.max())
    RECORDS.append((name, plain, err / rms if rms > 0 else err))
    assert err <= tol * rms + 1e-30, (
        f"{name}: max(|err| - {rtol:.4g}|ref|) {err:.3e} > {tol} * RMS {rms:.3e} "
        f"(max|err|/RMS {plain:.3e}; at flat index {i}: got {got.reshape(-1)[i]:.6g}, "
        f"ref {ref.reshape(-1)[i]:.6g})")


def cuda_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()
