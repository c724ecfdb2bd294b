"""Shared test helpers (no method arithmetic here)."""
import numpy as np
import torch

# Tolerance for floating-point results: max|err| <= TOL * RMS(ref) per output
# tensor.  For bf16 outputs the storage resolution at each element is added:
# the GPU rounds its float32 result and the oracle its float64 result to
# bf16 once each, so two correct results may sit one bf16 step apart, and a
# step at a tail element of a heavy-tailed tensor (|ref| ~ 10 RMS) is larger
# than TOL * RMS by itself.  BF16_RTOL = 2^-7 is one bf16 step relative to
# |ref| (for |ref| just above a power of two; at most two steps just below).
TOL = 2e-2
BF16_RTOL = 2.0 ** -7


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_rms_close(got, ref, name, tol=TOL, rtol=BF16_RTOL):
    """max_i (|got_i - ref_i| - rtol |ref_i|) <= tol * RMS(ref); pass rtol=0
    for float32 outputs."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    rms = float(np.sqrt((ref ** 2).mean()))
    excess = np.abs(got - ref) - rtol * np.abs(ref)
    i = int(np.argmax(excess))
    err = float(excess.reshape(-1)[i])
    assert err <= tol * rms + 1e-30, (
        f"{name}: max(|err| - {rtol:.4g}|ref|) {err:.3e} > {tol} * RMS {rms:.3e} "
        f"(at flat index {i}: got {got.reshape(-1)[i]:.6g}, ref {ref.reshape(-1)[i]:.6g})")


def cuda_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, np.int32))).cuda()
