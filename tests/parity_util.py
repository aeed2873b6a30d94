"""Shared tolerance checks for the GPU-vs-oracle parity tests.

Floating-point bar: relative L2 error <= 1e-2 over the compared tensor and
max |err| <= 5e-2 * RMS(reference) (bf16 inputs, fp32 accumulation).
"""
import numpy as np

REL_L2 = 1e-2
MAX_REL_RMS = 5e-2


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    mx = float(np.abs(err).max()) if err.size else 0.0
    return float(rel), mx, rms


def assert_parity(got, ref, what=""):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    rel, mx, rms = errors(got, ref)
    assert rel <= REL_L2 and mx <= MAX_REL_RMS * rms, (
        f"{what}: rel_l2={rel:.3e} (<= {REL_L2}), max_err={mx:.3e} (<= {MAX_REL_RMS}*rms={MAX_REL_RMS * rms:.3e})")
    return rel, mx, rms
