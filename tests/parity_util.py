"""Shared tolerance checks for the GPU-vs-oracle parity tests.

Floating-point bar (bf16 inputs, fp32 accumulation): relative L2 error <= 1e-2 over the
compared tensor, and max |err| <= 5e-2 * RMS(reference) for the kernel's arithmetic.
The result is then cast to the output dtype, which by itself moves each element by up
to half a unit in the last place (2^-8 |o| for bf16, 2^-24 |o| for fp32); that cast is
charged separately, element by element, so the max-error bar reads
    max(|err| - half_ulp(o_ref)) <= 5e-2 * RMS(o_ref).
(With bf16 outputs whose largest element is ~18 RMS, the cast alone already moves an
element by ~0.045 RMS, so the bar could not otherwise separate kernels.)
"""
import numpy as np

REL_L2 = 1e-2
MAX_REL_RMS = 5e-2
HALF_ULP = {"bf16": 2.0 ** -8, "f32": 2.0 ** -24}


def _fmt(dtype) -> str:
    s = str(dtype)
    return "bf16" if "bfloat16" in s or s == "bf16" else "f32"


def errors(got, ref, dtype="bf16"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    excess = err - HALF_ULP[_fmt(dtype)] * np.abs(ref)
    mx = float(excess.max()) if err.size else 0.0
    return float(rel), mx, rms


def raw_max_err(got, ref) -> float:
    """max |got - ref| with nothing charged for the output cast."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max()) if ref.size else 0.0


def assert_parity(got, ref, what="", dtype="bf16"):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    rel, mx, rms = errors(got, ref, dtype)
    if not (rel <= REL_L2 and mx <= MAX_REL_RMS * rms):
        raw = raw_max_err(got, ref)
        raise AssertionError(
            f"{what}: rel_l2={rel:.3e} (<= {REL_L2}), max_err-cast={mx:.3e} "
            f"(<= {MAX_REL_RMS}*rms={MAX_REL_RMS * rms:.3e}); raw max|err|={raw:.3e} = "
            f"{raw / rms if rms > 0 else float('inf'):.3e}*rms")
    return rel, mx, rms
