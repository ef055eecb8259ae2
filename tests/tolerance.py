"""Error metric of the parity tests.

Per element e_i = |g_i - r_i| / max(|r_i|, s), where s is the RMS of the
reference r over the whole tensor: relative error, with a floor that keeps
near-zero outputs (y crosses zero often) from dominating. The gate is
max_i e_i <= 1e-4 for fp32 I/O and <= 5e-3 for bf16 I/O (fp32 state and
accumulation in both). Rounding y to bf16 alone contributes up to 2^-9
(about 1.95e-3) relative.
"""
import numpy as np

TOL = {"float32": 1e-4, "bfloat16": 5e-3}


def max_rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    s = float(np.sqrt(np.mean(ref * ref)))
    floor = np.maximum(np.abs(ref), s if s > 0 else 1e-30)
    return float(np.max(np.abs(got - ref) / floor))


def report(got, ref) -> dict:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nref = float(np.linalg.norm(ref))
    return {"max_rel": max_rel_err(got, ref),
            "normwise": float(np.linalg.norm(got - ref)) / nref if nref > 0 else 0.0,
            "max_abs_over_max": float(np.max(np.abs(got - ref))) / max(float(np.max(np.abs(ref))), 1e-300)
            if ref.size else 0.0}
