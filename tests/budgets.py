"""Acceptance rules against the FP64 oracle (host logic used by the tests).

The budgets are the deterministic package's absolute error budgets stated on
the FlashInfer page "perf(cake_dense_projection_gemm): restore the K1
weight-gradient routes that meet the deterministic package's absolute FP64
budgets" (PR body):

  * BF16 output: atol = rtol = 1e-2 with zero violating elements;
  * FP32 output: relative Frobenius error <= 5e-5 and max_abs <= 1e-3 * max|ref|.

Non-finite GPU values always count as violations.
"""
from __future__ import annotations

import numpy as np

BF16_ATOL = 1e-2
BF16_RTOL = 1e-2
F32_REL_FRO = 5e-5
F32_MAX_ABS_FRAC = 1e-3


def bf16_violations(got, ref) -> int:
    """Number of elements with |g - r| > atol + rtol * |r|, or g not finite."""
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    bad = ~np.isfinite(g) | (np.abs(g - r) > BF16_ATOL + BF16_RTOL * np.abs(r))
    return int(bad.sum())


def f32_errors(got, ref) -> tuple[float, float, float]:
    """(rel_fro, max_abs, max|ref|)."""
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    if not np.all(np.isfinite(g)):
        return float("inf"), float("inf"), float(np.abs(r).max(initial=0.0))
    d = g - r
    nr = float(np.sqrt((r * r).sum()))
    nd = float(np.sqrt((d * d).sum()))
    rel = nd / nr if nr > 0 else (0.0 if nd == 0 else float("inf"))
    return rel, float(np.abs(d).max(initial=0.0)), float(np.abs(r).max(initial=0.0))


def f32_within_budget(got, ref) -> bool:
    rel, mx, mref = f32_errors(got, ref)
    return rel <= F32_REL_FRO and mx <= F32_MAX_ABS_FRAC * mref


def check(got, ref, out_dtype: str) -> tuple[bool, str]:
    """Apply the budget for ``out_dtype`` ('bf16' or 'f32'); returns (ok, message)."""
    if out_dtype == "bf16":
        v = bf16_violations(got, ref)
        return v == 0, f"bf16 violations={v} of {np.asarray(ref).size}"
    rel, mx, mref = f32_errors(got, ref)
    ok = rel <= F32_REL_FRO and mx <= F32_MAX_ABS_FRAC * mref
    return ok, f"f32 rel_fro={rel:.3e} max_abs={mx:.3e} max|ref|={mref:.3e}"
