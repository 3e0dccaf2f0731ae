"""Coefficients of the softplus polynomials of the vector kernels.

The kernels evaluate softplus(x) = max(x, 0) + log1p(e), e = exp(-|x|) in
(0, 1], with log1p(e) = e * g(e) and g a polynomial fitted to log1p(e)/e by
least squares on Chebyshev nodes of [0, 1] (degree 8 for fp32 I/O, degree 5
for bf16 I/O).  This script recomputes those coefficients and the relative
error of their fp32 Horner evaluation (one rounding per fused multiply-add),
so that the constants in csrc/ss_device.cuh can be checked or regenerated:

    python -m mamba_selective_scan_ss_gb300.softplus_fit
"""
from __future__ import annotations

import numpy as np


def fit(degree: int, nodes: int = 200) -> np.ndarray:
    """Least-squares coefficients (constant term first) of log1p(e)/e on [0, 1]."""
    k = np.arange(nodes)
    e = 0.5 + 0.5 * np.cos((2 * k + 1) * np.pi / (2 * nodes))
    g = np.log1p(e) / e
    coef, *_ = np.linalg.lstsq(np.vander(e, degree + 1, increasing=True), g, rcond=None)
    return coef


def eval_fp32(coef, e) -> np.ndarray:
    """e * g(e) in fp32 as the kernel does: Horner with fused multiply-adds."""
    c = np.asarray(coef, np.float32)
    e = np.asarray(e, np.float32)
    g = np.full_like(e, c[-1])
    for a in c[-2::-1]:
        g = (g.astype(np.float64) * e + np.float64(a)).astype(np.float32)
    return (e.astype(np.float64) * g).astype(np.float32)


def max_rel_error(coef) -> float:
    """Largest relative error of eval_fp32 against log1p over (0, 1], including
    e down to 2^-125 (softplus of very negative x)."""
    e = np.linspace(0.0, 1.0, 2_000_001)[1:].astype(np.float32)
    e = np.concatenate([e, np.float32(2.0) ** -np.arange(1, 126, 0.25).astype(np.float32)])
    ref = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(eval_fp32(coef, e) - ref) / ref))


if __name__ == "__main__":
    for deg in (8, 5):
        c = fit(deg).astype(np.float32)
        print(f"degree {deg}: max rel error {max_rel_error(c):.2e}")
        print("  highest degree first:", ", ".join(f"{float(a):.9g}f" for a in c[::-1]))
