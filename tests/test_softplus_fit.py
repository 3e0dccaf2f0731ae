"""The softplus polynomials of the vector kernels, re-derived on the CPU.

dt = softplus(delta + bias) (task spec Этап 1 step 3) is evaluated in the
kernels as max(x, 0) + e*g(e), e = exp(-|x|), with g fitted to log1p(e)/e.
These tests re-fit g with numpy, check the constants written in the kernel
header against the fit, and bound the fp32 evaluation against log1p."""
import re
from pathlib import Path

import numpy as np
import pytest

from mamba_selective_scan_ss_gb300 import softplus_fit

HEADER = Path(__file__).resolve().parent.parent / "mamba_selective_scan_ss_gb300" / "csrc" / \
    "ss_device.cuh"


def header_coefficients(function: str) -> np.ndarray:
    """Coefficients of `function` in the header, constant term first."""
    text = HEADER.read_text()
    body = text[text.index(f"f2 {function}(f2 e)"):]
    body = body[:body.index("return")]
    vals = [float(v) for v in re.findall(r"splat\(([-0-9.e]+)f\)", body)]
    return np.array(vals[::-1])  # Horner starts from the highest degree


@pytest.mark.parametrize("function,degree,bound", [("log1p_unit2", 8, 2e-7),
                                                   ("log1p_unit2_d5", 5, 1e-5)])
def test_header_constants_are_the_fit(function, degree, bound):
    got = header_coefficients(function)
    assert got.size == degree + 1
    want = softplus_fit.fit(degree)
    np.testing.assert_allclose(got, want, rtol=2e-7, atol=2e-8)
    assert softplus_fit.max_rel_error(got) <= bound


def test_fit_is_the_least_squares_fit_of_log1p():
    # the fit reproduces log1p(e)/e at points off the nodes, and is stable in the
    # number of nodes (a property of the least-squares solution, not of the data)
    c8 = softplus_fit.fit(8)
    e = np.linspace(1e-6, 1.0, 1001)
    g = np.polynomial.polynomial.polyval(e, c8)
    assert np.max(np.abs(g - np.log1p(e) / e)) < 1e-7
    np.testing.assert_allclose(softplus_fit.fit(8, nodes=1000), c8, rtol=1e-6, atol=1e-9)
    # a mistake in the evaluation would show: dropping the last term costs 1e-3
    wrong = c8.copy()
    wrong[-1] = 0.0
    assert softplus_fit.max_rel_error(wrong) > 1e-4


def test_softplus_through_the_fit_matches_logaddexp():
    # the kernel's form max(x, 0) + e*g(e), e = exp(-|x|), against numpy's
    # log(1 + e^x) over the range dt's argument takes, for both polynomials
    x = np.linspace(-40, 40, 8001)
    e = np.exp(-np.abs(x)).astype(np.float32)
    ref = np.logaddexp(0.0, x)
    for function, bound in (("log1p_unit2", 2e-7), ("log1p_unit2_d5", 1e-5)):
        sp = np.maximum(x, 0) + softplus_fit.eval_fp32(header_coefficients(function), e)
        assert np.max(np.abs(sp - ref) / ref) < bound, function
