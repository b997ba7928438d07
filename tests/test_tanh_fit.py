"""The softcap tanh of the stream kernel and the fused-linear epilogue
(ce_device.cuh, softcap_fast / softcap_vec): both polynomials' constants are
the ones tanh_fit.py computes, and each polynomial, evaluated in fp32 the way
the kernel does (Horner with fused multiply-adds), stays within its bound of
fp64 tanh on its range (narrow |u| < 0.3: 1.5 units in the last place; wide
|u| < 0.8: 2.5). The third branch (the exponential identity) runs on the
hardware exponential and is covered by the GPU parity tests with softcap."""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "softmax_cross_entropy_pass_gb300", "csrc")


def _fit():
    spec = importlib.util.spec_from_file_location("tanh_fit", os.path.join(CSRC, "tanh_fit.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _header():
    return open(os.path.join(CSRC, "ce_device.cuh")).read()


def _header_constants(prefix: str, degree: int):
    """k<prefix>1 .. k<prefix><degree> as the header defines them (index k-1 holds c_k)."""
    found = dict(re.findall(rf"constexpr float k{prefix}(\d) = (-?\d+\.\d+(?:e-?\d+)?)f;", _header()))
    assert sorted(found) == [str(k) for k in range(1, degree + 1)]
    return [float(found[str(k)]) for k in range(1, degree + 1)]


def _header_edge(name: str) -> float:
    return float(re.search(rf"constexpr float {name} = (\d+\.\d+)f;", _header()).group(1))


def test_header_constants_are_the_fits():
    fit = _fit()
    assert np.array_equal(np.float32(_header_constants("TanhC", fit.DEGREE)), fit.coefficients())
    assert np.array_equal(np.float32(_header_constants("TanhN", fit.NARROW_DEGREE)), fit.narrow_coefficients())
    assert _header_edge("kTanhNarrowEdge") == fit.NARROW_U0
    assert _header_edge("kTanhPolyEdge") == fit.U0


def _max_ulp(c, u0):
    u = np.linspace(-u0, u0, 400001, dtype=np.float32)
    u = u[(u != 0) & (np.abs(u) < np.float32(u0))]
    w = (u * u).astype(np.float32)

    def fma(a, b, d):  # one rounding of a*b + d, as the kernel's fmaf
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(d)).astype(np.float32)

    p = np.full_like(w, c[-1])
    for ck in list(c[-2::-1]) + [np.float32(1.0)]:
        p = fma(p, w, ck)
    t = (u * p).astype(np.float32)
    ref = np.tanh(u.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return float(np.max(np.abs(t.astype(np.float64) - ref) / ulp))


@pytest.mark.parametrize("which,bound", [("narrow", 1.5), ("wide", 2.5)])
def test_polynomial_within_bound_in_fp32(which, bound):
    fit = _fit()
    if which == "narrow":
        c, u0 = fit.narrow_coefficients(), fit.NARROW_U0
    else:
        c, u0 = fit.coefficients(), fit.U0
    assert _max_ulp(c, u0) <= bound


def test_dropping_a_term_breaks_the_bound():
    """The ulp check is sharp enough to see a truncated polynomial."""
    fit = _fit()
    assert _max_ulp(fit.coefficients()[:-1], fit.U0) > 2.5
    assert _max_ulp(fit.narrow_coefficients()[:-1], fit.NARROW_U0) > 1.5
