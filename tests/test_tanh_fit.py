"""The softcap tanh of the stream kernel (ce_device.cuh, tanh_fast): its
polynomial constants are the ones tanh_fit.py computes, and the polynomial,
evaluated in fp32 the way the kernel does (Horner with fused multiply-adds),
stays within 2.5 units in the last place of fp64 tanh on |u| < 0.8. The
other branch (the exponential identity) runs on the hardware exponential
and is covered by the GPU parity tests with softcap."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "softmax_cross_entropy_pass_gb300", "csrc")


def _fit():
    spec = importlib.util.spec_from_file_location("tanh_fit", os.path.join(CSRC, "tanh_fit.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _header_constants():
    text = open(os.path.join(CSRC, "ce_device.cuh")).read()
    body = text[text.index("__device__ inline float tanh_fast"):]
    body = body[:body.index("return a < 0.8f")]
    return [float(x) for x in re.findall(r"(-?\d+\.\d+(?:e-?\d+)?)f", body)]


def test_header_constants_are_the_fit():
    c = _fit().coefficients()
    got = _header_constants()
    # Horner order in the header: c6, c5, c4, c3, c2, c1, then 1, the clamp constants
    assert np.array_equal(np.float32(got[:6]), c[::-1])


def test_polynomial_within_two_and_a_half_ulp_in_fp32():
    c = _fit().coefficients()
    u = np.linspace(-0.8, 0.8, 400001, dtype=np.float32)
    u = u[u != 0]
    w = (u * u).astype(np.float32)

    def fma(a, b, d):  # one rounding of a*b + d, as the kernel's fmaf
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(d)).astype(np.float32)

    p = np.full_like(w, c[5])
    for ck in (c[4], c[3], c[2], c[1], c[0], np.float32(1.0)):
        p = fma(p, w, ck)
    t = (u * p).astype(np.float32)
    ref = np.tanh(u.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert float(np.max(np.abs(t.astype(np.float64) - ref) / ulp)) <= 2.5
