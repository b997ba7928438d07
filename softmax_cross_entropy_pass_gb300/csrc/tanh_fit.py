"""Coefficients of the polynomial parts of the stream kernel's softcap tanh.

The kernel evaluates tanh(u) = u * (1 + sum_k c_k (u^2)^k) in fp32 with
Horner's rule on two ranges:
  narrow: |u| < 0.3, k = 1..3 (the range of ordinary logits under a cap of
          30: |x| < 9);
  wide:   |u| < 0.8, k = 1..6;
and for larger |u| the identity tanh|u| = 1 - 2 / (1 + e^(2|u|)). Each set
of c_k comes from a least-squares fit of (tanh(u) / u - 1) on 600 Chebyshev
nodes of w = u^2 in [0, u0^2] (a plain linear fit in the monomials of w,
with the constant term fixed at 1). Evaluated in fp32 the narrow polynomial
stays within about 1.2 units in the last place of tanh, the wide one within
2.5. Run this file to print the constants that ce_device.cuh holds
(kTanhN1..kTanhN3 and kTanhC1..kTanhC6)."""
import numpy as np

NARROW_U0, NARROW_DEGREE = 0.3, 3
U0, DEGREE = 0.8, 6
NODES = 600


def coefficients(u0: float = U0, degree: int = DEGREE) -> np.ndarray:
    """c_1 .. c_degree as fp32."""
    k = np.arange(NODES)
    w = (u0 ** 2) * 0.5 * (1.0 - np.cos(np.pi * (k + 0.5) / NODES))
    u = np.sqrt(w)
    f = np.tanh(u) / u
    A = np.vander(w, degree + 1, increasing=True)[:, 1:]
    c, *_ = np.linalg.lstsq(A, f - 1.0, rcond=None)
    return c.astype(np.float32)


def narrow_coefficients() -> np.ndarray:
    return coefficients(NARROW_U0, NARROW_DEGREE)


if __name__ == "__main__":
    for i, c in enumerate(narrow_coefficients(), start=1):
        print(f"kTanhN{i} = {float(c)!r}f")
    for i, c in enumerate(coefficients(), start=1):
        print(f"kTanhC{i} = {float(c)!r}f")
