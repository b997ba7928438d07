"""Coefficients of the polynomial part of the stream kernel's softcap tanh.

For |u| < 0.8 the kernel evaluates tanh(u) = u * (1 + sum_k c_k (u^2)^k),
k = 1..6, in fp32 with Horner's rule; for larger |u| it uses the identity
tanh|u| = 1 - 2 / (1 + e^(2|u|)). The c_k come from a least-squares fit of
(tanh(u) / u - 1) on 600 Chebyshev nodes of w = u^2 in [0, 0.64] (a plain
linear fit in the monomials of w, with the constant term fixed at 1). The
fit's fp64 relative error is below 4e-9; evaluated in fp32 it stays within
about 2 units in the last place. Run this file to print the constants that
`softcap_logit_fast` (ce_device.cuh) holds."""
import numpy as np

U0 = 0.8
DEGREE = 6
NODES = 600


def coefficients() -> np.ndarray:
    k = np.arange(NODES)
    w = (U0 ** 2) * 0.5 * (1.0 - np.cos(np.pi * (k + 0.5) / NODES))
    u = np.sqrt(w)
    f = np.tanh(u) / u
    A = np.vander(w, DEGREE + 1, increasing=True)[:, 1:]
    c, *_ = np.linalg.lstsq(A, f - 1.0, rcond=None)
    return c.astype(np.float32)


if __name__ == "__main__":
    for i, c in enumerate(coefficients(), start=1):
        print(f"c{i} = {float(c)!r}f")
