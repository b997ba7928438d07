"""Comparison helpers for the parity tests (CUDA path vs the fp64 oracle).

Tolerances (derived from the arithmetic; the reasoning is in the design
notes):
  * loss per row: 1e-5 relative (the floor 1e-6 absolute covers rows whose
    loss is ~0); reduced loss: 1e-6 relative.
  * bf16 / f16 gradient: |got - RNE(oracle)| <= max(1 ulp of RNE(oracle),
    2^-18 * T_ic * |s_i|), T_ic the sum of the magnitudes of the gradient's
    terms before they cancel: (1-eps) w_y p_ic + (1-eps) w_y [c = y]
    + (eps/V) p_ic W_all + (eps/V) w_c. fp32 gradient: 2^-18 * T_ic * |s_i|
    plus 2 fp32 ulps of the value.
  * dx_y: relative error <= 0.4%.
"""
from __future__ import annotations

import torch

LOSS_ROW_RTOL = 1e-5
LOSS_ROW_ATOL = 1e-6
LOSS_RED_RTOL = 1e-6
FLOOR = 2.0 ** -18
DXY_RTOL = 4e-3


def ulp_of(v: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Spacing of the representable values of ``dtype`` at |v| (v already
    representable in dtype), as float64."""
    a = v.abs().to(dtype)
    if dtype == torch.float32:
        up = torch.nextafter(a, torch.full_like(a, float("inf")))
    else:
        bits = a.view(torch.int16).to(torch.int32) + 1
        up = bits.to(torch.int16).view(dtype)
    return (up.double() - a.double()).abs()


def rne(v64: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return v64.to(torch.float32).to(dtype)


def magnitude_T(x: torch.Tensor, target: torch.Tensor, stats64: torch.Tensor, weight, eps: float,
                w_all: float, scale: torch.Tensor, softcap: float = 0.0, z_loss: float = 0.0) -> torch.Tensor:
    """|s_i| * T_ic for every element, in fp64 (rows not valid: 0). With a
    softcap the terms are those of the capped logits times dz/dx, and times
    max(1, |z| / 8) for the fp32 rounding of z itself; z-loss adds its
    |2 lambda LSE p| term. Runs on the device of ``x`` (every other tensor
    is moved there)."""
    dev = x.device
    xd = x.double()
    deriv = None
    if softcap > 0:
        xd = softcap * torch.tanh(xd / softcap)
        deriv = 1.0 - (xd / softcap) ** 2
    R, V = xd.shape
    st = stats64.to(dev, torch.float64)
    m, s, xy = st[:, 0:1], st[:, 1:2], st[:, 2:3]
    lse = m + torch.log(s + torch.exp(xy - m))
    p = torch.exp(xd - lse)
    target = target.to(dev)
    valid = (target >= 0) & (target < V)
    tt = target.clamp(0, V - 1)
    w = weight.to(dev, torch.float64) if weight is not None else torch.ones(V, dtype=torch.float64, device=dev)
    wy = w[tt][:, None]
    # (1-eps) w_y p + (eps/V)(p W_all + w_c), then (1-eps) w_y at the target column
    T = (1 - eps) * wy * p + (eps / V) * (p * w_all + w[None, :])
    rows = torch.arange(R, device=dev)
    T[rows, tt] += (1 - eps) * wy[:, 0]
    if z_loss > 0:
        T = T + (2 * z_loss * lse).abs() * p
    if deriv is not None:
        # the capped logit z = c tanh(x / c) carries ~2.5 ulp of fp32 rounding,
        # up to 2^-21.7 |z| absolute, which moves p by that relative amount: the
        # 2^-18 floor covers it up to |z| = 16, so scale the terms by |z| / 8 beyond
        T = T * deriv * torch.clamp(xd.abs() / 8.0, min=1.0)
    T = T * scale.to(dev).abs().reshape(-1, 1).double()
    T[~valid] = 0.0
    return T


def grad_mismatch_detail(got: torch.Tensor, want64: torch.Tensor, T: torch.Tensor) -> dict:
    """Per-element acceptance of a gradient block, computed on the device of
    ``got``: n_bad elements outside the tolerance; n_floor elements that pass
    only through the 2^-18 T floor, not within one ulp of the rounded oracle
    value; worst_ulp the largest error in ulps of the rounded oracle value
    (large only where that value is near 0); worst_tol the largest error as a
    share of the element's tolerance (<= 1 when every element passes)."""
    dtype = got.dtype
    want64 = want64.to(got.device)
    T = T.to(got.device)
    g = got.double()
    if g.numel() == 0:
        return {"n_bad": 0, "n_floor": 0, "worst_ulp": 0.0, "worst_tol": 0.0}
    if dtype == torch.float32:
        u = ulp_of(want64.to(torch.float32), torch.float32)
        tol = FLOOR * T + 2.0 * u
        err = (g - want64).abs()
        return {"n_bad": int((err > tol).sum()), "n_floor": 0,
                "worst_ulp": float((err / u.clamp_min(1e-300)).max()),
                "worst_tol": float((err / tol.clamp_min(1e-300)).max())}
    ref = rne(want64, dtype)
    u = ulp_of(ref, dtype)
    err = (g - ref.double()).abs()
    floor = FLOOR * T
    ok_ulp = err <= u
    ok_floor = err <= floor
    bad = ~(ok_ulp | ok_floor)
    return {"n_bad": int(bad.sum()), "n_floor": int((~ok_ulp & ok_floor).sum()),
            "worst_ulp": float((err / u).max()),
            "worst_tol": float((err / torch.maximum(u, floor).clamp_min(1e-300)).max())}


def grad_mismatch(got: torch.Tensor, want64: torch.Tensor, T: torch.Tensor):
    """(n_bad, n_floor, worst error in ulps) of grad_mismatch_detail."""
    d = grad_mismatch_detail(got, want64, T)
    return d["n_bad"], d["n_floor"], d["worst_ulp"]


def check_loss_rows(got: torch.Tensor, want64: torch.Tensor):
    err = (got.double() - want64).abs()
    tol = LOSS_ROW_RTOL * want64.abs() + LOSS_ROW_ATOL
    bad = err > tol
    assert not bad.any(), f"{int(bad.sum())} row losses off; worst rel {float((err / want64.abs().clamp_min(1e-30)).max()):.3e}"


def check_loss_reduced(got: float, want: float):
    assert abs(got - want) <= LOSS_RED_RTOL * abs(want) + 1e-30, f"reduced loss {got!r} vs oracle {want!r}"


def row_scale(reduction: str, grad_output, n_rows: int, norm_wy: float) -> torch.Tensor:
    """s_i of the gradient for every row (fp64)."""
    if grad_output is None:
        g = torch.ones(1, dtype=torch.float64)
    else:
        g = grad_output.detach().double().cpu().reshape(-1)
    if reduction == "none":
        return g.expand(n_rows).clone() if g.numel() == 1 else g
    s = g[0] / norm_wy if reduction == "mean" and norm_wy != 0 else (g[0] if reduction != "mean" else 0.0)
    return torch.full((n_rows,), float(s), dtype=torch.float64)
