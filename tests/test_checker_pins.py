"""Pins for the tolerance helpers that every parity verdict rests on:
``ce_check.magnitude_T`` (the magnitudes of the gradient's terms before they
cancel), ``ce_check.grad_mismatch`` (the per-element acceptance rule) and
the magnitude sums of ``oracle.flce(..., abs_sums=True)``. Each is checked
against an independent computation on a tiny case: explicit loops over the
terms, hand-built values a known number of ulps away, and products taken by
the test itself from a torch autograd gradient. CPU only."""
import math

import pytest
import torch
import torch.nn.functional as F

import oracle
from ce_check import FLOOR, grad_mismatch, grad_mismatch_detail, magnitude_T, row_scale


def _term_by_term(x, target, weight, eps, scale, softcap, z_loss):
    """|s_i| T_ic from the definition, one element at a time in Python floats."""
    R, V = x.shape
    w = [1.0] * V if weight is None else [float(v) for v in weight]
    w_all = sum(w)
    out = [[0.0] * V for _ in range(R)]
    for i in range(R):
        y = int(target[i])
        if not (0 <= y < V):
            continue
        z = [float(v) for v in x[i]]
        if softcap > 0:
            z = [softcap * math.tanh(v / softcap) for v in z]
        lse = math.log(sum(math.exp(v) for v in z))
        for c in range(V):
            p = math.exp(z[c] - lse)
            t = 0.0
            t += (1 - eps) * w[y] * p                 # softmax term of the target part
            t += (1 - eps) * w[y] * (1.0 if c == y else 0.0)   # one-hot term
            t += (eps / V) * p * w_all                # smoothing: p times the class-weight sum
            t += (eps / V) * w[c]                     # smoothing: the class's own weight
            t += abs(2 * z_loss * lse) * p            # z-loss
            if softcap > 0:
                t *= 1.0 - (z[c] / softcap) ** 2
                t *= max(1.0, abs(z[c]) / 8.0)
            out[i][c] = t * abs(float(scale[i]))
    return torch.tensor(out, dtype=torch.float64)


def _stats_by_hand(x, target, softcap):
    """{m, s, x_y, r} per row as the library stores them (s without the
    target column), from plain loops; r is not read by magnitude_T."""
    R, V = x.shape
    st = torch.zeros(R, 4, dtype=torch.float64)
    for i in range(R):
        z = [float(v) for v in x[i]]
        if softcap > 0:
            z = [softcap * math.tanh(v / softcap) for v in z]
        y = int(target[i])
        m = max(z)
        inr = 0 <= y < V
        st[i, 0] = m
        st[i, 1] = sum(math.exp(z[c] - m) for c in range(V) if not (inr and c == y))
        st[i, 2] = z[y] if inr else 0.0
    return st


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("softcap", [0.0, 2.5])
@pytest.mark.parametrize("z_loss", [0.0, 1e-2])
def test_magnitude_T_matches_term_by_term(weighted, softcap, z_loss):
    g = torch.Generator().manual_seed(7)
    R, V = 5, 9
    x = torch.randn(R, V, generator=g, dtype=torch.float64) * 3.0
    target = torch.tensor([3, -100, 8, 11, 0])          # one ignored, one out of range
    weight = (0.5 + torch.rand(V, generator=g, dtype=torch.float64)) if weighted else None
    eps = 0.15
    scale = torch.tensor([0.3, -1.2, -0.7, 2.0, 1.5], dtype=torch.float64)   # signs: |s_i| is used
    stats = _stats_by_hand(x, target, softcap)
    w_all = float(weight.sum()) if weighted else float(V)
    got = magnitude_T(x, target, stats, weight, eps, w_all, scale, softcap, z_loss)
    want = _term_by_term(x, target, weight, eps, scale, softcap, z_loss)
    assert got.shape == want.shape
    assert torch.allclose(got, want, rtol=1e-12, atol=0)
    assert torch.all(got[1] == 0) and torch.all(got[3] == 0)   # rows that are not valid


def test_row_scale_per_reduction():
    g = torch.tensor([0.37])
    assert torch.allclose(row_scale("mean", g, 4, 2.5), torch.full((4,), 0.37 / 2.5, dtype=torch.float64))
    assert torch.allclose(row_scale("sum", g, 3, 2.5), torch.full((3,), 0.37, dtype=torch.float64))
    gi = torch.tensor([0.1, 0.2, 0.3])
    assert torch.equal(row_scale("none", gi, 3, 2.5), gi.double())
    assert torch.equal(row_scale("mean", None, 2, 4.0), torch.full((2,), 0.25, dtype=torch.float64))
    assert torch.equal(row_scale("mean", g, 2, 0.0), torch.zeros(2, dtype=torch.float64))


def _bf16_step(v: torch.Tensor, k: int) -> torch.Tensor:
    """v (bf16) moved k representable steps away from zero."""
    bits = v.view(torch.int16).to(torch.int32) + k
    return bits.to(torch.int16).view(torch.bfloat16)


def test_grad_mismatch_counts_ulps_and_floor():
    # exact values whose bf16 rounding is known, all positive
    want = torch.tensor([1.0, 0.75, 3.0e-3, 5.0e-6, 2.0, 1.5, 1.0e-7, 0.5], dtype=torch.float64)
    ref = want.to(torch.float32).to(torch.bfloat16)
    got = ref.clone()
    got[1] = _bf16_step(ref[1:2], 1)[0]      # 1 ulp off: accepted by the ulp rule
    got[2] = _bf16_step(ref[2:3], 2)[0]      # 2 ulps off, no floor: bad
    got[3] = _bf16_step(ref[3:4], 2)[0]      # 2 ulps off, inside the floor: floor
    got[4] = _bf16_step(ref[4:5], -1)[0]     # 1 ulp below: accepted
    got[6] = _bf16_step(ref[6:7], 3)[0]      # 3 ulps off, floor too small: bad
    T = torch.zeros(8, dtype=torch.float64)
    err3 = float((got[3].double() - ref[3].double()).abs())
    T[3] = 1.01 * err3 / FLOOR               # floor just covers element 3
    err6 = float((got[6].double() - ref[6].double()).abs())
    T[6] = 0.99 * err6 / FLOOR               # floor just misses element 6
    bad, n_floor, worst = grad_mismatch(got.reshape(2, 4), want.reshape(2, 4), T.reshape(2, 4))
    assert (bad, n_floor) == (2, 1)
    assert worst == pytest.approx(3.0)
    # the share of the tolerance: element 2 is 2 ulps off with no floor
    d = grad_mismatch_detail(got, want, T)
    assert d["worst_tol"] == pytest.approx(2.0)


def test_grad_mismatch_fp32_rule():
    want = torch.tensor([1.0, 1e-3, 2.0 ** -30], dtype=torch.float64)
    ulp = lambda v: float(torch.nextafter(torch.tensor(v, dtype=torch.float32),
                                          torch.tensor(float("inf"))).double() - v)
    got = want.to(torch.float32).clone()
    got[0] += 2 * ulp(1.0)                   # 2 ulps: the fp32 rule's limit
    got[1] = torch.nextafter(torch.nextafter(torch.nextafter(got[1], torch.tensor(1.0)), torch.tensor(1.0)),
                             torch.tensor(1.0))   # 3 ulps, no floor: bad
    T = torch.zeros(3, dtype=torch.float64)
    bad, n_floor, _ = grad_mismatch(got, want, T)
    assert (bad, n_floor) == (1, 0)


def test_flce_abs_sums_against_products_of_autograd_gradient():
    """|dZ| |W| on the sampled rows and |dZ|^T |h| on the sampled columns,
    with dZ from torch's float64 cross-entropy autograd (independent of the
    row oracle) and z = h W^T formed by the test. 1100 rows span three of the
    reference's 512-row blocks."""
    g = torch.Generator().manual_seed(3)
    BT, H, V = 1100, 6, 10
    h = torch.randn(BT, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * 0.7).to(torch.bfloat16)
    t = torch.randint(0, V, (BT,), generator=g)
    t[torch.randperm(BT, generator=g)[:60]] = -100
    rows = torch.tensor([0, 5, 511, 512, 1023, 1024, 1099])
    cols = torch.tensor([0, 3, 9])
    ref = oracle.flce(h, W, t, label_smoothing=0.1, reduction="mean", sample_rows=rows, sample_cols=cols,
                      abs_sums=True)
    hd, Wd = h.double(), W.double()
    z = (hd @ Wd.T).requires_grad_(True)
    loss = F.cross_entropy(z, t, ignore_index=-100, label_smoothing=0.1, reduction="mean")
    (dz,) = torch.autograd.grad(loss, z)
    want_h = dz[rows].abs() @ Wd.abs()
    want_w = dz[:, cols].abs().T @ hd.abs()
    assert torch.allclose(ref["grad_hidden_abs"], want_h, rtol=1e-10, atol=1e-18)
    assert torch.allclose(ref["grad_weight_abs"], want_w, rtol=1e-10, atol=1e-18)
    # and the signed products, as a cross-check of the same sampling
    assert torch.allclose(ref["grad_hidden"], dz[rows] @ Wd, rtol=1e-9, atol=1e-15)
    assert torch.allclose(ref["grad_weight"], dz[:, cols].T @ hd, rtol=1e-9, atol=1e-15)
