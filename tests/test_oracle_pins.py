"""Pins for the fp64 oracle: closed forms, invariants, finite differences,
a library cross-check and the pages' printed numbers. None of these retype
the oracle's own formulas; each checks it against something independent.
CPU only."""
import json
import math
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import IGNORE_INDEX, make_logits, make_targets, make_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(R, V, seed, dtype=torch.float64, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(R, V, generator=g, dtype=torch.float64) * scale).to(dtype)


# ----------------------------------------------------------------- decoding
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_decode_matches_torch_upcast(dtype):
    """The oracle reads bf16 / f16 / f32 storage exactly (compared with
    torch's exact widening to float64) -- via the max statistic."""
    x = _rand(8, 37, 0, torch.float64, 3.0)
    x[0, 0] = 6.0e-8   # f16 subnormal range
    x[1, 1] = -1.0e-40  # f32/bf16 subnormal
    xs = x.to(dtype)
    t = torch.zeros(8, dtype=torch.int64)
    out = oracle.rows(xs, t, want_grad=False)
    ref = xs.to(torch.float64)
    assert torch.equal(out["stats"][:, 0], ref.max(dim=1).values)
    assert torch.equal(out["stats"][:, 2], ref[:, 0])


# ----------------------------------------------------------------- closed forms
@pytest.mark.parametrize("V", [7, 1024])
@pytest.mark.parametrize("eps", [0.0, 0.1, 0.3])
def test_uniform_logits_closed_form(V, eps):
    """All logits equal: loss = log V for every eps; unweighted gradient is
    (1-eps)/(V N) off target and (1/V - (1-eps) - eps/V)/N at the target."""
    N = 5
    x = torch.full((N, V), 0.37, dtype=torch.float64)
    t = torch.tensor([0, 3, V - 1, 2, 1])
    out = oracle.ce(x, t, label_smoothing=eps, reduction="mean")
    assert out["loss"] == pytest.approx(math.log(V), rel=1e-14)
    assert torch.allclose(out["row_loss"], torch.full((N,), math.log(V), dtype=torch.float64),
                          rtol=1e-14, atol=0)
    g = out["grad"]
    off = (1 - eps) / (V * N)
    on = (1.0 / V - (1 - eps) - eps / V) / N
    for i in range(N):
        row = g[i].clone()
        assert row[t[i]].item() == pytest.approx(on, rel=1e-12, abs=1e-15)
        row[t[i]] = off
        assert torch.allclose(row, torch.full((V,), off, dtype=torch.float64), rtol=1e-12, atol=1e-16)


def test_uniform_logits_eps0_dxy():
    """At eps = 0: dx_y = (1/V - 1)/N."""
    V, N = 1000, 4
    x = torch.zeros(N, V, dtype=torch.float64)
    t = torch.tensor([5, 6, 7, 8])
    g = oracle.ce(x, t)["grad"]
    for i in range(N):
        assert g[i, t[i]].item() == pytest.approx((1.0 / V - 1.0) / N, rel=1e-13)


def test_two_class_closed_form():
    """V = 2, eps = 0: loss = softplus(x_other - x_y), dx_y = -sigmoid(x_other - x_y)/N."""
    N = 6
    x = _rand(N, 2, 11, scale=4.0)
    t = torch.tensor([0, 1, 1, 0, 1, 0])
    out = oracle.ce(x, t, reduction="mean")
    for i in range(N):
        y, o = int(t[i]), 1 - int(t[i])
        z = (x[i, o] - x[i, y]).item()
        sp = max(z, 0.0) + math.log1p(math.exp(-abs(z)))
        sig = 1.0 / (1.0 + math.exp(-z))
        assert out["row_loss"][i].item() == pytest.approx(sp, rel=1e-13)
        assert out["grad"][i, y].item() == pytest.approx(-sig / N, rel=1e-12)
        assert out["grad"][i, o].item() == pytest.approx(sig / N, rel=1e-12)


def test_smoothing_explicit_formula():
    """Unweighted: loss = (1-eps)(LSE - x_y) + eps (LSE - mean_c x_c), LSE from
    torch.logsumexp."""
    x = _rand(9, 50, 3, scale=2.0)
    t = make_targets(9, 50, 0.0, 3)
    eps = 0.17
    out = oracle.ce(x, t, label_smoothing=eps, reduction="none")
    lse = torch.logsumexp(x, dim=1)
    xy = x.gather(1, t[:, None]).squeeze(1)
    expect = (1 - eps) * (lse - xy) + eps * (lse - x.mean(dim=1))
    assert torch.allclose(out["row_loss"], expect, rtol=1e-13, atol=0)


# ----------------------------------------------------------------- invariants
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("eps", [0.0, 0.25])
def test_gradient_rows_sum_to_zero(weighted, eps):
    R, V = 12, 333
    x = _rand(R, V, 5, scale=2.0)
    t = make_targets(R, V, 0.2, 5)
    w = make_weights(V, 5).double() if weighted else None
    out = oracle.ce(x, t, weight=w, label_smoothing=eps, reduction="sum", grad_output=torch.tensor([1.7]))
    g = out["grad"]
    scale = g.abs().sum(dim=1).clamp_min(1e-300)
    assert torch.all(g.sum(dim=1).abs() <= 1e-13 * scale)


def test_ignored_rows_zero_and_excluded():
    R, V = 10, 64
    x = _rand(R, V, 7)
    t = make_targets(R, V, 0.0, 7)
    t[[1, 4, 8]] = IGNORE_INDEX
    out = oracle.ce(x, t, label_smoothing=0.1, reduction="mean")
    for i in (1, 4, 8):
        assert out["row_loss"][i].item() == 0.0
        assert torch.count_nonzero(out["grad"][i]) == 0
    keep = torch.tensor([i for i in range(R) if i not in (1, 4, 8)])
    sub = oracle.ce(x[keep], t[keep], label_smoothing=0.1, reduction="mean")
    assert out["loss"] == pytest.approx(sub["loss"], rel=1e-14)
    assert torch.allclose(out["grad"][keep], sub["grad"], rtol=1e-14, atol=0)
    assert out["n_valid"] == R - 3


def test_out_of_range_targets_are_counted_and_ignored():
    x = _rand(4, 10, 9)
    t = torch.tensor([3, 10, -5, IGNORE_INDEX])
    out = oracle.ce(x, t)
    assert out["n_out_of_range"] == 2 and out["n_valid"] == 1
    assert out["row_loss"][1] == 0 and out["row_loss"][2] == 0


def test_mean_with_every_row_ignored_is_zero():
    x = _rand(3, 10, 9)
    t = torch.full((3,), IGNORE_INDEX)
    out = oracle.ce(x, t, reduction="mean")
    assert out["loss"] == 0.0 and torch.count_nonzero(out["grad"]) == 0


def test_shift_invariance():
    R, V = 6, 200
    x = _rand(R, V, 13, scale=3.0)
    t = make_targets(R, V, 0.0, 13)
    w = make_weights(V, 13).double()
    shift = torch.tensor([1000.0, -500.0, 0.0, 37.25, -1e4, 3.0], dtype=torch.float64)[:, None]
    a = oracle.ce(x, t, weight=w, label_smoothing=0.05, reduction="none")
    b = oracle.ce(x + shift, t, weight=w, label_smoothing=0.05, reduction="none")
    assert torch.allclose(a["row_loss"], b["row_loss"], rtol=1e-10, atol=0)
    assert torch.allclose(a["grad"], b["grad"], rtol=1e-8, atol=1e-15)


def test_row_strided_view_matches_contiguous():
    full = make_logits(5, 40, "bf16", 1.0, 21, ld=56)
    assert full.stride(0) == 56
    t = make_targets(5, 40, 0.0, 21)
    a = oracle.ce(full, t, label_smoothing=0.1)
    b = oracle.ce(full.contiguous(), t, label_smoothing=0.1)
    assert torch.equal(a["grad"], b["grad"]) and a["loss"] == b["loss"]


def test_int32_and_int64_targets_agree():
    x = _rand(7, 30, 2)
    t = make_targets(7, 30, 0.3, 2)
    a = oracle.ce(x, t)
    b = oracle.ce(x, t.to(torch.int32))
    assert a["loss"] == b["loss"] and torch.equal(a["grad"], b["grad"])


def test_threads_do_not_change_results():
    x = _rand(33, 77, 4)
    t = make_targets(33, 77, 0.1, 4)
    a = oracle.ce(x, t, label_smoothing=0.1, n_threads=1)
    b = oracle.ce(x, t, label_smoothing=0.1, n_threads=7)
    assert a["loss"] == b["loss"] and torch.equal(a["grad"], b["grad"])


# ----------------------------------------------------------------- statistics
def test_stats_against_library_reductions():
    """stats = {m, off-target exp-sum, x_y, smoothing sum relative to m}:
    m is torch.max; m + log(s + exp(x_y - m)) is torch.logsumexp; x_y is a
    gather; r + W_all * m is the weighted sum (a dot product)."""
    R, V = 9, 123
    x = _rand(R, V, 17, scale=2.5)
    t = make_targets(R, V, 0.0, 17)
    t[2] = IGNORE_INDEX
    w = make_weights(V, 17).double()
    st = oracle.ce(x, t, weight=w, label_smoothing=0.1)["stats"]
    m, s, xy, r = st.unbind(1)
    assert torch.equal(m, x.max(dim=1).values)
    lse = torch.logsumexp(x, dim=1)
    valid = t >= 0
    d = torch.where(valid, s + torch.exp(xy - m), s)
    assert torch.allclose(m + torch.log(d), lse, rtol=1e-14, atol=0)
    assert torch.equal(xy[valid], x[valid].gather(1, t[valid, None]).squeeze(1))
    assert xy[2] == 0
    assert torch.allclose(r + w.sum() * m, x @ w, rtol=1e-12, atol=1e-10)


# ----------------------------------------------------------------- finite differences
def _objective(x, t, w, eps, red, g):
    out = oracle.ce(x, t, weight=w, label_smoothing=eps, reduction=red, want_grad=False)
    if red == "none":
        return float((out["row_loss"] * g).sum())
    return float(out["loss"]) * float(g[0])


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("eps", [0.0, 0.2])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
@pytest.mark.parametrize("ignore", [False, True])
def test_gradient_matches_central_differences(weighted, eps, red, ignore):
    R, V = 5, 9
    x = _rand(R, V, 23, scale=1.5)
    t = make_targets(R, V, 0.0, 23)
    if ignore:
        t[3] = IGNORE_INDEX
    w = make_weights(V, 23).double() if weighted else None
    g = torch.tensor([0.3, 1.1, 0.7, 2.0, 0.5], dtype=torch.float64) if red == "none" \
        else torch.tensor([0.8], dtype=torch.float64)
    grad = oracle.ce(x, t, weight=w, label_smoothing=eps, reduction=red, grad_output=g)["grad"]
    h = 1e-6
    fd = torch.zeros_like(x)
    for i in range(R):
        for c in range(V):
            xp = x.clone(); xp[i, c] += h
            xm = x.clone(); xm[i, c] -= h
            fd[i, c] = (_objective(xp, t, w, eps, red, g) - _objective(xm, t, w, eps, red, g)) / (2 * h)
    assert torch.allclose(grad, fd, rtol=1e-6, atol=1e-8), (grad - fd).abs().max()


# ----------------------------------------------------------------- library cross-check
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_against_torch_cross_entropy_fp64(weighted, eps, red):
    """torch.nn.functional.cross_entropy in float64 on the CPU, with autograd."""
    R, V = 17, 301
    x = _rand(R, V, 29, scale=2.0)
    t = make_targets(R, V, 0.2, 29)
    # a few confident rows
    x[0, t[0].clamp_min(0)] += 12.0
    x[1, t[1].clamp_min(0)] += 9.0
    w = make_weights(V, 29).double() if weighted else None
    g = torch.rand(R, dtype=torch.float64, generator=torch.Generator().manual_seed(1)) if red == "none" \
        else torch.tensor([0.37], dtype=torch.float64)
    xr = x.clone().requires_grad_(True)
    loss = F.cross_entropy(xr, t, weight=w, ignore_index=IGNORE_INDEX, label_smoothing=eps, reduction=red)
    (loss * g if red == "none" else loss * g[0]).sum().backward()
    out = oracle.ce(x, t, weight=w, label_smoothing=eps, reduction=red, grad_output=g)
    if red == "none":
        assert torch.allclose(out["row_loss"], loss.detach(), rtol=1e-12, atol=1e-14)
    else:
        assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    assert torch.allclose(out["grad"], xr.grad, rtol=1e-10, atol=1e-16)


def test_flce_against_torch_autograd_fp64():
    """Fused-linear reference vs torch autograd through F.linear + cross_entropy."""
    BT, H, V = 40, 24, 70
    g = torch.Generator().manual_seed(3)
    h = torch.randn(BT, H, generator=g, dtype=torch.float64)
    W = torch.randn(V, H, generator=g, dtype=torch.float64) * 0.3
    b = torch.randn(V, generator=g, dtype=torch.float64) * 0.1
    t = make_targets(BT, V, 0.1, 3)
    hr, Wr, br = (a.clone().requires_grad_(True) for a in (h, W, b))
    loss = F.cross_entropy(F.linear(hr, Wr, br), t, ignore_index=IGNORE_INDEX, label_smoothing=0.05)
    loss.backward()
    rows = [0, 5, 39, 17]
    cols = [0, 69, 33]
    out = oracle.flce(h, W, t, bias=b, label_smoothing=0.05, sample_rows=rows, sample_cols=cols)
    assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    assert torch.allclose(out["grad_hidden"], hr.grad[rows], rtol=1e-10, atol=1e-15)
    assert torch.allclose(out["grad_weight"], Wr.grad[cols], rtol=1e-10, atol=1e-15)
    assert torch.allclose(out["grad_bias"], br.grad[cols], rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_flce_class_weight_grad_output_against_torch_autograd_fp64(reduction):
    """The fused-linear reference with class weights, label smoothing and a
    grad_output (per row for none) vs torch autograd of the same composition."""
    BT, H, V = 36, 16, 50
    g = torch.Generator().manual_seed(4)
    h = torch.randn(BT, H, generator=g, dtype=torch.float64)
    W = torch.randn(V, H, generator=g, dtype=torch.float64) * 0.3
    w = torch.rand(V, generator=g, dtype=torch.float64) + 0.5
    t = make_targets(BT, V, 0.2, 4)
    go = torch.rand(BT, generator=g, dtype=torch.float64) if reduction == "none" else torch.tensor(0.37,
                                                                                                 dtype=torch.float64)
    hr, Wr = (a.clone().requires_grad_(True) for a in (h, W))
    loss = F.cross_entropy(F.linear(hr, Wr), t, weight=w, ignore_index=IGNORE_INDEX, label_smoothing=0.1,
                           reduction=reduction)
    loss.backward(go)
    out = oracle.flce(h, W, t, label_smoothing=0.1, reduction=reduction, class_weight=w, grad_output=go)
    if reduction == "none":
        assert torch.allclose(out["loss"], loss.detach(), rtol=1e-12, atol=1e-15)
    else:
        assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    assert torch.allclose(out["grad_hidden"], hr.grad, rtol=1e-10, atol=1e-15)
    assert torch.allclose(out["grad_weight"], Wr.grad, rtol=1e-10, atol=1e-15)


def test_flce_softcap_zloss_accuracy_against_torch_autograd_fp64():
    """The fused-linear reference with softcap and z-loss vs torch autograd of
    linear -> c tanh(. / c) -> cross_entropy + lambda logsumexp^2 (valid rows,
    the cross-entropy's normaliser); its token accuracy vs the argmax of the
    linear layer's output."""
    BT, H, V = 30, 12, 40
    c, lam = 2.0, 1e-3
    g = torch.Generator().manual_seed(6)
    h = torch.randn(BT, H, generator=g, dtype=torch.float64)
    W = torch.randn(V, H, generator=g, dtype=torch.float64)
    t = make_targets(BT, V, 0.2, 6)
    hr, Wr = (a.clone().requires_grad_(True) for a in (h, W))
    z = c * torch.tanh(F.linear(hr, Wr) / c)
    valid = t != IGNORE_INDEX
    base = F.cross_entropy(z, t, ignore_index=IGNORE_INDEX, label_smoothing=0.1)
    loss = base + lam * (torch.logsumexp(z, dim=1) ** 2 * valid).sum() / valid.sum()
    loss.backward()
    out = oracle.flce(h, W, t, label_smoothing=0.1, softcap=c, z_loss=lam)
    assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    assert torch.allclose(out["grad_hidden"], hr.grad, rtol=1e-10, atol=1e-15)
    assert torch.allclose(out["grad_weight"], Wr.grad, rtol=1e-10, atol=1e-15)
    am = (h @ W.T).argmax(dim=1)
    assert out["accuracy"] == pytest.approx(float((am[valid] == t[valid]).double().mean()), abs=1e-15)


# ----------------------------------------------------------------- the pages' numbers
def _bf16_round(v: torch.Tensor) -> torch.Tensor:
    return v.to(torch.float32).to(torch.bfloat16).to(torch.float64)


def test_dxy_error_table_shape_reproduced():
    """The #1329 commit message prints the max relative dx_y error of the
    #1268 kernel (bf16, V=32000): 1.95% / 19.99% / 100% at softmax(x_y) =
    0.9 / 0.99 / 0.999. That kernel rounded softmax(x_y)/N to bf16 and then
    subtracted 1/N. Rows whose realised softmax(x_y) sweeps a narrow band
    around each printed value (off-target logits 0, target logit set in
    fp64; the band is one bf16 ulp wide) give the oracle's exact dx_y; modelling the #1268 double rounding
    on top of the oracle's softmax and taking the worst row of each band must
    reproduce the printed maxima. A wrong sign, scale or a missing -1 in the
    oracle's dx_y breaks the match. One RNE rounding of the oracle's value
    errs by at most 2^-8 = 0.39% relative, the bound the before-#1268 column
    (single rounding) also keeps."""
    table = json.load(open(os.path.join(GOLDEN, "dxy_error_table_v32000_bf16.json")))
    V = table["vocab"]
    R = 128                              # N = 128 valid rows: 1/N exact in bf16
    for p0, before, at1268, torch_col in table["rows"]:
        half = min(2.0 ** -9, 0.25 * (1.0 - p0))   # at most half a bf16 ulp in [0.5, 1)
        p = torch.linspace(p0 - half, p0 + half, R, dtype=torch.float64)
        x = torch.zeros(R, V, dtype=torch.float64)
        t = torch.arange(R, dtype=torch.int64) * 97 % V
        x[torch.arange(R), t] = torch.log(p / (1.0 - p) * (V - 1))
        out = oracle.ce(x, t, reduction="mean")
        N = out["n_valid"]
        assert N == R
        dxy = out["grad"].gather(1, t[:, None]).squeeze(1)            # exact, fp64
        st = out["stats"]
        e_y = torch.exp(st[:, 2] - st[:, 0])
        p_y = e_y / (st[:, 1] + e_y)
        assert torch.allclose(p_y, p, rtol=1e-12, atol=0)
        model_1268 = _bf16_round(_bf16_round(p_y / N) - 1.0 / N)
        rel_1268 = (model_1268 - dxy).abs() / dxy.abs()
        rel_single = (_bf16_round(dxy) - dxy).abs() / dxy.abs()
        got = 100.0 * rel_1268.max().item()
        if at1268 >= 100.0:
            assert got == pytest.approx(100.0, abs=1e-9)
        else:
            assert got == pytest.approx(at1268, rel=0.02)
        assert 100.0 * rel_single.max().item() <= 100 * 2.0 ** -8
        assert before <= 100 * 2.0 ** -8


def test_peak_memory_table_is_one_logits_tensor():
    """The pages' peak-memory tables equal one logits tensor (BT*V*element
    size, in MiB) to within 3 MB of small per-row buffers: the gradient is
    written over the logits. This fixes the memory rule the library keeps."""
    d = json.load(open(os.path.join(GOLDEN, "peak_memory_mb.json")))
    for key, esz in (("bf16_vocab_sweep_bt8192", 2), ("fp32_vocab_sweep_bt8192", 4)):
        for v, mb in d[key].items():
            assert 0 <= mb - 8192 * int(v) * esz / 2 ** 20 <= 3
    for key, esz in (("bf16_bt_sweep_v128256", 2), ("fp32_bt_sweep_v128256", 4)):
        for bt, mb in d[key].items():
            assert -1 <= mb - int(bt) * 128256 * esz / 2 ** 20 <= 3


# ----------------------------------------------------------------- softcap, z-loss, accuracy
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_softcap_zloss_against_torch_autograd(weighted, red):
    """Softcap and z-loss against torch autograd through the composed library
    routines: z = c tanh(x / c), cross_entropy(z) + lambda * logsumexp(z)^2 on
    the valid rows (reduced with the cross-entropy's normaliser)."""
    R, V = 13, 97
    c, lam, eps = 3.0, 1e-3, 0.1
    x = _rand(R, V, 31, scale=4.0)
    t = make_targets(R, V, 0.2, 31)
    w = make_weights(V, 31).double() if weighted else None
    g = torch.rand(R, dtype=torch.float64, generator=torch.Generator().manual_seed(2)) if red == "none" \
        else torch.tensor([0.6], dtype=torch.float64)
    xr = x.clone().requires_grad_(True)
    z = c * torch.tanh(xr / c)
    ce_l = F.cross_entropy(z, t, weight=w, ignore_index=IGNORE_INDEX, label_smoothing=eps, reduction="none")
    valid = t != IGNORE_INDEX
    zl = lam * torch.logsumexp(z, dim=1) ** 2 * valid
    if red == "none":
        loss = ce_l + zl
        (loss * g).sum().backward()
    else:
        denom = (w[t.clamp_min(0)] * valid).sum() if weighted else valid.sum()
        base = F.cross_entropy(z, t, weight=w, ignore_index=IGNORE_INDEX, label_smoothing=eps, reduction=red)
        loss = base + (zl.sum() / denom if red == "mean" else zl.sum())
        (loss * g[0]).backward()
    out = oracle.ce(x, t, weight=w, label_smoothing=eps, reduction=red, grad_output=g, softcap=c, z_loss=lam)
    if red == "none":
        assert torch.allclose(out["row_loss"], loss.detach(), rtol=1e-12, atol=1e-14)
    else:
        assert out["loss"] == pytest.approx(loss.item(), rel=1e-12)
    assert torch.allclose(out["grad"], xr.grad, rtol=1e-10, atol=1e-16)


def test_huge_softcap_is_no_softcap():
    x = _rand(6, 40, 5, scale=2.0)
    t = make_targets(6, 40, 0.0, 5)
    a = oracle.ce(x, t, label_smoothing=0.1)
    b = oracle.ce(x, t, label_smoothing=0.1, softcap=1e7)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    assert torch.allclose(a["grad"], b["grad"], rtol=1e-10, atol=1e-13)


def test_zloss_uniform_logits_closed_form():
    """All logits x0: LSE = x0 + log V, so loss = log V + lambda (x0 + log V)^2
    and every off-target gradient is (1 + 2 lambda LSE) / (V N)."""
    R, V, x0, lam = 4, 50, 0.3, 0.01
    x = torch.full((R, V), x0, dtype=torch.float64)
    t = torch.tensor([0, 7, 49, 3])
    out = oracle.ce(x, t, z_loss=lam)
    lse = x0 + math.log(V)
    assert out["loss"] == pytest.approx(math.log(V) + lam * lse * lse, rel=1e-13)
    off = (1 + 2 * lam * lse) / (V * R)
    g = out["grad"][1].clone()
    g[7] = off
    assert torch.allclose(g, torch.full((V,), off, dtype=torch.float64), rtol=1e-12, atol=0)


@pytest.mark.parametrize("z_loss", [0.0, 1e-4])
def test_zloss_and_softcap_finite_differences(z_loss):
    R, V = 4, 7
    x = _rand(R, V, 8, scale=2.0)
    t = torch.tensor([1, IGNORE_INDEX, 6, 0])
    g = torch.tensor([0.9], dtype=torch.float64)
    grad = oracle.ce(x, t, label_smoothing=0.2, grad_output=g, softcap=2.5, z_loss=z_loss)["grad"]
    h = 1e-6
    fd = torch.zeros_like(x)
    for i in range(R):
        for c in range(V):
            xp, xm = x.clone(), x.clone()
            xp[i, c] += h
            xm[i, c] -= h
            lp = oracle.ce(xp, t, label_smoothing=0.2, softcap=2.5, z_loss=z_loss, want_grad=False)["loss"]
            lm = oracle.ce(xm, t, label_smoothing=0.2, softcap=2.5, z_loss=z_loss, want_grad=False)["loss"]
            fd[i, c] = 0.9 * (lp - lm) / (2 * h)
    assert torch.allclose(grad, fd, rtol=1e-6, atol=1e-9)


def test_argmax_and_accuracy_against_torch_argmax():
    R, V = 40, 300
    x = _rand(R, V, 77, scale=2.0).to(torch.bfloat16)   # bf16 makes ties common enough
    x[3, 10] = x[3, 20] = 50.0                            # a tie: the first column wins
    t = torch.argmax(x.double(), dim=1)
    t[::3] = make_targets(R, V, 0.0, 77)[::3]
    t[5] = IGNORE_INDEX
    out = oracle.ce(x, t, want_grad=False)
    assert torch.equal(out["argmax"], torch.argmax(x.double(), dim=1))
    assert out["argmax"][3] == 10
    valid = t != IGNORE_INDEX
    expect = float((torch.argmax(x.double(), dim=1)[valid] == t[valid]).double().mean())
    assert out["accuracy"] == pytest.approx(expect, rel=0, abs=1e-15)
