"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases cover every dtype, reduction, smoothing / weight combination,
ragged vocabularies, padded and misaligned row strides and every fused
cluster size; the full-size workloads are checked on every row's loss and
every element of every row's gradient."""
import time
import zlib

import pytest
import torch

import oracle
from ce_check import (DXY_RTOL, FLOOR, check_loss_reduced, check_loss_rows, grad_mismatch,
                      grad_mismatch_detail, magnitude_T, row_scale, ulp_of)
from workloads import (CONFIGS, IGNORE_INDEX, make_ce_inputs, make_grad_output, make_logits,
                       make_targets, make_weights)

pytestmark = pytest.mark.gpu
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def ce():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import softmax_cross_entropy_pass_gb300 as ce
    return ce


def _oracle(x, t, w, eps, red, g):
    return oracle.ce(x.cpu(), t.cpu(), weight=None if w is None else w.cpu(), label_smoothing=eps,
                     reduction=red, grad_output=None if g is None else g.cpu())


def _check_all(got_x, t, w, eps, red, g, ref, got_loss, x_in, softcap=0.0, z_loss=0.0):
    R, V = got_x.shape
    if red == "none":
        check_loss_rows(got_loss.cpu(), ref["row_loss"])
    else:
        check_loss_reduced(float(got_loss.cpu()[0]), ref["loss"])
    scale = row_scale(red, g, R, ref["norm_wy"])
    T = magnitude_T(x_in, t.cpu(), ref["stats"], None if w is None else w.cpu(), eps, ref["w_all"], scale,
                    softcap, z_loss)
    bad, n_floor, worst = grad_mismatch(got_x.cpu(), ref["grad"], T)
    assert bad == 0, f"{bad} gradient elements outside tolerance (worst {worst:.2f} ulp, floor used {n_floor})"
    # dx_y of every valid row
    valid = (t.cpu() >= 0) & (t.cpu() < V)
    if valid.any() and got_x.dtype != torch.float32:
        rows = valid.nonzero().flatten()
        tt = t.cpu()[rows]
        want = ref["grad"][rows, tt]
        gotv = got_x.cpu()[rows, tt].double()
        nz = want.abs() > 0
        rel = ((gotv - want).abs() / want.abs())[nz]
        # rows where dx_y itself cancels (smoothing) are covered by the element check
        big = (want.abs() > 1e-3 * T[rows, tt])[nz]
        if big.any():
            assert rel[big].max() <= DXY_RTOL, f"dx_y rel err {float(rel[big].max()):.3e}"


SMALL = [
    # (rows, vocab, ld_extra)
    (1, 1, 0), (3, 2, 0), (5, 7, 0), (17, 1000, 0), (8, 4097, 0), (9, 33000, 0),
    (6, 70001, 0), (4, 131077, 0), (12, 1000, 3), (7, 2048, 8),
]


RAGGED = [
    # (rows, vocab, ld, first column of the view inside a wider buffer)
    (7, 1001, 1001, 0), (5, 4099, 4103, 3), (3, 3, 5, 1), (9, 65537, 65537, 1), (4, 20000, 20011, 5),
    (2, 9, 9, 7),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: f"{s[0]}x{s[1]}ld{s[2]}@{s[3]}")
@pytest.mark.parametrize("opt", ["plain", "weighted_smooth"])
@pytest.mark.parametrize("tune", [0, 8, 9, 16, 24, 54], ids=lambda t: f"tune{t}")
def test_stream_ragged_rows(ce, dtype, shape, opt, tune):
    """The stream kernel on rows that do not start on a 16-byte boundary: the
    head and tail of each row (and of each part for a CTA pair or quad) go
    through plain accesses, the interior through the bulk-copy ring; the
    view starts inside a wider buffer so the base itself is misaligned."""
    R, V, ld, off = shape
    dev = torch.device("cuda")
    seed = zlib.crc32(repr((R, V, ld, off, dtype, opt)).encode()) % 10007
    buf = make_logits(R, ld + off, dtype, 2.0, seed, device=dev)
    x = buf[:, off:off + V]
    t = make_targets(R, V, 0.25, seed, device=dev)
    if R > 2:
        t[1] = V - 1
        t[2] = 0
    w = make_weights(V, seed, device=dev) if opt == "weighted_smooth" else None
    eps = 0.0 if opt == "plain" else 0.1
    g = torch.tensor([0.37], device=dev)
    x_in = x.cpu()
    ref = _oracle(x, t, w, eps, "mean", g)
    outside = buf.clone()
    loss = ce.ce_fwd_bwd(x, t, grad_output=g, weight=w, label_smoothing=eps, reduction="mean",
                         variant="stream", tune=tune)
    torch.cuda.synchronize()
    _check_all(x, t, w, eps, "mean", g, ref, loss, x_in)
    # columns of the buffer outside the view are untouched
    keep = torch.ones(ld + off, dtype=torch.bool)
    keep[off:off + V] = False
    assert torch.equal(buf[:, keep.to(dev)].cpu(), outside[:, keep.to(dev)].cpu())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: f"{s[0]}x{s[1]}+{s[2]}")
@pytest.mark.parametrize("opt", ["plain", "smooth", "weighted_smooth"])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
@pytest.mark.parametrize("api", ["fused", "split", "rowpass", "stream", "stream-pair", "fwd+bwd calls"])
def test_parity_small(ce, dtype, shape, opt, red, api):
    R, V, extra = shape
    dev = torch.device("cuda")
    seed = zlib.crc32(repr((R, V, extra, dtype, opt, red)).encode()) % 10007
    x = make_logits(R, V, dtype, 2.0, seed, device=dev, ld=V + extra if extra else None)
    t = make_targets(R, V, 0.25, seed, device=dev)
    if R > 2:
        t[1] = V - 1
    w = make_weights(V, seed, device=dev) if opt == "weighted_smooth" else None
    eps = 0.0 if opt == "plain" else 0.1
    g = (torch.rand(R, generator=torch.Generator().manual_seed(seed)).to(dev) if red == "none"
         else torch.tensor([0.37], device=dev))
    x_in = x.cpu()
    ref = _oracle(x, t, w, eps, red, g)
    if api == "fwd+bwd calls":
        loss, stats = ce.ce_forward(x, t, weight=w, label_smoothing=eps, reduction=red)
        ce.ce_backward(x, t, stats, grad_output=g, weight=w, label_smoothing=eps, reduction=red)
        torch.cuda.synchronize()
        st = stats.cpu().double()
        valid = (t.cpu() >= 0)
        assert torch.equal(st[:, 0], ref["stats"][:, 0].float().double())       # max is exact
        assert torch.equal(st[valid, 2], ref["stats"][valid, 2].float().double())  # x_y is exact
        assert torch.allclose(st[:, 1], ref["stats"][:, 1], rtol=2e-5, atol=0)
    else:
        variant, tune = (api, 0) if api != "stream-pair" else ("stream", 8)
        ld = x.stride(0) if R > 1 else V
        fusable = x.data_ptr() % 16 == 0 and (R == 1 or (ld * x.element_size()) % 16 == 0)
        if variant == "fused" and not fusable:
            with pytest.raises(ce.CEError):
                ce.ce_fwd_bwd(x, t, grad_output=g, weight=w, label_smoothing=eps, reduction=red,
                              variant=variant)
            return
        if variant == "fused" and ce.ce_fused_plan(R, V, DT[dtype]) is None:
            pytest.skip("fused kernel does not take this shape")
        loss = ce.ce_fwd_bwd(x, t, grad_output=g, weight=w, label_smoothing=eps, reduction=red,
                             variant=variant, tune=tune)
        torch.cuda.synchronize()
    _check_all(x, t, w, eps, red, g, ref, loss, x_in)
    if extra:
        full = x.as_strided((R, V + extra), (V + extra, 1))
        assert torch.equal(full[:, V:].cpu(), torch.full((R, extra), 777.0).to(x.dtype)), "padding written"


@pytest.mark.parametrize("cluster", [1, 2, 3, 4, 5, 8, 16])
def test_fused_every_cluster_size(ce, cluster):
    R, V = 40, 128256
    dev = torch.device("cuda")
    x = make_logits(R, V, "bf16", 1.0, 100 + cluster, device=dev)
    t = make_targets(R, V, 0.05, 100 + cluster, device=dev)
    if ce.ce_fused_plan(R, V, torch.bfloat16, label_smoothing=0.1, cluster=cluster) is None:
        pytest.skip(f"cluster {cluster} cannot hold this row")
    x_in = x.cpu()
    ref = _oracle(x, t, None, 0.1, "mean", None)
    loss = ce.ce_fwd_bwd(x, t, label_smoothing=0.1, reduction="mean", variant="fused", cluster=cluster)
    torch.cuda.synchronize()
    _check_all(x, t, None, 0.1, "mean", None, ref, loss, x_in)


def test_more_rows_than_clusters_and_int32_targets(ce):
    R, V = 3000, 5000
    dev = torch.device("cuda")
    x = make_logits(R, V, "bf16", 1.0, 5, device=dev)
    t = make_targets(R, V, 0.1, 5, device=dev).to(torch.int32)
    x_in = x.cpu()
    ref = _oracle(x, t, None, 0.0, "mean", None)
    loss = ce.ce_fwd_bwd(x, t, variant="fused")
    torch.cuda.synchronize()
    _check_all(x, t, None, 0.0, "mean", None, ref, loss, x_in)


# ---------------------------------------------------------------- edge cases
def test_zero_rows(ce):
    x = torch.empty(0, 100, dtype=torch.bfloat16, device="cuda")
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    loss = torch.full((1,), 5.0, device="cuda")
    ce.ce_fwd_bwd(x, t, loss=loss)
    assert float(loss.item()) == 0.0


@pytest.mark.parametrize("variant", ["fused", "split"])
def test_all_rows_ignored_mean(ce, variant):
    x = make_logits(6, 304, "bf16", 1.0, 3, device="cuda")
    t = torch.full((6,), IGNORE_INDEX, device="cuda")
    ws = ce.workspace(6)
    loss = ce.ce_fwd_bwd(x, t, variant=variant, ws=ws)
    assert ce.ce_get_status(ws) & ce.CE_FLAG_NO_VALID_ROWS
    assert float(loss.item()) == 0.0
    assert torch.count_nonzero(x) == 0


@pytest.mark.parametrize("variant", ["fused", "split"])
def test_out_of_range_target_flag_and_ignored(ce, variant):
    R, V = 5, 400
    x = make_logits(R, V, "bf16", 1.0, 4, device="cuda")
    t = torch.tensor([3, V, -7, IGNORE_INDEX, 10], device="cuda")
    x_in = x.cpu()
    ref = _oracle(x, t, None, 0.0, "sum", None)
    ws = ce.workspace(R)
    loss = ce.ce_fwd_bwd(x, t, variant=variant, reduction="sum", ws=ws)
    assert ce.ce_get_status(ws) & ce.CE_FLAG_TARGET_OUT_OF_RANGE
    _check_all(x, t, None, 0.0, "sum", None, ref, loss, x_in)
    assert torch.count_nonzero(x[1:4]) == 0


def test_argument_errors_enqueue_nothing(ce):
    x = make_logits(4, 64, "bf16", 1.0, 1, device="cuda")
    t = make_targets(4, 64, 0.0, 1, device="cuda")
    before = x.clone()
    ws = ce.workspace(4)
    with pytest.raises(ce.CEError):
        ce.ce_fwd_bwd(x, t, label_smoothing=1.5, ws=ws)
    with pytest.raises(ce.CEError):
        ce.ce_fwd_bwd(x, t, ws=ws[:8])
    torch.cuda.synchronize()
    assert torch.equal(x, before)


# ---------------------------------------------------------------- grad_output scaling
def test_scale_grad_skips_at_one_and_scales(ce):
    x = make_logits(10, 1000, "bf16", 1.0, 9, device="cuda")
    before = x.clone()
    ce.ce_scale_grad(x, torch.tensor([1.0], device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(x, before)
    ce.ce_scale_grad(x, torch.tensor([0.5], device="cuda"))
    assert torch.equal(x, (before.float() * 0.5).to(torch.bfloat16))
    g = torch.rand(10, device="cuda")
    y = before.clone()
    ce.ce_scale_grad(y, g, reduction="none")
    assert torch.equal(y, (before.float() * g[:, None]).to(torch.bfloat16))


@pytest.mark.parametrize("grad_mode", ["inplace", "exact"])
@pytest.mark.parametrize("reduction", ["mean", "none"])
@pytest.mark.parametrize("gscale", [1.0, 0.37])
def test_autograd_function(ce, gscale, reduction, grad_mode):
    """cross_entropy's autograd path against the oracle element by element.
    The exact mode, and the in-place mode at grad_output 1, round each
    element once (1 ulp, or the cancellation floor); the in-place mode at
    grad_output != 1 rounds the g = 1 gradient, then its product with g:
    within 2 ulps of the once-rounded oracle value (the first rounding errs
    by half an ulp of the unscaled value, which g maps to at most one ulp of
    the result; the second adds half an ulp), or the floor scaled the same
    way."""
    R, V = 32, 5000
    x = make_logits(R, V, "bf16", 1.0, 12, device="cuda")
    t = make_targets(R, V, 0.1, 12, device="cuda")
    w = make_weights(V, 12, device="cuda")
    x_in = x.cpu()
    gvec = (torch.rand(R, generator=torch.Generator().manual_seed(5)) * gscale if reduction == "none"
            else torch.tensor([gscale]))
    ref = _oracle(x, t, w, 0.1, reduction, gvec)
    xr = x.clone().requires_grad_(True)
    buf = xr.detach()
    loss = ce.cross_entropy(xr, t, weight=w, label_smoothing=0.1, reduction=reduction, grad_mode=grad_mode)
    if reduction == "none":
        (loss * gvec.to("cuda")).sum().backward()
        check_loss_rows(loss.detach().cpu(), ref["row_loss"])
    else:
        (loss * gscale).backward()
        check_loss_reduced(float(loss.item()), ref["loss"])
    torch.cuda.synchronize()
    assert xr.grad.data_ptr() == buf.data_ptr()  # gradient lives in the logits buffer
    got = xr.grad.cpu()
    scale = row_scale(reduction, gvec, R, ref["norm_wy"])
    T = magnitude_T(x_in, t.cpu(), ref["stats"], w.cpu(), 0.1, ref["w_all"], scale)
    twice = grad_mode == "inplace" and not (gscale == 1.0 and reduction != "none")
    if not twice:
        bad, _, worst = grad_mismatch(got, ref["grad"], T)
        assert bad == 0, worst
    else:
        want = ref["grad"].to(torch.float32).to(torch.bfloat16)
        u = ulp_of(want, torch.bfloat16)
        err = (got.double() - want.double()).abs()
        bad = err > torch.maximum(2 * u, FLOOR * T)
        assert int(bad.sum()) == 0, float((err / u).max())


# ---------------------------------------------------------------- no host synchronisation
@pytest.mark.parametrize("V,variants", [(32000, ("fused", "split", "stream")), (160000, ("stream",))],
                         ids=["64KB-rows", "320KB-rows"])
def test_calls_capture_into_a_cuda_graph(ce, V, variants):
    """Stream capture fails on any synchronising call or pageable copy; the
    replayed graph (class weights: the eight-block normaliser kernels, their
    combining kernel and the row kernel with its programmatic dependency)
    gives the eager call's bits. 320 KB rows with class weights run on
    clusters of four."""
    R = 64
    x0 = make_logits(R, V, "bf16", 1.0, 21, device="cuda")
    t = make_targets(R, V, 0.1, 21, device="cuda")
    g = torch.tensor([0.37], device="cuda")
    w = make_weights(V, 21, device="cuda")
    outs = {}
    for red in ("mean", "sum", "none"):
        for variant in variants:
            x = x0.clone()
            xe = x0.clone()
            ws = ce.workspace(R)
            loss = torch.empty(R if red == "none" else 1, device="cuda")
            gg = torch.rand(R, device="cuda") if red == "none" else g
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=0.05, reduction=red, grad_output=gg,
                              variant=variant, loss=loss, ws=ws, stream=s)  # warm-up (plan cache)
                x.copy_(x0)
                with torch.cuda.graph(graph, stream=s):
                    ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=0.05, reduction=red, grad_output=gg,
                                  variant=variant, loss=loss, ws=ws, stream=s)
            x.copy_(x0)
            graph.replay()
            torch.cuda.synchronize()
            le = ce.ce_fwd_bwd(xe, t, weight=w, label_smoothing=0.05, reduction=red, grad_output=gg,
                               variant=variant)
            torch.cuda.synchronize()
            assert torch.equal(x, xe) and torch.equal(loss, le)
            outs[(red, variant)] = loss


def test_host_returns_without_waiting(ce):
    R, V = 512, 128256
    x = make_logits(R, V, "bf16", 1.0, 22, device="cuda")
    t = make_targets(R, V, 0.05, 22, device="cuda")
    ws = ce.workspace(R)
    loss = torch.empty(1, device="cuda")
    g = torch.tensor([0.5], device="cuda")
    ce.ce_fwd_bwd(x, t, loss=loss, ws=ws, grad_output=g)  # plan cache warm
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # ~0.1 s of device work queued ahead
    t0 = time.perf_counter()
    for red in ("mean", "sum"):
        ce.ce_fwd_bwd(x, t, loss=loss, ws=ws, grad_output=g, reduction=red)
        ce.ce_fwd_bwd(x, t, loss=loss, ws=ws, grad_output=g, reduction=red, variant="split")
    host_ms = (time.perf_counter() - t0) * 1e3
    torch.cuda.synchronize()
    assert host_ms < 20.0, f"host blocked for {host_ms:.1f} ms"


def test_library_allocates_no_device_memory(ce):
    R, V = 256, 50000
    x = make_logits(R, V, "bf16", 1.0, 23, device="cuda")
    t = make_targets(R, V, 0.0, 23, device="cuda")
    ws = ce.workspace(R)
    loss = torch.empty(1, device="cuda")
    ce.ce_fwd_bwd(x, t, loss=loss, ws=ws)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for variant in ("fused", "split"):
        ce.ce_fwd_bwd(x, t, loss=loss, ws=ws, variant=variant)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 == free1


# ---------------------------------------------------------------- full-size workloads
# Share of gradient elements allowed to pass through the 2^-18 T floor
# instead of one ulp. The floor is for elements whose exact value is near 0
# (p_ic close to eps/V, or a softcap / weighted cancellation). With N(0,1)
# bf16 logits and eps/V smoothing, the fp32 p of an element carries about
# 2^-20 relative error, so the floor is needed when |G| < 2^-12 p, i.e. for
# logits within ~2^-12 of the row's crossing point x0 = log(eps/V) + LSE: a
# density of ~0.08 per unit times 2 * 2^-12, about 4e-5 of the elements at
# most (measured on the full workloads: 7e-6 headline, 1.3e-5 large
# vocabulary, 0 on the confident rows, which have no smoothing).
FLOOR_SHARE_MAX = 5e-5


def _record(entry: dict):
    """Appends a JSON line to the file named by CE_PARITY_RECORD (if set)."""
    import json
    import os
    path = os.environ.get("CE_PARITY_RECORD")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(entry) + "\n")


def _full_size_check(ce, cfg, variant, block_elems=1 << 27):
    """One call of the hot path on the whole workload, then every row of it
    against the oracle: the reduced (or per-row) loss, and the gradient
    element by element. The oracle runs on the CPU over blocks of rows
    (about 128 M elements each, so host memory stays bounded); each block's
    fp64 gradient is compared with the library's output on the GPU."""
    dev = torch.device("cuda")
    inp = make_ce_inputs(cfg, device=dev)
    x, t, w, g = inp["logits"], inp["target"], inp["weight"], inp["grad_output"]
    R, V = x.shape
    x0 = x.clone()                       # the logits, kept on the device for the tolerance terms
    x_host = x.cpu()
    w_host = None if w is None else w.cpu()
    t_host = t.cpu()
    g_host = g.cpu()
    n, wy, wall, _ = oracle.normalizers(t_host, V, IGNORE_INDEX, w_host)
    variant, tune = (variant, 0) if variant != "stream-pair" else ("stream", 8)
    loss = ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=cfg.label_smoothing, reduction=cfg.reduction,
                         grad_output=g, variant=variant, tune=tune)
    torch.cuda.synchronize()
    block = max(1, block_elems // V)
    row_loss = torch.empty(R, dtype=torch.float64)
    dxy_want = torch.zeros(R, dtype=torch.float64)
    n_bad = n_floor = 0
    worst = worst_tol = 0.0
    for r0 in range(0, R, block):
        r1 = min(R, r0 + block)
        g_rows = g_host[r0:r1] if cfg.reduction == "none" else g_host
        ref = oracle.rows(x_host[r0:r1], t_host[r0:r1], weight=w_host, label_smoothing=cfg.label_smoothing,
                          reduction=cfg.reduction, grad_output=g_rows, norm_wy=wy, w_all=wall)
        row_loss[r0:r1] = ref["row_loss"]
        tb = t_host[r0:r1]
        ok = (tb >= 0) & (tb < V)
        rr = ok.nonzero().flatten()
        dxy_want[r0 + rr] = ref["grad"][rr, tb[rr]]
        scale = row_scale(cfg.reduction, g_rows, r1 - r0, wy)
        want = ref["grad"].to(dev)
        T = magnitude_T(x0[r0:r1], tb, ref["stats"], w_host, cfg.label_smoothing, wall, scale)
        d = grad_mismatch_detail(x[r0:r1], want, T)
        n_bad, n_floor = n_bad + d["n_bad"], n_floor + d["n_floor"]
        worst, worst_tol = max(worst, d["worst_ulp"]), max(worst_tol, d["worst_tol"])
        del want, T, ref
    if cfg.reduction == "none":
        check_loss_rows(loss.cpu(), row_loss)
    else:
        check_loss_reduced(float(loss.item()), oracle.reduce(row_loss, cfg.reduction, wy))
    share = n_floor / float(R * V)
    _record({"test": "full_size", "workload": cfg.name, "variant": variant, "tune": tune, "rows": R, "vocab": V,
             "elements": R * V, "bad": n_bad, "n_floor": n_floor, "floor_share": share,
             "worst_err_over_ulp": worst, "worst_err_over_tolerance": worst_tol})
    assert n_bad == 0, f"{n_bad} gradient elements outside tolerance (worst {worst_tol:.2f} of the tolerance)"
    assert share <= FLOOR_SHARE_MAX, f"{n_floor} elements ({share:.2e}) needed the cancellation floor"
    # ignored rows are exactly zero
    ign = (t_host < 0) | (t_host >= V)
    if ign.any():
        assert torch.count_nonzero(x[ign.to(dev)]) == 0
    valid = ~ign
    got_dxy = torch.zeros(R, dtype=torch.float64)
    vr = valid.nonzero().flatten()
    got_dxy[vr] = x[vr.to(dev), t[vr.to(dev)]].double().cpu()
    return {"valid": valid, "dxy_want": dxy_want, "dxy_got": got_dxy, "n_floor": n_floor, "share": share}


@pytest.mark.parametrize("variant", ["fused", "split", "rowpass", "stream"])
def test_confident_full_size_dxy(ce, variant):
    """4096 x 32000 bf16, softmax(x_y) near 0.9 / 0.99 / 0.999: every element
    of every row against the oracle, and dx_y within 0.4% of the oracle in
    every third (the #1329 accuracy table's workload)."""
    cfg = CONFIGS["confident"]
    res = _full_size_check(ce, cfg, variant)
    rows = res["valid"].nonzero().flatten()
    want, got = res["dxy_want"][rows], res["dxy_got"][rows]
    rel = (got - want).abs() / want.abs()
    R = cfg.n_rows
    third = (R + 2) // 3
    worst = []
    for k in range(3):
        sel = (rows >= k * third) & (rows < (k + 1) * third)
        worst.append(float(rel[sel].max()))
    _record({"test": "confident_dxy", "variant": variant, "dxy_max_rel_err_per_third": worst})
    for k in range(3):
        assert worst[k] <= DXY_RTOL, f"third {k}: dx_y max rel err {worst[k]:.4%}"


@pytest.mark.parametrize("variant", ["fused", "split", "rowpass", "stream", "stream-pair"])
def test_headline_full_size(ce, variant):
    _full_size_check(ce, CONFIGS["headline"], variant)


@pytest.mark.parametrize("name", ["large_vocab", "large_vocab_none"])
def test_large_vocab_full_size(ce, name):
    _full_size_check(ce, CONFIGS[name], "auto")


def test_tiny_config(ce):
    cfg = CONFIGS["tiny"]
    inp = make_ce_inputs(cfg, device="cuda")
    x, t = inp["logits"], inp["target"]
    x_in = x.cpu()
    ref = _oracle(x, t, None, 0.0, "mean", None)
    loss = ce.ce_fwd_bwd(x, t)
    torch.cuda.synchronize()
    _check_all(x, t, None, 0.0, "mean", None, ref, loss, x_in)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", RAGGED + [(33, 32000, 32000, 0), (6, 128256, 128256, 0), (5, 24, 24, 0)],
                         ids=lambda s: f"{s[0]}x{s[1]}ld{s[2]}@{s[3]}")
@pytest.mark.parametrize("opt", ["plain", "smooth"])
@pytest.mark.parametrize("red", ["mean", "none"])
def test_forward_statistics_every_row(ce, dtype, shape, opt, red):
    """ce_forward by the stream kernel's first pass: the statistics of every
    row, ignored ones included (max and off-target exp-sum over all columns,
    x_y = 0), and the losses, against the oracle; rows that start off a
    16-byte boundary, and ignored rows whose placeholder column 0 sits in a
    row's unaligned head."""
    R, V, ld, off = shape
    seed = zlib.crc32(repr((dtype, shape, opt, red)).encode()) % 9973
    base = make_logits(R, ld + off, dtype, 2.0, seed, device="cuda")
    x = base[:, off:off + V]
    t = make_targets(R, V, 0.3, seed, device="cuda")
    t[0] = -100                                   # an ignored first row
    if R > 2:
        t[2] = 0                                  # a valid row whose target is column 0
    eps = 0.1 if opt == "smooth" else 0.0
    ref = oracle.ce(x.cpu(), t.cpu(), label_smoothing=eps, reduction=red, want_grad=False)
    loss, stats = ce.ce_forward(x, t, label_smoothing=eps, reduction=red)
    torch.cuda.synchronize()
    if red == "none":
        check_loss_rows(loss.cpu(), ref["row_loss"])
    else:
        check_loss_reduced(float(loss.item()), ref["loss"])
    st = stats.cpu().double()
    valid = t.cpu() >= 0
    assert torch.equal(st[:, 0], ref["stats"][:, 0].float().double())          # the max is exact
    assert torch.equal(st[valid, 2], ref["stats"][valid, 2].float().double())  # x_y is exact
    assert torch.all(st[~valid, 2] == 0)
    assert torch.allclose(st[:, 1], ref["stats"][:, 1], rtol=2e-5, atol=0)    # exp-sum, all columns when ignored
    # the logits are read only
    assert torch.equal(x.cpu(), make_logits(R, ld + off, dtype, 2.0, seed, device="cuda")[:, off:off + V].cpu())


@pytest.mark.parametrize("tune", [0, 1, 2, 3, 4, 8, 9, 10, 12, 15, 16, 24, 26, 48, 52, 54, 80, 86, 88, 94, 112,
                                  118, 119, 30 + 2 * 128, 86 + 4 * 128, 118 + 7 * 128, 86 + 1024,
                                  86 + 1024 + 3 * 128, 94 + 1024])
@pytest.mark.parametrize("shape", [(70, 128256), (33, 33008), (9, 256000), (5, 1000), (6, 40), (4, 24)])
def test_stream_tuning_variants(ce, tune, shape):
    """Every stream-kernel tuning combination (wide CTA, reversed second
    pass, no L2 evict-last, CTA pairs and quads, class weights through the
    shared-memory weight ring at three or two CTAs per SM, a share of the
    first pass under evict-first) against the oracle; class weights on the odd
    tunes, on 54 (a quad) and on every weight-ring tune (64 set); at V = 40
    the last CTA of a quad has no columns (the parts are 16, 16 and 8
    columns), at V = 24 the last two."""
    R, V = shape
    x = make_logits(R, V, "bf16", 1.5, 300 + tune, device="cuda")
    t = make_targets(R, V, 0.1, 300 + tune, device="cuda")
    w = make_weights(V, 300 + tune, device="cuda") if tune % 2 or tune == 54 or tune & 64 else None
    x_in = x.cpu()
    g = torch.tensor([0.37], device="cuda")
    ref = _oracle(x, t, w, 0.05, "sum", g)
    loss = ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=0.05, reduction="sum", grad_output=g,
                         variant="stream", tune=tune)
    torch.cuda.synchronize()
    _check_all(x, t, w, 0.05, "sum", g, ref, loss, x_in)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("w_offset", [0, 1, 2, 4])
@pytest.mark.parametrize("shape", [(40, 64000), (24, 128256), (12, 250000), (8, 300000), (9, 8200)])
def test_class_weight_ring_and_its_fallbacks(ce, dtype, w_offset, shape):
    """Class-weighted smoothing on the automatic path: weights starting on a
    16-byte boundary go through the shared-memory weight ring (one CTA per
    row) and give the same bits as the per-lane loads with
    the same row split; weights at a 4- or 8-byte offset take the per-lane
    loads. All against the oracle."""
    R, V = shape
    seed = zlib.crc32(repr((dtype, w_offset, shape)).encode()) % 9973
    x = make_logits(R, V, dtype, 1.5, seed, device="cuda")
    t = make_targets(R, V, 0.1, seed, device="cuda")
    wbuf = torch.empty(V + 8, dtype=torch.float32, device="cuda")
    wbuf[w_offset:w_offset + V] = make_weights(V, seed, device="cuda")
    w = wbuf[w_offset:w_offset + V]
    g = torch.tensor([0.37], device="cuda")
    x_in = x.cpu()
    ref = _oracle(x, t, w, 0.05, "sum", g)
    x2 = x.clone()
    loss = ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=0.05, reduction="sum", grad_output=g)
    torch.cuda.synchronize()
    _check_all(x, t, w, 0.05, "sum", g, ref, loss, x_in)
    if w_offset != 0:
        return
    # the per-lane-load path on the same inputs with the same row split (one CTA
    # per row): bit-identical
    tune = 16 | 4
    loss2 = ce.ce_fwd_bwd(x2, t, weight=w, label_smoothing=0.05, reduction="sum", grad_output=g, variant="stream",
                          tune=tune)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int16), x2.view(torch.int16))
    assert torch.equal(loss, loss2)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("opt", ["plain", "smooth", "weighted_smooth"])
@pytest.mark.parametrize("tune", [0, 30, 86], ids=lambda t: f"tune{t}")
def test_exponent_forms_by_row_maximum(ce, dtype, opt, tune):
    """On 16-bit rows the gradient's exponent is one FMA, x log2e + c with
    c = -log2e LSE, while |c| < 32, and subtracts the row maximum exactly
    otherwise: rows on both sides of that bound (and far beyond, either
    sign), one CTA per row, pairs and the class-weight ring, against the
    oracle."""
    if tune == 86 and opt != "weighted_smooth":
        pytest.skip("the class-weight ring serves class-weighted smoothing")
    R, V = 12, 9000
    seed = zlib.crc32(repr((dtype, opt, tune)).encode()) % 9973
    base = make_logits(R, V, "f32", 1.5, seed, device="cuda")
    offs = torch.tensor([0., 8., 10., 11., 12., 14., 20., -20., -25., -35., 300., -300.], device="cuda")
    x = (base + offs[:, None]).to(DT[dtype])
    t = make_targets(R, V, 0.1, seed, device="cuda")
    w = make_weights(V, seed, device="cuda") if opt == "weighted_smooth" else None
    eps = 0.0 if opt == "plain" else 0.1
    g = torch.tensor([0.37], device="cuda")
    c = (torch.logsumexp(x.double(), dim=1) * 1.4426950408889634).abs().cpu()
    assert bool((c < 31).any()) and bool((c > 33).any())
    x_in = x.cpu()
    ref = _oracle(x, t, w, eps, "sum", g)
    loss = ce.ce_fwd_bwd(x, t, weight=w, label_smoothing=eps, reduction="sum", grad_output=g, variant="stream",
                         tune=tune)
    torch.cuda.synchronize()
    _check_all(x, t, w, eps, "sum", g, ref, loss, x_in)


@pytest.mark.parametrize("case", ["mean", "sum_weighted", "none_ragged", "int32_ld", "one_part", "tiny"])
def test_from_host_matches_device_call(ce, case):
    """ce_fwd_bwd_from_host (row blocks copied from pinned host memory on a
    second stream, each block's kernel started when its copy lands): the same
    gradient, bit for bit, as ce_fwd_bwd on a device copy, and losses within
    the oracle's tolerances; called twice in a row on the same buffers."""
    R, V, ld, red, eps, weighted, t32, parts = {
        "mean": (300, 4096, 4096, "mean", 0.1, False, False, 8),
        "sum_weighted": (257, 3000, 3000, "sum", 0.05, True, False, 5),
        "none_ragged": (129, 1001, 1001, "none", 0.1, False, False, 7),
        "int32_ld": (64, 2000, 2011, "mean", 0.0, False, True, 3),
        "one_part": (33, 5000, 5000, "mean", 0.1, True, False, 1),
        "tiny": (3, 7, 7, "sum", 0.0, False, False, 8),
    }[case]
    dev = torch.device("cuda")
    seed = zlib.crc32(case.encode()) % 10007
    x = make_logits(R, V, "bf16", 2.0, seed, device=dev, ld=ld if ld > V else None)
    t = make_targets(R, V, 0.2, seed, device=dev)
    if t32:
        t = t.to(torch.int32)
    w = make_weights(V, seed, device=dev) if weighted else None
    g = (torch.rand(R, generator=torch.Generator().manual_seed(seed)).to(dev) if red == "none"
         else torch.tensor([0.37], device=dev))
    x_in = x.cpu()
    ref = _oracle(x, t, w, eps, red, g)
    want = torch.empty((R, ld), dtype=x.dtype, device=dev)[:, :V]   # the same layout as the call under test
    want.copy_(x)
    want_loss = ce.ce_fwd_bwd(want, t, weight=w, label_smoothing=eps, reduction=red, grad_output=g)
    host = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype).pin_memory() if ld == V else \
        torch.empty(R, ld, dtype=x.dtype).pin_memory()[:, :V]
    host.copy_(x_in)
    for _ in range(2):
        got = torch.full((R, ld), float("nan"), dtype=x.dtype, device=dev)[:, :V]
        loss = ce.ce_fwd_bwd_from_host(host, got, t, weight=w, label_smoothing=eps, reduction=red, grad_output=g,
                                       n_parts=parts)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        _check_all(got, t, w, eps, red, g, ref, loss, x_in)
        if red == "none":
            assert torch.equal(loss, want_loss)


def test_bounded_wait_gives_up_with_status_and_context_survives(ce):
    """A device wait that nothing satisfies ends after its limit with
    CE_FLAG_WAIT_TIMEOUT, and the context keeps working."""
    t0 = time.perf_counter()
    flags = ce.ce_selftest_wait_timeout(100_000_000)
    elapsed = time.perf_counter() - t0
    assert flags & ce.CE_FLAG_WAIT_TIMEOUT
    assert 0.09 <= elapsed < 5.0
    x = make_logits(8, 512, "bf16", 1.0, 1, device="cuda")
    t = make_targets(8, 512, 0.0, 1, device="cuda")
    ws = ce.workspace(8)
    ce.ce_fwd_bwd(x, t, ws=ws)
    assert ce.ce_get_status(ws) == 0


@pytest.mark.parametrize("api", ["auto", "stream-pair", "stream-wide", "stream-quad", "rowpass", "split",
                                 "fwd+bwd calls"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("red", ["mean", "sum", "none"])
@pytest.mark.parametrize("opts", [(15.0, 0.0), (0.0, 1e-4), (30.0, 1e-4), (0.0, 0.0)],
                         ids=["softcap", "zloss", "both", "accuracy"])
@pytest.mark.parametrize("shape", [(17, 1000), (9, 33000), (5, 7), (6, 1001)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_softcap_zloss_accuracy(ce, api, dtype, red, opts, shape):
    """Softcap, z-loss and token accuracy against the oracle, in the stream
    kernel (automatic path, CTA pairs, wide CTAs, clusters of four), the row
    pass and the split kernels; the token accuracy is asked for in every
    case."""
    R, V = shape
    cap, zl = opts
    seed = zlib.crc32(repr((R, V, dtype, red, opts)).encode()) % 9973
    x = make_logits(R, V, dtype, 6.0, seed, device="cuda")   # wide logits: the cap bites
    t = make_targets(R, V, 0.2, seed, device="cuda")
    t[0] = int(torch.argmax(x[0].float()))                    # at least one correct row
    w = make_weights(V, seed, device="cuda") if red == "sum" else None
    g = (torch.rand(R, generator=torch.Generator().manual_seed(seed)).to("cuda") if red == "none"
         else torch.tensor([0.37], device="cuda"))
    x_in = x.cpu()
    ref = oracle.ce(x_in, t.cpu(), weight=None if w is None else w.cpu(), label_smoothing=0.1, reduction=red,
                    grad_output=g.cpu(), softcap=cap, z_loss=zl)
    acc = torch.zeros(1, device="cuda")
    if api == "fwd+bwd calls":
        loss, stats = ce.ce_forward(x, t, weight=w, label_smoothing=0.1, reduction=red, softcap=cap, z_loss=zl,
                                    accuracy=acc)
        ce.ce_backward(x, t, stats, grad_output=g, weight=w, label_smoothing=0.1, reduction=red, softcap=cap,
                       z_loss=zl)
    else:
        variant, tune = {"stream-pair": ("stream", 8), "stream-wide": ("stream", 9),
                         "stream-quad": ("stream", 52)}.get(api, (api, 0))
        loss = ce.ce_fwd_bwd(x, t, grad_output=g, weight=w, label_smoothing=0.1, reduction=red,
                             variant=variant, tune=tune, softcap=cap, z_loss=zl, accuracy=acc)
    torch.cuda.synchronize()
    _check_all(x, t, w, 0.1, red, g, ref, loss, x_in, softcap=cap, z_loss=zl)
    assert float(acc.item()) == pytest.approx(ref["accuracy"], abs=1e-7)


def test_options_refused_where_not_implemented(ce):
    x = make_logits(4, 1024, "bf16", 1.0, 1, device="cuda")
    t = make_targets(4, 1024, 0.0, 1, device="cuda")
    with pytest.raises(ce.CEError, match="UNSUPPORTED"):
        ce.ce_fwd_bwd(x, t, variant="fused", softcap=10.0)


@pytest.mark.parametrize("variant", ["auto", "fused", "split", "rowpass", "stream", "stream-pair"])
@pytest.mark.parametrize("V", [1000, 33000, 128256])
def test_nothing_written_past_the_buffer(ce, variant, V):
    """The logits sit at the start of a larger allocation whose tail holds a
    canary pattern; after the call the canary is intact (no write past
    n_rows x ld)."""
    R = 7
    canary_len = 1 << 16
    base = make_logits(1, R * V + canary_len, "bf16", 1.0, 55, device="cuda").reshape(-1)
    base[R * V:] = 123.0
    x = base[:R * V].view(R, V)
    t = make_targets(R, V, 0.0, 55, device="cuda")
    var, tune = (variant, 0) if variant != "stream-pair" else ("stream", 8)
    ce.ce_fwd_bwd(x, t, label_smoothing=0.1, variant=var, tune=tune)
    torch.cuda.synchronize()
    assert torch.all(base[R * V:] == 123.0)
