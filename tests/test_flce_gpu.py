"""Tensor-core GEMM and fused-linear cross-entropy on the GPU.

The GEMM is checked against a float64 matmul of the same bf16 operands in
all four operand layouts; the fused-linear path against the fp64 oracle
(float64 matmul + the row oracle). Tolerances come from the arithmetic:
the GEMMs accumulate exact bf16 products in fp32; dZ is rounded once to
bf16 (relative error <= 2^-9 per element) before the two gradient GEMMs,
so |error| <= 2^-8 * sum |dZ| |operand| (factor 2 margin) plus one output
rounding."""
import pytest
import torch

import oracle
from workloads import FLCE_CONFIGS, make_flce_inputs, make_targets

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ce():
    assert torch.cuda.is_available()
    import softmax_cross_entropy_pass_gb300 as ce
    return ce


def _rand_bf16(*shape, seed=0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("shape", [(128, 256, 64), (200, 296, 136), (1024, 2048, 1024), (384, 512, 4096),
                                   (520, 776, 200), (2048, 1536, 2112)])
def test_gemm_layouts_against_float64(ce, a_mn, b_mn, shape):
    """M and N both >= 512 take the CTA-pair kernel (256 x 256 tiles), the
    others one CTA per 128 x 256 tile."""
    M, N, K = shape
    A = _rand_bf16(M, K, seed=1)                # logical [M, K]
    B = _rand_bf16(N, K, seed=2)                # logical [N, K] (B^T)
    ref = A.double() @ B.double().T
    A_mem = (A.T.contiguous() if a_mn else A).cuda()
    B_mem = (B.T.contiguous() if b_mn else B).cuda()
    D = ce.ce_gemm_bf16(A_mem, B_mem, a_mn_major=a_mn, b_mn_major=b_mn)
    torch.cuda.synchronize()
    bound = (A.double().abs() @ B.double().abs().T) * (K * 2.0 ** -23) + 1e-30
    err = (D.double().cpu() - ref).abs()
    assert (err <= bound).all(), f"max err {float(err.max()):.3e}"


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (768, 1024, 320)])
def test_gemm_bias_accumulate_and_bf16_out(ce, M, N, K):
    A = _rand_bf16(M, K, seed=3).cuda()
    B = _rand_bf16(N, K, seed=4).cuda()
    bias = torch.randn(N, device="cuda")
    ref = A.double() @ B.double().T
    D = ce.ce_gemm_bf16(A, B, bias=bias)
    assert torch.allclose(D.double(), ref + bias.double(), rtol=1e-5, atol=1e-3)
    ce.ce_gemm_bf16(A, B, out=D, out_kind=ce.CE_GEMM_F32_ACCUM)
    assert torch.allclose(D.double(), 2 * ref + bias.double(), rtol=1e-5, atol=2e-3)
    Db = ce.ce_gemm_bf16(A, B, out_kind=ce.CE_GEMM_BF16_STORE)
    assert torch.equal(Db, ref.float().to(torch.bfloat16)) or \
        ((Db.double() - ref).abs() <= ref.abs() * 2.0 ** -8 + 1e-3).all()


def _flce_check(out, ref, hidden, weight, rows, cols, dz_abs_rows=None):
    loss, gh, gw, gb = out
    # loss: bf16 operands exact, fp32 GEMM accumulation and fp32 CE
    if ref["loss"] is not None and not torch.is_tensor(ref["loss"]):
        assert abs(float(loss.item()) - ref["loss"]) <= 1e-4 * abs(ref["loss"])
    return loss, gh, gw, gb


@pytest.mark.parametrize("reduction", ["mean", "sum"])
@pytest.mark.parametrize("chunk", [128, 1000])
@pytest.mark.parametrize("with_bias", [False, True])
def test_flce_small_against_oracle(ce, reduction, chunk, with_bias):
    cfg = FLCE_CONFIGS["flce_small"]
    inp = make_flce_inputs(cfg, device="cuda")
    h, W, t = inp["hidden"], inp["weight"], inp["target"]
    BT, H = h.shape
    V = W.shape[0]
    bias = (torch.randn(V, generator=torch.Generator().manual_seed(9)) * 0.1).cuda() if with_bias else None
    eps = 0.05
    loss, gh, gw, gb = ce.flce_fwd_bwd(h, W, t, bias=bias, label_smoothing=eps, reduction=reduction,
                                        chunk_rows=chunk)
    torch.cuda.synchronize()
    ref = oracle.flce(h.cpu(), W.cpu(), t.cpu(), bias=None if bias is None else bias.cpu(),
                      label_smoothing=eps, reduction=reduction)
    assert abs(float(loss.item()) - ref["loss"]) <= 1e-4 * abs(ref["loss"])
    # dZ (oracle, fp64) for the error bounds
    z = h.double().cpu() @ W.double().cpu().T + (0 if bias is None else bias.double().cpu())
    dz = oracle.rows(z, t.cpu(), label_smoothing=eps, reduction=reduction, norm_wy=ref["norm_wy"],
                     want_stats=False)["grad"]
    bound_h = (dz.abs() @ W.double().cpu().abs()) * 2.0 ** -8 + 1e-30
    ref_h = ref["grad_hidden"]
    err_h = (gh.double().cpu() - ref_h).abs()
    ulp_h = ref_h.abs() * 2.0 ** -7
    assert (err_h <= bound_h + ulp_h).all(), f"grad_hidden max err {float(err_h.max()):.3e}"
    bound_w = (dz.abs().T @ h.double().cpu().abs()) * 2.0 ** -8 + 1e-30
    err_w = (gw.double().cpu() - ref["grad_weight"]).abs()
    assert (err_w <= bound_w + ref["grad_weight"].abs() * 2.0 ** -20).all(), \
        f"grad_weight max err {float(err_w.max()):.3e}"
    if with_bias:
        err_b = (gb.double().cpu() - ref["grad_bias"]).abs()
        assert (err_b <= dz.abs().sum(0) * 2.0 ** -8 + 1e-30).all()


def _ignored_case(case, BT, V):
    """Targets, reduction, chunk rows, label smoothing, class weights and
    grad_output of one ignored-row case (seeded)."""
    seeds = {"mixed": 21, "all_ignored": 22, "mostly_ignored": 23, "none_rows": 24, "int32_out_of_range": 25}
    g = torch.Generator().manual_seed(seeds[case])
    t = torch.randint(0, V, (BT,), generator=g)
    perm = torch.randperm(BT, generator=g)
    red, chunk, eps, weighted, go = "mean", 128, 0.0, False, None
    if case == "mixed":          # 5% ignored, valid count not a multiple of 64
        t[perm[:27]] = -100
    elif case == "all_ignored":
        t[:] = -100
        chunk = 200
    elif case == "mostly_ignored":  # whole chunks past the valid count
        t[perm[:int(0.8 * BT)]] = -100
        red, chunk = "sum", 64
        go = torch.tensor([0.37])
    elif case == "none_rows":    # per-row loss and grad_output, weights, smoothing
        t[perm[:int(0.3 * BT)]] = -100
        red, chunk, eps, weighted = "none", 100, 0.1, True
        go = torch.rand(BT, generator=g)
    elif case == "int32_out_of_range":
        t[perm[:40]] = -100
        t[perm[40]] = V + 5
        t = t.to(torch.int32)
    w = (torch.rand(V, generator=g) + 0.5) if weighted else None
    return t, red, chunk, eps, w, go


@pytest.mark.parametrize("ce_cluster", [False, True], ids=["stats_map", "cluster"])
@pytest.mark.parametrize("dense", [False, True], ids=["compact", "dense"])
@pytest.mark.parametrize("case", ["mixed", "all_ignored", "mostly_ignored", "none_rows", "int32_out_of_range"])
def test_flce_ignored_rows_against_oracle(ce, case, dense, ce_cluster):
    """Ignored (and out-of-range) rows, with and without the device-side
    compaction of the valid rows, and with either chunk cross-entropy (the
    logits GEMM's row statistics + streaming map, or the cluster kernel):
    every output against the fp64 oracle with the dZ-rounding bound;
    workspace and outputs start as NaN so nothing a kernel skips can leak
    into a result. V = 1000 leaves a ragged last column tile (232 columns)."""
    BT, H, V = 520, 128, 1000
    h = _rand_bf16(BT, H, seed=11)
    W = _rand_bf16(V, H, seed=12, scale=0.05)
    t, red, chunk, eps, w, go = _ignored_case(case, BT, V)
    bias = (torch.randn(V, generator=torch.Generator().manual_seed(13)) * 0.2) if case == "mixed" else None
    dev = "cuda"
    ws = torch.full((ce.flce_workspace_size(BT, H, V, chunk, dense, ce_cluster),), 0xFF, dtype=torch.uint8,
                    device=dev)
    loss = torch.full((BT if red == "none" else 1,), float("nan"), device=dev)
    gh = torch.full((BT, H), float("nan"), dtype=torch.bfloat16, device=dev)
    gw = torch.full((V, H), float("nan"), device=dev)
    gb = torch.full((V,), float("nan"), device=dev) if bias is not None else None
    out = ce.flce_fwd_bwd(h.to(dev), W.to(dev), t.to(dev), bias=None if bias is None else bias.to(dev),
                          class_weight=None if w is None else w.to(dev),
                          label_smoothing=eps, reduction=red, grad_output=None if go is None else go.to(dev),
                          chunk_rows=chunk, loss=loss, grad_hidden=gh, grad_weight=gw, grad_bias=gb, ws=ws,
                          dense=dense, ce_cluster=ce_cluster)
    flags = ce.ce_get_status(ws)
    ref = oracle.flce(h, W, t, bias=bias, label_smoothing=eps, reduction=red, class_weight=w, grad_output=go,
                      abs_sums=True)
    want_flags = (ce.CE_FLAG_TARGET_OUT_OF_RANGE if case == "int32_out_of_range" else 0) | \
        (ce.CE_FLAG_NO_VALID_ROWS if case == "all_ignored" and red == "mean" else 0)
    assert flags == want_flags, f"status flags {flags:#x}, expected {want_flags:#x}"
    loss_c = out[0].double().cpu()
    if red == "none":
        err = (loss_c - ref["loss"]).abs()
        assert (err <= 1e-4 * ref["loss"].abs() + 1e-6).all(), f"row losses: max err {float(err.max()):.3e}"
    else:
        assert abs(float(loss_c[0]) - ref["loss"]) <= 1e-4 * abs(ref["loss"]) + 1e-30
    gh_c = gh.double().cpu()
    gw_c = gw.double().cpu()
    assert torch.isfinite(gh_c).all() and torch.isfinite(gw_c).all()
    err_h = (gh_c - ref["grad_hidden"]).abs()
    assert (err_h <= ref["grad_hidden_abs"] * 2.0 ** -8 + ref["grad_hidden"].abs() * 2.0 ** -7).all(), \
        f"grad_hidden max err {float(err_h.max()):.3e}"
    err_w = (gw_c - ref["grad_weight"]).abs()
    assert (err_w <= ref["grad_weight_abs"] * 2.0 ** -8 + ref["grad_weight"].abs() * 2.0 ** -20).all(), \
        f"grad_weight max err {float(err_w.max()):.3e}"
    if bias is not None:
        z = h.double() @ W.double().T + bias.double()
        dz = oracle.rows(z, t, label_smoothing=eps, reduction=red, norm_wy=ref["norm_wy"], want_stats=False)["grad"]
        err_b = (gb.double().cpu() - ref["grad_bias"]).abs()
        assert (err_b <= dz.abs().sum(0) * 2.0 ** -8 + 1e-30).all(), f"grad_bias max err {float(err_b.max()):.3e}"
    tt = t.to(torch.int64)
    skipped = (tt < 0) | (tt >= V)
    assert torch.count_nonzero(gh_c[skipped]) == 0
    if red == "none":
        assert torch.count_nonzero(loss_c[skipped]) == 0


@pytest.mark.parametrize("opts", [(15.0, 0.0), (0.0, 1e-4), (30.0, 1e-4)], ids=["softcap", "zloss", "both"])
@pytest.mark.parametrize("red", ["mean", "none"])
@pytest.mark.parametrize("dense", [False, True], ids=["compact", "dense"])
def test_flce_softcap_zloss_accuracy(ce, opts, red, dense):
    """Softcap (applied to the GEMM's logits), z-loss and token accuracy in
    the fused-linear path against the fp64 oracle; the bound on the
    gradients is the bf16 rounding of dZ, as for the plain path."""
    cap, zl = opts
    BT, H, V = 300, 128, 1000
    h = _rand_bf16(BT, H, seed=41)
    W = _rand_bf16(V, H, seed=42, scale=0.3)          # logits of a few units: the cap bites
    t = make_targets(BT, V, 0.1, 43)
    am = (h.double() @ W.double().T).argmax(dim=1)
    t[:40] = am[:40]                                    # some correct rows
    g = torch.rand(BT, generator=torch.Generator().manual_seed(44)) if red == "none" else None
    acc = torch.full((1,), float("nan"), device="cuda")
    loss, gh, gw, _ = ce.flce_fwd_bwd(h.cuda(), W.cuda(), t.cuda(), label_smoothing=0.1, reduction=red,
                                      grad_output=None if g is None else g.cuda(), chunk_rows=128, dense=dense,
                                      softcap=cap, z_loss=zl, accuracy=acc)
    torch.cuda.synchronize()
    ref = oracle.flce(h, W, t, label_smoothing=0.1, reduction=red, grad_output=g, softcap=cap, z_loss=zl,
                      abs_sums=True)
    if red == "none":
        err = (loss.double().cpu() - ref["loss"]).abs()
        assert (err <= 1e-4 * ref["loss"].abs() + 1e-6).all()
    else:
        assert abs(float(loss.item()) - ref["loss"]) <= 1e-4 * abs(ref["loss"])
    err_h = (gh.double().cpu() - ref["grad_hidden"]).abs()
    assert (err_h <= ref["grad_hidden_abs"] * 2.0 ** -8 + ref["grad_hidden"].abs() * 2.0 ** -7).all(), \
        f"grad_hidden max err {float(err_h.max()):.3e}"
    err_w = (gw.double().cpu() - ref["grad_weight"]).abs()
    assert (err_w <= ref["grad_weight_abs"] * 2.0 ** -8 + ref["grad_weight"].abs() * 2.0 ** -20).all(), \
        f"grad_weight max err {float(err_w.max()):.3e}"
    assert float(acc.item()) == pytest.approx(ref["accuracy"], abs=1e-7)


def test_flce_options_refused_with_the_cluster_chunk_kernel(ce):
    h = _rand_bf16(64, 64, seed=1).cuda()
    W = _rand_bf16(256, 64, seed=2).cuda()
    t = make_targets(64, 256, 0.0, 3, device="cuda")
    with pytest.raises(ce.CEError, match="UNSUPPORTED"):
        ce.flce_fwd_bwd(h, W, t, ce_cluster=True, softcap=10.0)


@pytest.mark.slow
def test_flce_grad_hidden_without_split_k(ce):
    """A chunk whose grad_hidden GEMM has 2048 output tiles (16384 rows x H
    4096) takes one product per tile (no split-K) and stores bf16 rows
    through the compaction's row map in the GEMM epilogue: sampled rows and
    vocabulary rows against the fp64 oracle."""
    BT, H, V = 16384, 4096, 1024
    g = torch.Generator(device="cuda").manual_seed(31)
    h = torch.randn(BT, H, generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    t = make_targets(BT, V, 0.05, 31, device="cuda")
    loss, gh, gw, _ = ce.flce_fwd_bwd(h, W, t, reduction="mean", chunk_rows=BT)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(32)
    rows = torch.randperm(BT, generator=gen)[:128].sort().values
    cols = torch.randperm(V, generator=gen)[:64].sort().values
    ref = oracle.flce(h.cpu(), W.cpu(), t.cpu(), reduction="mean", sample_rows=rows, sample_cols=cols,
                      abs_sums=True)
    assert abs(float(loss.item()) - ref["loss"]) <= 1e-4 * abs(ref["loss"])
    gh_s = gh[rows.cuda()].double().cpu()
    err_h = (gh_s - ref["grad_hidden"]).abs()
    assert (err_h <= ref["grad_hidden_abs"] * 2.0 ** -8 + ref["grad_hidden"].abs() * 2.0 ** -7).all()
    gw_s = gw[cols.cuda()].double().cpu()
    err_w = (gw_s - ref["grad_weight"]).abs()
    assert (err_w <= ref["grad_weight_abs"] * 2.0 ** -8 + ref["grad_weight"].abs() * 2.0 ** -20).all()
    valid = t.cpu()[rows] >= 0
    assert torch.count_nonzero(gh_s[~valid]) == 0


@pytest.mark.slow
def test_flce_full_size_sampled(ce):
    """hidden 8192 x 4096, W 128256 x 4096: loss over all rows, grad_hidden on
    256 sampled rows and grad_weight on 256 sampled vocabulary rows against
    the fp64 oracle, with the same rounding bound as the small cases
    (dZ rounded once to bf16: |error| <= 2^-8 sum |dZ| |operand|)."""
    cfg = FLCE_CONFIGS["flce"]
    inp = make_flce_inputs(cfg, device="cuda")
    h, W, t = inp["hidden"], inp["weight"], inp["target"]
    loss, gh, gw, _ = ce.flce_fwd_bwd(h, W, t, reduction="mean", chunk_rows=2048)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(77)
    rows = torch.randperm(cfg.n_rows, generator=gen)[:256].sort().values
    cols = torch.randperm(cfg.vocab, generator=gen)[:256].sort().values
    ref = oracle.flce(h.cpu(), W.cpu(), t.cpu(), reduction="mean", sample_rows=rows, sample_cols=cols,
                      abs_sums=True)
    assert abs(float(loss.item()) - ref["loss"]) <= 1e-4 * abs(ref["loss"])
    gh_s = gh[rows.cuda()].double().cpu()
    gw_s = gw[cols.cuda()].double().cpu()
    err_h = (gh_s - ref["grad_hidden"]).abs()
    bound_h = ref["grad_hidden_abs"] * 2.0 ** -8 + ref["grad_hidden"].abs() * 2.0 ** -7
    assert (err_h <= bound_h).all(), f"grad_hidden: {int((err_h > bound_h).sum())} elements off"
    err_w = (gw_s - ref["grad_weight"]).abs()
    bound_w = ref["grad_weight_abs"] * 2.0 ** -8 + ref["grad_weight"].abs() * 2.0 ** -20
    assert (err_w <= bound_w).all(), f"grad_weight: {int((err_w > bound_w).sum())} elements off"
    valid = t.cpu()[rows] >= 0
    assert torch.count_nonzero(gh_s[~valid]) == 0
