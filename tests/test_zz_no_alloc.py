"""ce_fwd_bwd_noalloc, the entry point for callers that cannot allocate
device memory (hosts that give their extensions no allocator, such as a
runtime that keeps all device memory in its own pool), against the workspace
entry point ce_fwd_bwd: calls in a row through the C ABI, with different
shapes, reductions, class weights and smoothing, so each call runs on
scratch that still holds the previous call's contents. The two entry points
run the same kernels on the same inputs and every reduction is in a fixed
order, so their outputs must be bit-identical. This file is collected last."""
import pytest
import torch

from workloads import make_logits, make_targets, make_weights

pytestmark = pytest.mark.gpu


def _pair(ce, R, V, reduction, eps, seed, variant, weighted):
    x = make_logits(R, V, "bf16", 1.0, seed, device="cuda")
    t = make_targets(R, V, 0.1, seed, device="cuda")
    w = make_weights(V, seed, device="cuda") if weighted else None
    g = torch.rand(R, device="cuda") if reduction == "none" else torch.tensor([0.37], device="cuda")
    xa, xb = x.clone(), x.clone()
    la = ce.ce_fwd_bwd(xa, t, grad_output=g, weight=w, label_smoothing=eps, reduction=reduction, variant=variant)
    lb = torch.full_like(la, float("nan"))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    ce.ce_fwd_bwd_noalloc(xb, t, grad_output=g, weight=w, label_smoothing=eps, reduction=reduction,
                          variant=variant, loss=lb)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    return la, lb, xa, xb, free0 - free1


def _first_call_setup(ce):
    """The first call in a process looks up the scratch array's device
    address; the CUDA driver may place the array (its module) in device memory
    then. Later calls must not change device memory in use."""
    x = make_logits(4, 64, "bf16", 1.0, 1, device="cuda")
    t = make_targets(4, 64, 0.0, 1, device="cuda")
    ce.ce_fwd_bwd_noalloc(x, t)
    torch.cuda.synchronize()


@pytest.mark.parametrize("variant", ["auto", "split", "rowpass"])
def test_noalloc_matches_workspace_entry_bitwise(variant):
    import softmax_cross_entropy_pass_gb300 as ce
    _first_call_setup(ce)
    cases = [(3000, 32000, "mean", 0.1, 11, False), (700, 50000, "sum", 0.0, 12, False),
             (257, 4096, "none", 0.05, 13, False),
             # class-weighted and smoothed, after batches of other sizes: the
             # scratch still holds their normalisers and row losses
             (1500, 20000, "mean", 0.1, 14, True), (1500, 20000, "mean", 0.1, 14, True),
             (64, 1024, "sum", 0.2, 15, True)]
    for R, V, red, eps, seed, weighted in cases:
        la, lb, xa, xb, grown = _pair(ce, R, V, red, eps, seed, variant, weighted)
        assert torch.equal(lb, la), (R, V, red, weighted, float((lb - la).abs().max()))
        assert torch.equal(xb, xa), (R, V, red, weighted)
        assert grown == 0, f"device memory in use grew by {grown} bytes during the call"


def test_noalloc_rejects_prepared_variant():
    import softmax_cross_entropy_pass_gb300 as ce
    x = make_logits(16, 100, "bf16", 1.0, 21, device="cuda")
    t = make_targets(16, 100, 0.0, 21, device="cuda")
    loss = torch.full((1,), 3.0, device="cuda")
    with pytest.raises(ce.CEError, match="INVALID_ARG"):
        ce.ce_fwd_bwd_noalloc(x, t, loss=loss, variant=ce.CE_VARIANT_PREPARED)
    torch.cuda.synchronize()
    assert float(loss.item()) == 3.0


def test_noalloc_rejects_too_many_rows_without_launching():
    import softmax_cross_entropy_pass_gb300 as ce
    R = ce.CE_NOALLOC_MAX_ROWS + 1
    x = torch.zeros(R, 8, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(R, dtype=torch.int64, device="cuda")
    loss = torch.full((1,), 3.0, device="cuda")
    with pytest.raises(ce.CEError, match="WORKSPACE"):
        ce.ce_fwd_bwd_noalloc(x, t, loss=loss)
    torch.cuda.synchronize()
    assert float(loss.item()) == 3.0
