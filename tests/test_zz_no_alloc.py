"""ce_fwd_bwd_noalloc, the entry point for callers that cannot allocate
device memory (hosts that give their extensions no allocator), against the
workspace entry point ce_fwd_bwd: two calls in a row through the C ABI,
different shapes and reductions, so the second call runs on scratch that
still holds the first call's contents. This file is collected last."""
import pytest
import torch

from workloads import make_logits, make_targets

pytestmark = pytest.mark.gpu


def _pair(ce, R, V, reduction, eps, seed, variant):
    x = make_logits(R, V, "bf16", 1.0, seed, device="cuda")
    t = make_targets(R, V, 0.1, seed, device="cuda")
    g = torch.rand(R, device="cuda") if reduction == "none" else torch.tensor([0.37], device="cuda")
    xa, xb = x.clone(), x.clone()
    la = ce.ce_fwd_bwd(xa, t, grad_output=g, label_smoothing=eps, reduction=reduction, variant=variant)
    lb = ce.ce_fwd_bwd_noalloc(xb, t, grad_output=g, label_smoothing=eps, reduction=reduction, variant=variant)
    torch.cuda.synchronize()
    return la, lb, xa, xb


@pytest.mark.parametrize("variant", ["auto", "split"])
def test_noalloc_matches_workspace_entry_twice(variant):
    import softmax_cross_entropy_pass_gb300 as ce
    cases = [(3000, 32000, "mean", 0.1, 11), (700, 50000, "sum", 0.0, 12), (257, 4096, "none", 0.05, 13)]
    for R, V, red, eps, seed in cases:
        la, lb, xa, xb = _pair(ce, R, V, red, eps, seed, variant)
        # same kernels, same inputs: the loss within the reduced-loss tolerance
        # of the parity tests (1e-6 relative), the gradient within 1 bf16 ulp
        assert torch.allclose(lb, la, rtol=1e-6, atol=0), (red, float((lb - la).abs().max()))
        diff = (xb.float() - xa.float()).abs()
        assert (diff <= xa.float().abs() * 2.0 ** -7).all()


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
