"""GB300 (sm_103a) fused softmax cross-entropy: Python binding of libce.so.

Thin ctypes layer over the C ABI in include/ce.h. It only marshals
arguments: device pointers from torch tensors, the current CUDA stream, and
workspace memory allocated through torch. Every step of the computation
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback,
and importing this package fails if the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).

Entry points (same names as the C ABI):
  ce_forward(logits, target, ...)            -> (loss, stats)
  ce_backward(logits, target, stats, ...)    gradient written over logits
  ce_fwd_bwd(logits, target, ...)            -> loss; gradient over logits
  ce_scale_grad(grad, grad_output, ...)      in-place grad_output scaling
  ce_workspace_size / ce_fused_plan / ce_get_status
and ``cross_entropy``: a torch.autograd entry with two modes.
``CrossEntropyFunction`` computes the gradient in the forward (in place) and
scales it by grad_output in the backward, with a device-side skip when
grad_output is 1 (one logits read and write; a second rounding when
grad_output is not 1). ``CrossEntropyExactFunction`` saves the row
statistics in the forward and forms the gradient in the backward with
grad_output applied before the one rounding (the logits read twice).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libce.so")

CE_OK, CE_ERR_INVALID_ARG, CE_ERR_UNSUPPORTED, CE_ERR_CUDA, CE_ERR_WORKSPACE = 0, 1, 2, 3, 4
CE_RED = {"none": 0, "mean": 1, "sum": 2}
CE_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
CE_FLAG_TARGET_OUT_OF_RANGE, CE_FLAG_NO_VALID_ROWS, CE_FLAG_WAIT_TIMEOUT = 1, 2, 4
VARIANTS = {"auto": 0, "split": 1, "fused": 2, "rowpass": 3, "stream": 4}
CE_VARIANT_PREPARED = 0x10000


class CEError(RuntimeError):
    pass


class ce_params(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("vocab", ctypes.c_int64), ("ld", ctypes.c_int64),
                ("ignore_index", ctypes.c_int64), ("class_weight", ctypes.c_void_p),
                ("label_smoothing", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("reduction", ctypes.c_int32), ("target_is_int32", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("z_loss", ctypes.c_float), ("accuracy", ctypes.c_void_p)]


assert ctypes.sizeof(ce_params) == 80


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libce.so is not built ({LIB_PATH}); run softmax_cross_entropy_pass_gb300._build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(ce_params)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    sigs = {
        "ce_version": (ctypes.c_char_p, []),
        "ce_status_string": (ctypes.c_char_p, [st]),
        "ce_last_cuda_error": (ctypes.c_char_p, []),
        "ce_workspace_size": (st, [P, ctypes.POINTER(sz)]),
        "ce_prepare": (st, [P, vp, vp, sz, vp]),
        "ce_forward": (st, [P, vp, vp, vp, vp, vp, sz, vp]),
        "ce_backward": (st, [P, vp, vp, vp, vp, vp, sz, vp]),
        "ce_fwd_bwd": (st, [P, vp, vp, vp, vp, vp, sz, vp]),
        "ce_fwd_bwd_noalloc": (st, [P, vp, vp, vp, vp, vp]),
        "ce_fwd_bwd_from_host": (st, [P, vp, vp, vp, vp, vp, vp, sz, vp, vp, ctypes.c_int32]),
        "ce_scale_grad": (st, [P, vp, vp, vp]),
        "ce_fused_plan": (st, [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                               ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]),
        "ce_get_status": (st, [vp, ctypes.POINTER(ctypes.c_uint32), vp]),
        "ce_select_variant": (st, [P, vp, ctypes.POINTER(ctypes.c_int32)]),
        "ce_selftest_wait_timeout": (st, [ctypes.c_uint64, vp, vp]),
        "ce_gemm_bf16": (st, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int64, ctypes.c_int32,
                              vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp, ctypes.c_int64, vp, vp]),
        "flce_workspace_size": (st, [P, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(sz)]),
        "flce_fwd_bwd": (st, [P, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, sz, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def version() -> str:
    return _lib.ce_version().decode()


def _check(status: int, what: str):
    if status != CE_OK:
        msg = _lib.ce_status_string(status).decode()
        if status == CE_ERR_CUDA:
            msg += " (" + _lib.ce_last_cuda_error().decode() + ")"
        raise CEError(f"{what}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_params(logits: torch.Tensor, target: torch.Tensor, *, weight=None, ignore_index: int = -100,
                label_smoothing: float = 0.0, reduction: str = "mean", variant="auto",
                cluster: int = 0, tune: int = 0, softcap: float = 0.0, z_loss: float = 0.0,
                accuracy=None) -> ce_params:
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D tensor with unit column stride")
    if logits.dtype not in CE_DT:
        raise TypeError(f"unsupported logits dtype {logits.dtype}")
    if target.dtype not in (torch.int64, torch.int32):
        raise TypeError("target must be int64 or int32")
    n, v = logits.shape
    if target.numel() != n:
        raise ValueError("target must have one entry per row")
    if weight is not None and (weight.dtype != torch.float32 or weight.numel() != v or not weight.is_contiguous()):
        raise ValueError("weight must be a contiguous fp32 tensor of vocab entries")
    p = ce_params()
    p.n_rows, p.vocab = n, v
    p.ld = logits.stride(0) if n > 1 else v
    p.ignore_index = ignore_index
    p.class_weight = weight.data_ptr() if weight is not None else None
    p.label_smoothing = float(label_smoothing)
    p.dtype = CE_DT[logits.dtype]
    p.reduction = CE_RED[reduction]
    p.target_is_int32 = 1 if target.dtype == torch.int32 else 0
    p.variant = ((VARIANTS[variant] if isinstance(variant, str) else int(variant)) | (int(cluster) << 8)
                 | (int(tune) << 20))
    p.reserved = 0
    p.softcap = float(softcap)
    p.z_loss = float(z_loss)
    if accuracy is not None:
        if accuracy.dtype != torch.float32 or not accuracy.is_cuda:
            raise ValueError("accuracy must be a device fp32 tensor")
        p.accuracy = accuracy.data_ptr()
    return p


def ce_workspace_size(n_rows: int) -> int:
    p = ce_params()
    p.n_rows, p.vocab, p.ld = n_rows, 1, 1
    out = ctypes.c_size_t()
    _check(_lib.ce_workspace_size(ctypes.byref(p), ctypes.byref(out)), "ce_workspace_size")
    return out.value


def workspace(n_rows: int, device=None) -> torch.Tensor:
    """Workspace tensor for n_rows (device memory from torch's allocator)."""
    nbytes = ce_workspace_size(n_rows)
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws(ws, n_rows, device):
    if ws is None:
        ws = workspace(n_rows, device)
    return ws, ws.numel() * ws.element_size()


def _check_dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must live on the GPU")


def ce_prepare(logits, target, *, weight=None, ignore_index=-100, label_smoothing=0.0,
               reduction="mean", ws=None, stream=None):
    """Batch normalisers into a workspace; later calls on it may pass prepared=True."""
    _check_dev(logits, target, weight)
    p = make_params(logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction)
    ws, wsb = _ws(ws, logits.shape[0], logits.device)
    _check(_lib.ce_prepare(ctypes.byref(p), _ptr(target), _ptr(ws), wsb, _stream(stream)), "ce_prepare")
    return ws


def ce_forward(logits, target, *, weight=None, ignore_index=-100, label_smoothing=0.0,
               reduction="mean", stats=None, loss=None, ws=None, stream=None, softcap=0.0, z_loss=0.0,
               accuracy=None):
    """Loss and per-row statistics [n_rows, 4] (m, off-target exp-sum, x_y, smoothing sum)."""
    _check_dev(logits, target, weight)
    p = make_params(logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction, softcap=softcap, z_loss=z_loss,
                    accuracy=accuracy)
    n = logits.shape[0]
    if loss is None:
        loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=logits.device)
    if stats is None:
        stats = torch.empty(n, 4, dtype=torch.float32, device=logits.device)
    ws, wsb = _ws(ws, n, logits.device)
    _check(_lib.ce_forward(ctypes.byref(p), _ptr(logits), _ptr(target), _ptr(loss), _ptr(stats),
                           _ptr(ws), wsb, _stream(stream)), "ce_forward")
    return loss, stats


def ce_backward(logits, target, stats, *, grad_output=None, weight=None, ignore_index=-100,
                label_smoothing=0.0, reduction="mean", ws=None, stream=None, softcap=0.0, z_loss=0.0):
    """Writes the gradient over ``logits`` (in place) and returns it."""
    _check_dev(logits, target, stats, grad_output, weight)
    p = make_params(logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction, softcap=softcap, z_loss=z_loss)
    ws, wsb = _ws(ws, logits.shape[0], logits.device)
    _check(_lib.ce_backward(ctypes.byref(p), _ptr(logits), _ptr(target), _ptr(stats),
                            _ptr(grad_output), _ptr(ws), wsb, _stream(stream)), "ce_backward")
    return logits


def ce_fwd_bwd(logits, target, *, grad_output=None, weight=None, ignore_index=-100,
               label_smoothing=0.0, reduction="mean", variant="auto", cluster=0, loss=None,
               ws=None, stream=None, prepared=False, tune=0, softcap=0.0, z_loss=0.0, accuracy=None):
    """Loss; the gradient (times grad_output, or 1) is written over ``logits``.
    ``prepared``: ``ws`` already holds this batch's normalisers (ce_prepare)."""
    _check_dev(logits, target, grad_output, weight)
    p = make_params(logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction, variant=variant,
                    cluster=cluster, tune=tune, softcap=softcap, z_loss=z_loss, accuracy=accuracy)
    if prepared:
        if ws is None:
            raise ValueError("prepared=True needs the prepared workspace")
        p.variant |= CE_VARIANT_PREPARED
    n = logits.shape[0]
    if loss is None:
        loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=logits.device)
    ws, wsb = _ws(ws, n, logits.device)
    _check(_lib.ce_fwd_bwd(ctypes.byref(p), _ptr(logits), _ptr(target), _ptr(loss),
                           _ptr(grad_output), _ptr(ws), wsb, _stream(stream)), "ce_fwd_bwd")
    return loss


CE_NOALLOC_MAX_ROWS = 65536


def ce_fwd_bwd_noalloc(logits, target, *, grad_output=None, weight=None, ignore_index=-100,
                       label_smoothing=0.0, reduction="mean", variant="auto", loss=None, stream=None):
    """ce_fwd_bwd without a workspace: for callers that cannot allocate device
    memory, the library uses its own fixed scratch (n_rows <= CE_NOALLOC_MAX_ROWS).
    Calls whose GPU work overlaps race on that scratch: keep them on one stream."""
    _check_dev(logits, target, grad_output, weight)
    p = make_params(logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction, variant=variant)
    if loss is None:
        loss = torch.empty(logits.shape[0] if reduction == "none" else 1, dtype=torch.float32,
                           device=logits.device)
    _check(_lib.ce_fwd_bwd_noalloc(ctypes.byref(p), _ptr(logits), _ptr(target), _ptr(loss),
                                   _ptr(grad_output), _stream(stream)), "ce_fwd_bwd_noalloc")
    return loss


def ce_fwd_bwd_from_host(host_logits, dev_logits, target, *, grad_output=None, weight=None, ignore_index=-100,
                         label_smoothing=0.0, reduction="mean", loss=None, ws=None, stream=None,
                         copy_stream=None, n_parts=8):
    """ce_fwd_bwd for logits in (page-locked) host memory: the rows are copied
    into ``dev_logits`` (same shape and strides) in ``n_parts`` blocks on
    ``copy_stream`` while each block's forward + backward runs on ``stream``;
    ``dev_logits`` holds the gradient afterwards. ``host_logits`` must stay
    unchanged until ``stream`` has passed the call."""
    _check_dev(dev_logits, target, grad_output, weight)
    if host_logits.is_cuda or host_logits.shape != dev_logits.shape or host_logits.stride() != dev_logits.stride() \
            or host_logits.dtype != dev_logits.dtype:
        raise ValueError("host_logits must be a host tensor with the device tensor's shape, strides and dtype")
    p = make_params(dev_logits, target, weight=weight, ignore_index=ignore_index,
                    label_smoothing=label_smoothing, reduction=reduction)
    if loss is None:
        loss = torch.empty(dev_logits.shape[0] if reduction == "none" else 1, dtype=torch.float32,
                           device=dev_logits.device)
    ws, ws_bytes = _ws(ws, dev_logits.shape[0], dev_logits.device)
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=dev_logits.device)
    _check(_lib.ce_fwd_bwd_from_host(ctypes.byref(p), ctypes.c_void_p(host_logits.data_ptr()), _ptr(dev_logits),
                                     _ptr(target), _ptr(loss), _ptr(grad_output), _ptr(ws), ws_bytes,
                                     _stream(stream), _stream(copy_stream), int(n_parts)), "ce_fwd_bwd_from_host")
    return loss


def auto_variant(logits, target, *, weight=None, label_smoothing=0.0, softcap=0.0, z_loss=0.0,
                 accuracy=None) -> str:
    """The kernel path ce_fwd_bwd(variant="auto") takes for these tensors."""
    p = make_params(logits, target, weight=weight, label_smoothing=label_smoothing, softcap=softcap,
                    z_loss=z_loss, accuracy=accuracy)
    out = ctypes.c_int32()
    _check(_lib.ce_select_variant(ctypes.byref(p), _ptr(logits), ctypes.byref(out)), "ce_select_variant")
    return {v: k for k, v in VARIANTS.items()}[out.value]


def ce_scale_grad(grad, grad_output, *, reduction="mean", vocab=None, stream=None):
    """grad[i, :vocab] *= grad_output ([1]) or grad_output[i] (reduction none);
    skipped on the device when a [1] grad_output equals 1."""
    _check_dev(grad, grad_output)
    n, v = grad.shape
    p = ce_params()
    p.n_rows, p.vocab = n, v if vocab is None else vocab
    p.ld = grad.stride(0) if n > 1 else v
    p.dtype = CE_DT[grad.dtype]
    p.reduction = CE_RED[reduction]
    _check(_lib.ce_scale_grad(ctypes.byref(p), _ptr(grad), _ptr(grad_output), _stream(stream)),
           "ce_scale_grad")
    return grad


def ce_fused_plan(n_rows: int, vocab: int, dtype=torch.bfloat16, *, weighted=False,
                  label_smoothing=0.0, cluster=0):
    """(cluster_size, n_clusters, ctas_per_sm, slice_bytes) of the fused kernel, or None."""
    p = ce_params()
    p.n_rows, p.vocab, p.ld = n_rows, vocab, vocab
    p.dtype = CE_DT[dtype]
    p.label_smoothing = label_smoothing
    p.reduction = 1
    p.variant = int(cluster) << 8
    dummy = None
    if weighted:
        dummy = torch.empty(vocab, dtype=torch.float32, device="cuda")
        p.class_weight = dummy.data_ptr()
    c, ncl, per_sm = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    sb = ctypes.c_int64()
    st = _lib.ce_fused_plan(ctypes.byref(p), ctypes.byref(c), ctypes.byref(ncl), ctypes.byref(per_sm),
                            ctypes.byref(sb))
    if st == CE_ERR_UNSUPPORTED:
        return None
    _check(st, "ce_fused_plan")
    return c.value, ncl.value, per_sm.value, sb.value


def ce_selftest_wait_timeout(limit_ns: int = 100_000_000, stream=None) -> int:
    """Runs the bounded-wait self-test (a wait nothing satisfies) and returns
    the flags it reported (CE_FLAG_WAIT_TIMEOUT expected); synchronises."""
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(_lib.ce_selftest_wait_timeout(int(limit_ns), _ptr(flags), _stream(stream)), "ce_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(flags.item())


def ce_get_status(ws, stream=None) -> int:
    """Synchronises the stream and returns the CE_FLAG_* bits of the last call on ``ws``."""
    out = ctypes.c_uint32()
    _check(_lib.ce_get_status(_ptr(ws), ctypes.byref(out), _stream(stream)), "ce_get_status")
    return out.value


class CrossEntropyFunction(torch.autograd.Function):
    """loss = CE(logits, target), gradient formed in the forward pass: the
    fused pass runs with grad_output = 1 and leaves the gradient in the
    logits buffer (one read and one write of the logits, one logits tensor
    of peak memory); the backward multiplies it by grad_output in place,
    skipped on the device when grad_output == 1. With grad_output == 1 every
    element is rounded once; otherwise the product is rounded a second time
    (within 2 ulps). The logits tensor is consumed: its contents after the
    forward are the gradient."""

    @staticmethod
    def forward(ctx, logits, target, weight, ignore_index, label_smoothing, reduction):
        loss = ce_fwd_bwd(logits.detach(), target, weight=weight, ignore_index=ignore_index,
                          label_smoothing=label_smoothing, reduction=reduction)
        ctx.save_for_backward(logits.detach())
        ctx.reduction = reduction
        out = loss if reduction == "none" else loss.reshape(())
        return out

    @staticmethod
    def backward(ctx, grad_out):
        (grad,) = ctx.saved_tensors
        g = grad_out.detach().to(torch.float32).reshape(-1).contiguous()
        ce_scale_grad(grad, g, reduction=ctx.reduction)
        return grad, None, None, None, None, None


class CrossEntropyExactFunction(torch.autograd.Function):
    """loss = CE(logits, target) with the gradient formed in the backward
    pass: the forward reads the logits once and keeps the per-row statistics
    (16 bytes a row); the backward reads them again and writes the gradient,
    grad_output applied inside the one fp32 computation and rounded once, for
    any grad_output (TransformerEngine #2325's forward/backward split). It
    moves 1.5 times the bytes of CrossEntropyFunction. The logits must stay
    unchanged until the backward, which overwrites them with the gradient."""

    @staticmethod
    def forward(ctx, logits, target, weight, ignore_index, label_smoothing, reduction):
        x = logits.detach()
        loss, stats = ce_forward(x, target, weight=weight, ignore_index=ignore_index,
                                 label_smoothing=label_smoothing, reduction=reduction)
        ctx.save_for_backward(x, target, stats, weight)
        ctx.ignore_index, ctx.label_smoothing, ctx.reduction = ignore_index, label_smoothing, reduction
        return loss if reduction == "none" else loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        x, target, stats, weight = ctx.saved_tensors
        g = grad_out.detach().to(torch.float32).reshape(-1).contiguous()
        ce_backward(x, target, stats, grad_output=g, weight=weight, ignore_index=ctx.ignore_index,
                    label_smoothing=ctx.label_smoothing, reduction=ctx.reduction)
        return x, None, None, None, None, None


def cross_entropy(logits, target, weight=None, ignore_index=-100, label_smoothing=0.0, reduction="mean",
                  grad_mode="inplace"):
    """torch.nn.functional.cross_entropy-like entry; ``logits`` is overwritten
    by its gradient. ``grad_mode``: "inplace" (CrossEntropyFunction: one read
    and one write of the logits, one rounding when grad_output is 1, two
    otherwise) or "exact" (CrossEntropyExactFunction: one rounding for any
    grad_output, the logits read twice)."""
    if grad_mode == "inplace":
        return CrossEntropyFunction.apply(logits, target, weight, ignore_index, label_smoothing, reduction)
    if grad_mode == "exact":
        return CrossEntropyExactFunction.apply(logits, target, weight, ignore_index, label_smoothing, reduction)
    raise ValueError(f"unknown grad_mode {grad_mode!r}")


# ---------------------------------------------------------------------- fused linear
CE_GEMM_F32_STORE, CE_GEMM_F32_ACCUM, CE_GEMM_BF16_STORE = 0, 1, 2


def ce_gemm_bf16(A, B, *, a_mn_major=False, b_mn_major=False, out=None, out_kind=CE_GEMM_F32_STORE,
                 bias=None, stream=None):
    """D = A_op @ B_op on the tensor cores. A is [M, K] (or [K, M] when
    a_mn_major); B is [N, K] (or [K, N] when b_mn_major). Returns D [M, N]."""
    _check_dev(A, B, out, bias)
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B must have unit column stride")
    M = A.shape[1] if a_mn_major else A.shape[0]
    K = A.shape[0] if a_mn_major else A.shape[1]
    N = B.shape[1] if b_mn_major else B.shape[0]
    if (B.shape[0] if b_mn_major else B.shape[1]) != K:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = torch.empty(M, N, dtype=torch.bfloat16 if out_kind == CE_GEMM_BF16_STORE else torch.float32,
                          device=A.device)
    _check(_lib.ce_gemm_bf16(M, N, K, _ptr(A), A.stride(0), int(a_mn_major), _ptr(B), B.stride(0),
                             int(b_mn_major), out_kind, _ptr(out), out.stride(0), _ptr(bias), _stream(stream)),
           "ce_gemm_bf16")
    return out


CE_FLCE_DENSE, CE_FLCE_CE_CLUSTER = 1, 2


def _flce_variant(dense: bool, ce_cluster: bool) -> int:
    return (CE_FLCE_DENSE if dense else 0) | (CE_FLCE_CE_CLUSTER if ce_cluster else 0)


def flce_workspace_size(n_rows: int, hidden: int, vocab: int, chunk_rows: int, dense: bool = False,
                        ce_cluster: bool = False) -> int:
    p = ce_params()
    p.n_rows, p.vocab, p.ld, p.dtype = n_rows, vocab, vocab, CE_DT[torch.bfloat16]
    p.variant = _flce_variant(dense, ce_cluster)
    out = ctypes.c_size_t()
    _check(_lib.flce_workspace_size(ctypes.byref(p), hidden, chunk_rows, ctypes.byref(out)), "flce_workspace_size")
    return out.value


def flce_fwd_bwd(hidden, weight, target, *, bias=None, class_weight=None, ignore_index=-100,
                 label_smoothing=0.0, reduction="mean", grad_output=None, chunk_rows=4096, loss=None,
                 grad_hidden=None, grad_weight=None, grad_bias=None, ws=None, stream=None, dense=False,
                 ce_cluster=False, softcap=0.0, z_loss=0.0, accuracy=None):
    """Fused-linear cross-entropy: returns (loss, grad_hidden [BT, H] bf16,
    grad_weight [V, H] fp32, grad_bias [V] fp32 or None). ``dense=True``
    runs every row through the GEMMs instead of skipping ignored rows;
    ``ce_cluster=True`` runs each chunk's cross-entropy with the cluster
    kernel instead of the GEMM-epilogue statistics and the streaming map.
    ``softcap`` / ``z_loss`` / ``accuracy`` (a device fp32 [1] tensor) as in
    ce_fwd_bwd (not with ``ce_cluster``)."""
    _check_dev(hidden, weight, target, bias, class_weight, grad_output)
    BT, H = hidden.shape
    V = weight.shape[0]
    p = ce_params()
    p.n_rows, p.vocab, p.ld = BT, V, V
    p.ignore_index = ignore_index
    p.class_weight = class_weight.data_ptr() if class_weight is not None else None
    p.label_smoothing = float(label_smoothing)
    p.dtype = CE_DT[torch.bfloat16]
    p.reduction = CE_RED[reduction]
    p.target_is_int32 = 1 if target.dtype == torch.int32 else 0
    p.variant = _flce_variant(dense, ce_cluster)
    p.softcap, p.z_loss = float(softcap), float(z_loss)
    if accuracy is not None:
        _check_dev(accuracy)
        p.accuracy = accuracy.data_ptr()
    dev = hidden.device
    if loss is None:
        loss = torch.empty(BT if reduction == "none" else 1, dtype=torch.float32, device=dev)
    if grad_hidden is None:
        grad_hidden = torch.empty(BT, H, dtype=torch.bfloat16, device=dev)
    if grad_weight is None:
        grad_weight = torch.empty(V, H, dtype=torch.float32, device=dev)
    if bias is not None and grad_bias is None:
        grad_bias = torch.empty(V, dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(flce_workspace_size(BT, H, V, chunk_rows, dense, ce_cluster), dtype=torch.uint8,
                         device=dev)
    _check(_lib.flce_fwd_bwd(ctypes.byref(p), H, _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(target), _ptr(loss),
                             _ptr(grad_output), _ptr(grad_hidden), _ptr(grad_weight), _ptr(grad_bias), chunk_rows,
                             _ptr(ws), ws.numel(), _stream(stream)), "flce_fwd_bwd")
    return loss, grad_hidden, grad_weight, grad_bias

