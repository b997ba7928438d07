"""fp64 CPU oracle for softmax cross-entropy forward + backward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it. The CUDA library and its Python
binding never import it, and it imports nothing from them.

``ce_oracle.c`` holds the arithmetic (plain double precision, one row at a
time, threads over rows); this module compiles it with gcc and marshals
CPU tensors to it through ctypes. ``flce`` builds the fused-linear reference
from a float64 matmul (a library primitive used as one step) followed by the
same row oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ce_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libce_oracle.so")

OR_F32, OR_BF16, OR_F16, OR_F64 = 0, 1, 2, 3
OR_NONE, OR_MEAN, OR_SUM = 0, 1, 2
_RED = {"none": OR_NONE, "mean": OR_MEAN, "sum": OR_SUM}
_DT = {torch.float32: OR_F32, torch.bfloat16: OR_BF16, torch.float16: OR_F16, torch.float64: OR_F64}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ce_oracle.c into a shared object (plain gcc, IEEE semantics:
    no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.ce_oracle_normalizers.restype = i64
            lib.ce_oracle_normalizers.argtypes = [vp, i32, i64, i64, i64, vp, vp]
            lib.ce_oracle_rows.restype = i32
            lib.ce_oracle_rows.argtypes = [vp, i32, i64, i64, i64, vp, i32, i64, vp, dbl, i32,
                                           vp, i32, dbl, dbl, vp, vp, vp, i32]
            lib.ce_oracle_rows_ex.restype = i32
            lib.ce_oracle_rows_ex.argtypes = [vp, i32, i64, i64, i64, vp, i32, i64, vp, dbl, i32,
                                              vp, i32, dbl, dbl, vp, vp, vp, i32, dbl, dbl, vp]
            lib.ce_oracle_reduce.restype = dbl
            lib.ce_oracle_reduce.argtypes = [vp, i64, i32, dbl]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _cpu(t, dtype=None):
    if t is None:
        return None
    t = t.detach().to("cpu")
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def normalizers(target: torch.Tensor, vocab: int, ignore_index: int = -100,
                weight: torch.Tensor | None = None):
    """(n_valid, W_y, W_all, n_out_of_range) over every row of ``target``."""
    lib = _load()
    tgt = _cpu(target)
    is32 = 1 if tgt.dtype == torch.int32 else 0
    if not is32:
        tgt = tgt.to(torch.int64)
    w = _cpu(weight, torch.float64)
    out = (ctypes.c_double * 3)()
    bad = lib.ce_oracle_normalizers(tgt.data_ptr(), is32, tgt.numel(), vocab, ignore_index,
                                    w.data_ptr() if w is not None else None, out)
    return out[0], out[1], out[2], int(bad)


def rows(logits: torch.Tensor, target: torch.Tensor, *, weight=None, ignore_index: int = -100,
         label_smoothing: float = 0.0, reduction: str = "mean", grad_output=None,
         norm_wy: float | None = None, w_all: float | None = None, want_grad: bool = True,
         want_stats: bool = True, n_threads: int | None = None, softcap: float = 0.0,
         z_loss: float = 0.0) -> dict:
    """Per-row oracle on a block of rows. ``logits`` is a CPU (or device,
    copied here) [R, V] tensor in f32/bf16/f16/f64, possibly a row-strided
    view. ``norm_wy`` / ``w_all`` default to the normalisers of this block;
    pass the whole batch's values when the block is a sample. ``softcap``
    (c > 0: logits become c tanh(x / c)) and ``z_loss`` (lambda LSE^2 per valid
    row) are off at 0; ``argmax`` (first column of the row maximum) is
    always returned."""
    lib = _load()
    x = logits.detach().to("cpu")
    if x.dim() != 2 or x.stride(1) != 1:
        x = x.contiguous()
    R, V = x.shape
    ld = x.stride(0) if R > 1 else V
    if x.dtype not in _DT:
        raise TypeError(f"unsupported logits dtype {x.dtype}")
    tgt = _cpu(target)
    is32 = 1 if tgt.dtype == torch.int32 else 0
    if not is32:
        tgt = tgt.to(torch.int64)
    w = _cpu(weight, torch.float64)
    if norm_wy is None or w_all is None:
        n, wy, wa, _ = normalizers(tgt, V, ignore_index, weight)
        norm_wy = wy if norm_wy is None else norm_wy
        w_all = wa if w_all is None else w_all
    per_row = 0
    g = None
    if grad_output is not None:
        g = _cpu(torch.as_tensor(grad_output), torch.float64).reshape(-1)
        per_row = 1 if g.numel() > 1 or reduction == "none" else 0
        if per_row and g.numel() != R:
            raise ValueError("per-row grad_output must have one value per row")
    row_loss = torch.zeros(R, dtype=torch.float64)
    stats = torch.zeros(R, 4, dtype=torch.float64) if want_stats else None
    grad = torch.zeros(R, V, dtype=torch.float64) if want_grad else None
    argmax = torch.zeros(R, dtype=torch.int64)
    rc = lib.ce_oracle_rows_ex(
        x.data_ptr(), _DT[x.dtype], R, V, ld, tgt.data_ptr(), is32, ignore_index,
        w.data_ptr() if w is not None else None, float(label_smoothing), _RED[reduction],
        g.data_ptr() if g is not None else None, per_row, float(norm_wy), float(w_all),
        row_loss.data_ptr(), stats.data_ptr() if stats is not None else None,
        grad.data_ptr() if grad is not None else None, n_threads or default_threads(),
        float(softcap), float(z_loss), argmax.data_ptr())
    if rc != 0:
        raise RuntimeError(f"ce_oracle_rows failed with code {rc}")
    return {"row_loss": row_loss, "stats": stats, "grad": grad, "argmax": argmax,
            "norm_wy": norm_wy, "w_all": w_all}


def reduce(row_loss: torch.Tensor, reduction: str, norm_wy: float):
    """The reduced loss (a float) for mean / sum; the per-row tensor for none."""
    if reduction == "none":
        return row_loss
    lib = _load()
    rl = _cpu(row_loss, torch.float64)
    return lib.ce_oracle_reduce(rl.data_ptr(), rl.numel(), _RED[reduction], float(norm_wy))


def accuracy(argmax: torch.Tensor, target: torch.Tensor, vocab: int, ignore_index: int = -100) -> float:
    """Token accuracy: the share of valid rows whose argmax is the target (0
    when no row is valid)."""
    t = _cpu(target).to(torch.int64)
    valid = (t != ignore_index) & (t >= 0) & (t < vocab)
    n = int(valid.sum())
    return float((argmax[valid] == t[valid]).sum()) / n if n else 0.0


def ce(logits, target, *, weight=None, ignore_index: int = -100, label_smoothing: float = 0.0,
       reduction: str = "mean", grad_output=None, want_grad: bool = True,
       n_threads: int | None = None, softcap: float = 0.0, z_loss: float = 0.0) -> dict:
    """Whole-batch oracle: loss (reduced as asked), per-row losses, stats, the
    fp64 gradient of (grad_output * loss) with respect to the logits, the
    per-row argmax and the token accuracy."""
    V = logits.shape[1]
    n, wy, wall, bad = normalizers(target, V, ignore_index, weight)
    out = rows(logits, target, weight=weight, ignore_index=ignore_index,
               label_smoothing=label_smoothing, reduction=reduction, grad_output=grad_output,
               norm_wy=wy, w_all=wall, want_grad=want_grad, n_threads=n_threads,
               softcap=softcap, z_loss=z_loss)
    out["loss"] = reduce(out["row_loss"], reduction, wy)
    out["n_valid"], out["n_out_of_range"] = n, bad
    out["accuracy"] = accuracy(out["argmax"], target, V, ignore_index)
    return out


def flce_logits(hidden: torch.Tensor, weight: torch.Tensor, bias=None, row_block: int = 512):
    """fp64 logits z = hidden @ weight^T (+ bias), computed in row blocks.
    Yields (row_start, z_block) pairs so the caller never holds all rows."""
    h = _cpu(hidden, torch.float64)
    W = _cpu(weight, torch.float64)
    b = _cpu(bias, torch.float64) if bias is not None else None
    for r0 in range(0, h.shape[0], row_block):
        z = h[r0:r0 + row_block] @ W.T
        if b is not None:
            z += b
        yield r0, z


def flce(hidden, weight, target, *, bias=None, ignore_index: int = -100,
         label_smoothing: float = 0.0, reduction: str = "mean", sample_rows=None,
         sample_cols=None, abs_sums: bool = False, n_threads: int | None = None,
         class_weight=None, grad_output=None, softcap: float = 0.0, z_loss: float = 0.0) -> dict:
    """Fused-linear cross-entropy reference (fp64).

    Returns the reduced loss, the per-row losses, grad_hidden on
    ``sample_rows`` (all rows if None) and grad_weight on ``sample_cols``
    (all vocabulary rows if None): grad_hidden = dZ @ W, grad_weight = dZ^T @ h
    with dZ the oracle gradient of the loss with respect to z = h W^T + b.
    With ``abs_sums`` it also returns |dZ| @ |W| and |dZ|^T @ |h| on the same
    samples (the magnitudes that bound rounding errors of dZ in the tests).
    ``class_weight``, ``grad_output`` (scalar, or one value per row for
    reduction none), ``softcap`` and ``z_loss`` are handed to the row oracle
    unchanged; ``accuracy`` is the token accuracy of the logits' argmax."""
    BT, H = hidden.shape
    V = weight.shape[0]
    n, wy, wall, bad = normalizers(target, V, ignore_index, class_weight)
    g_all = None
    if grad_output is not None:
        g_all = _cpu(torch.as_tensor(grad_output), torch.float64).reshape(-1)
    Wd = _cpu(weight, torch.float64)
    hd = _cpu(hidden, torch.float64)
    tgt = _cpu(target).to(torch.int64)
    rows_sel = torch.arange(BT) if sample_rows is None else torch.as_tensor(sample_rows)
    cols_sel = torch.arange(V) if sample_cols is None else torch.as_tensor(sample_cols)
    row_mask = torch.zeros(BT, dtype=torch.bool)
    row_mask[rows_sel] = True
    row_loss = torch.zeros(BT, dtype=torch.float64)
    grad_h = torch.zeros(len(rows_sel), H, dtype=torch.float64)
    grad_w = torch.zeros(len(cols_sel), H, dtype=torch.float64)
    pos = torch.full((BT,), -1, dtype=torch.int64)
    pos[rows_sel] = torch.arange(len(rows_sel))
    grad_b = torch.zeros(len(cols_sel), dtype=torch.float64) if bias is not None else None
    abs_h = torch.zeros(len(rows_sel), H, dtype=torch.float64) if abs_sums else None
    abs_w = torch.zeros(len(cols_sel), H, dtype=torch.float64) if abs_sums else None
    amax = torch.zeros(BT, dtype=torch.int64)
    for r0, z in flce_logits(hidden, weight, bias):
        r1 = r0 + z.shape[0]
        g = None
        if g_all is not None:
            g = g_all[r0:r1] if reduction == "none" else g_all
        res = rows(z, tgt[r0:r1], weight=class_weight, ignore_index=ignore_index,
                   label_smoothing=label_smoothing, reduction=reduction, grad_output=g,
                   norm_wy=wy, w_all=wall, want_grad=True, want_stats=False, n_threads=n_threads,
                   softcap=softcap, z_loss=z_loss)
        amax[r0:r1] = res["argmax"]
        row_loss[r0:r1] = res["row_loss"]
        dz = res["grad"]
        grad_w += dz[:, cols_sel].T @ hd[r0:r1]
        if abs_w is not None:
            abs_w += dz[:, cols_sel].abs().T @ hd[r0:r1].abs()
        if grad_b is not None:
            grad_b += dz[:, cols_sel].sum(0)
        sel = row_mask[r0:r1].nonzero().flatten()
        if sel.numel():
            grad_h[pos[r0 + sel]] = dz[sel] @ Wd
            if abs_h is not None:
                abs_h[pos[r0 + sel]] = dz[sel].abs() @ Wd.abs()
    return {"loss": reduce(row_loss, reduction, wy), "row_loss": row_loss,
            "grad_hidden": grad_h, "grad_weight": grad_w, "grad_bias": grad_b,
            "grad_hidden_abs": abs_h, "grad_weight_abs": abs_w,
            "rows": rows_sel, "cols": cols_sel, "norm_wy": wy,
            "accuracy": accuracy(amax, tgt, V, ignore_index)}
