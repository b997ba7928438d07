"""Seeded synthetic inputs for the softmax cross-entropy hot path.

This module only draws random inputs. It holds none of the cross-entropy
arithmetic: both the CUDA path (through the tests and ``bench.py``) and the
CPU oracle receive the very same tensors from here.

The five workloads follow the shapes and value distributions that the
pages benchmark and test on:

* ``tiny``        64 x 1024 fp32 N(0,1), uniform targets, mean.
* ``confident``   4096 x 32000 bf16 N(0,1); the target logit of each row is
                  raised so that softmax(x_y) is about 0.9, 0.99 or 0.999
                  (equal thirds of the rows), 10% of rows ignored. This is
                  the dx_y cancellation workload of the Liger-Kernel #1329
                  commit message (accuracy table at V=32000, bf16).
* ``headline``    8192 x 128256 bf16 N(0,1), 5% ignored, label smoothing 0.1,
                  mean (the "reference config" of Liger-Kernel #1290 and the
                  BT=8192, V=128256 timing of #1268 / #1329).
* ``large_vocab`` 16384 x 256000 bf16 N(0, 1.5^2), class weights U(0.5, 1.5),
                  label smoothing 0.05, sum, grad_output 0.37; the ``none``
                  variant draws a per-row grad_output from U(0, 1).
* ``flce``        hidden 8192 x 4096 bf16 N(0,1), lm-head weight
                  128256 x 4096 bf16 N(0, 0.02^2), 5% ignored, mean
                  (the FLCE shape of Liger-Kernel #1622's measurements).

The pages measure on synthetic last-layer steps only, so no public dataset
is being stood in for.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

IGNORE_INDEX = -100

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class CEConfig:
    name: str
    n_rows: int
    vocab: int
    dtype: str = "bf16"          # storage dtype of the logits: f32 | bf16 | f16
    sigma: float = 1.0           # logits ~ N(0, sigma^2)
    ignore_frac: float = 0.0     # share of rows whose target is IGNORE_INDEX
    label_smoothing: float = 0.0
    reduction: str = "mean"      # mean | sum | none
    weighted: bool = False       # class weights ~ U(0.5, 1.5)
    grad_output: object = 1.0    # float, or "uniform" for a per-row U(0,1) draw
    confident: bool = False      # raise target logits to p in {0.9, 0.99, 0.999}
    seed: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def logits_bytes(self) -> int:
        return self.n_rows * self.vocab * torch.tensor([], dtype=self.torch_dtype).element_size()


CONFIGS = {
    "tiny": CEConfig("tiny", 64, 1024, "f32", seed=1),
    "confident": CEConfig("confident", 4096, 32000, "bf16", ignore_frac=0.10,
                          confident=True, seed=2),
    "headline": CEConfig("headline", 8192, 128256, "bf16", ignore_frac=0.05,
                         label_smoothing=0.1, seed=3),
    "large_vocab": CEConfig("large_vocab", 16384, 256000, "bf16", sigma=1.5,
                            label_smoothing=0.05, reduction="sum", weighted=True,
                            grad_output=0.37, seed=4),
    "large_vocab_none": CEConfig("large_vocab_none", 16384, 256000, "bf16", sigma=1.5,
                                 label_smoothing=0.05, reduction="none", weighted=True,
                                 grad_output="uniform", seed=4),
}

# softmax(x_y) targets of the confident workload, one per third of the rows.
CONFIDENT_P = (0.9, 0.99, 0.999)


@dataclasses.dataclass(frozen=True)
class FLCEConfig:
    name: str
    n_rows: int
    hidden: int
    vocab: int
    w_sigma: float = 0.02
    ignore_frac: float = 0.05
    label_smoothing: float = 0.0
    reduction: str = "mean"
    seed: int = 5


FLCE_CONFIGS = {
    "flce": FLCEConfig("flce", 8192, 4096, 128256),
    # small shapes that keep every tile loop and ragged edge busy, for parity
    "flce_small": FLCEConfig("flce_small", 384, 256, 1000, w_sigma=0.05, seed=15),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_targets(n_rows: int, vocab: int, ignore_frac: float, seed: int, device="cpu",
                 n_ignore: Optional[int] = None) -> torch.Tensor:
    """Uniform class ids in [0, vocab) with round(ignore_frac * n_rows) rows set
    to IGNORE_INDEX, picked by a seeded permutation. Drawn on the CPU so that
    every device sees the same targets."""
    g = _gen("cpu", seed * 7919 + 17)
    t = torch.randint(0, vocab, (n_rows,), generator=g, dtype=torch.int64)
    if n_ignore is None:
        n_ignore = int(round(ignore_frac * n_rows))
    if n_ignore:
        rows = torch.randperm(n_rows, generator=g)[:n_ignore]
        t[rows] = IGNORE_INDEX
    return t.to(device)


def make_logits(n_rows: int, vocab: int, dtype: str, sigma: float, seed: int,
                device="cpu", ld: Optional[int] = None) -> torch.Tensor:
    """N(0, sigma^2) logits, drawn in fp32 and rounded once to ``dtype``.

    With ``ld > vocab`` the result is a [n_rows, vocab] view of a
    [n_rows, ld] buffer (padding filled with a large sentinel so that any
    read or write past the vocabulary shows up in the tests)."""
    g = _gen(device, seed)
    ld = vocab if ld is None else ld
    full = torch.randn(n_rows, ld, generator=g, device=device, dtype=torch.float32)
    if sigma != 1.0:
        full.mul_(sigma)
    if ld > vocab:
        full[:, vocab:] = 777.0
    full = full.to(_DTYPES[dtype])
    return full[:, :vocab] if ld > vocab else full


def raise_confident_targets(logits: torch.Tensor, target: torch.Tensor, sigma: float = 1.0,
                            p_values=CONFIDENT_P) -> torch.Tensor:
    """Set the target logit of each non-ignored row so that softmax(x_y) lands
    near p (equal thirds of the rows get the three p values).

    The other logits are N(0, sigma^2), so the sum of their exponentials is
    close to (V - 1) * exp(sigma^2 / 2); the target logit is put at
    log(p / (1 - p)) plus the log of that expected sum. The realised softmax
    value differs a little (sampling noise and the rounding of x_y to the
    storage dtype); the tests read the realised value from the oracle.
    Returns the nominal p of each row (0 for ignored rows)."""
    n_rows, vocab = logits.shape
    third = (n_rows + 2) // 3
    p_row = torch.zeros(n_rows, dtype=torch.float64)
    base = math.log(vocab - 1) + 0.5 * sigma * sigma
    tgt = target.cpu()
    for k, p in enumerate(p_values):
        lo, hi = k * third, min(n_rows, (k + 1) * third)
        rows = torch.arange(lo, hi)
        rows = rows[tgt[lo:hi] >= 0]
        if rows.numel() == 0:
            continue
        val = math.log(p / (1.0 - p)) + base
        r = rows.to(logits.device)
        logits[r, target[r]] = torch.tensor(val, dtype=torch.float32).to(logits.dtype).to(logits.device)
        p_row[rows] = p
    return p_row


def make_weights(vocab: int, seed: int, device="cpu") -> torch.Tensor:
    """Class weights ~ U(0.5, 1.5), fp32."""
    g = _gen("cpu", seed * 104729 + 3)
    return (0.5 + torch.rand(vocab, generator=g, dtype=torch.float32)).to(device)


def make_grad_output(cfg: CEConfig, device="cpu") -> torch.Tensor:
    """grad_output as a device tensor: [1] for mean/sum, [n_rows] for none."""
    if cfg.grad_output == "uniform":
        g = _gen("cpu", cfg.seed * 31 + 11)
        return torch.rand(cfg.n_rows, generator=g, dtype=torch.float32).to(device)
    n = cfg.n_rows if cfg.reduction == "none" else 1
    return torch.full((n,), float(cfg.grad_output), dtype=torch.float32, device=device)


def make_ce_inputs(cfg: CEConfig, device="cpu", ld: Optional[int] = None) -> dict:
    """All inputs of one CE workload: logits, target, weight (or None),
    grad_output and, for the confident workload, the nominal p per row."""
    logits = make_logits(cfg.n_rows, cfg.vocab, cfg.dtype, cfg.sigma, cfg.seed, device, ld)
    target = make_targets(cfg.n_rows, cfg.vocab, cfg.ignore_frac, cfg.seed, device)
    out = {"logits": logits, "target": target, "p_nominal": None}
    if cfg.confident:
        out["p_nominal"] = raise_confident_targets(logits, target, cfg.sigma)
    out["weight"] = make_weights(cfg.vocab, cfg.seed, device) if cfg.weighted else None
    out["grad_output"] = make_grad_output(cfg, device)
    return out


def make_flce_inputs(cfg: FLCEConfig, device="cpu") -> dict:
    """hidden [BT, H] bf16 N(0,1); lm-head weight [V, H] bf16 N(0, w_sigma^2);
    targets uniform with ``ignore_frac`` ignored."""
    g = _gen(device, cfg.seed)
    hidden = torch.randn(cfg.n_rows, cfg.hidden, generator=g, device=device,
                         dtype=torch.float32).to(torch.bfloat16)
    w = torch.randn(cfg.vocab, cfg.hidden, generator=g, device=device, dtype=torch.float32)
    w.mul_(cfg.w_sigma)
    weight = w.to(torch.bfloat16)
    del w
    target = make_targets(cfg.n_rows, cfg.vocab, cfg.ignore_frac, cfg.seed, device)
    return {"hidden": hidden, "weight": weight, "target": target}
