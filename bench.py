"""Benchmark: softmax cross-entropy forward + backward tokens/s at BT=8192,
V=128256, bf16 (5% ignored rows, label smoothing 0.1, mean, grad_output 1,
gradient written over the logits), on N GPUs of one node.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is the whole hot path on one batch: the normaliser kernel and the
fused single-read cross-entropy kernel (ce_fwd_bwd). Inputs are 2.1 GB, far
above the 129 MB L2; before every step the logits are restored from a
pristine copy and a 256 MB buffer is written to flush L2, both outside the
timed region; each step is timed with CUDA events on its stream, and the
step times are summed (max over ranks). N > 1 runs N independent replicas
(one per GPU, torchrun); the value is the tokens of all ranks over the
slowest rank's time.

``--impl reference`` times the CPU fp64 oracle (the reference arm of this
build: there is no other implementation of the pages to run) on a bounded
sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "headline"
METRIC = "CE fwd+bwd tokens/s at BT=8192 V=128256 bf16; achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ce_stream_kernel_headline_traffic.json")
KERNEL_SOURCES = ["softmax_cross_entropy_pass_gb300/csrc/ce_stream.cuh",
                  "softmax_cross_entropy_pass_gb300/csrc/ce_stream.cu",
                  "softmax_cross_entropy_pass_gb300/csrc/ce_device.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def read_traffic(path: str, workload: str):
    """ncu DRAM bytes (read + write) per launch of the stream kernel on the
    headline workload, when the capture was taken on the current kernel
    source (else None)."""
    if path != "stream" or workload != WORKLOAD:
        return None
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return float(d["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(", ") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for k, name in enumerate(names):
                if r[5 + k].strip().lower() == "active":
                    reasons.add(name)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                   "samples": len(sm)}
        return out


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(rows_per_rank: int, steps: int, local_total_ms: float, world: int, device):
    """Whole-job tokens/s of N replicas: every rank's rows over the slowest
    rank's time (max over ranks). Returns (tokens_per_s, ms_per_step)."""
    total_ms = reduce_max(local_total_ms, world, device)
    ms_per_step = total_ms / steps
    return rows_per_rank * world / (ms_per_step / 1e3), ms_per_step


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_text(cfg, n_rows: int, vocab: int, n_ignored: int) -> str:
    """The workload as both arms name it in config.workload."""
    return (f"{cfg.name}: BT={n_rows}, V={vocab}, {cfg.dtype} logits N(0,{cfg.sigma:g}^2), "
            f"{n_ignored} rows ignore_index=-100, label_smoothing={cfg.label_smoothing:g}, "
            f"{cfg.reduction}, grad_output={cfg.grad_output}, "
            f"{'class weights, ' if cfg.weighted else ''}gradient in place")


# --------------------------------------------------------------------------- CPU oracle arm
def oracle_sample_run(cfg, n_rows: int, threads: int, block: int = 1024):
    """Oracle forward + backward (loss, statistics, fp64 gradient) on n_rows
    rows of the workload (its targets; synthetic logits of its distribution),
    normalised with the whole batch's normalisers, in blocks of ``block``
    rows so that host memory stays bounded; returns seconds of oracle work."""
    import oracle
    from workloads import IGNORE_INDEX, make_logits, make_targets
    t_all = make_targets(cfg.n_rows, cfg.vocab, cfg.ignore_frac, cfg.seed)
    n, wy, wall, _ = oracle.normalizers(t_all, cfg.vocab, IGNORE_INDEX, None)
    secs = 0.0
    for r0 in range(0, n_rows, block):
        r = min(block, n_rows - r0)
        x = make_logits(r, cfg.vocab, cfg.dtype, cfg.sigma, cfg.seed + 1000 + r0)
        t = t_all[(r0 + 0) % cfg.n_rows:(r0 % cfg.n_rows) + r].clone()
        if t.numel() < r:
            t = make_targets(r, cfg.vocab, cfg.ignore_frac, cfg.seed + r0)
        t0 = time.perf_counter()
        oracle.rows(x, t, label_smoothing=cfg.label_smoothing, reduction=cfg.reduction, norm_wy=wy,
                    w_all=wall, want_grad=True, n_threads=threads)
        secs += time.perf_counter() - t0
    return secs


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, timed on the host cores."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import oracle
    from workloads import CONFIGS, IGNORE_INDEX, make_targets
    cfg = CONFIGS[WORKLOAD]
    n_ignored = int((make_targets(cfg.n_rows, cfg.vocab, cfg.ignore_frac, cfg.seed) == IGNORE_INDEX).sum())
    oracle.build()
    threads = oracle.default_threads()
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample_run(cfg, rows, threads)
    times = [oracle_sample_run(cfg, rows, threads) for _ in range(args.steps)]
    per_step = sum(times) / len(times)
    value = rows / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_text(cfg, cfg.n_rows, cfg.vocab, n_ignored),
                   "global_batch": cfg.n_rows, "seq_len": None, "parallelism": "replicas x1",
                   "logits_dtype": cfg.dtype,
                   "sample": f"{rows} rows of the batch per step (in 1024-row blocks, normalised with all "
                             f"{cfg.n_rows} rows' targets)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows x 128256 per step, forward + fp64 gradient"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


E2E_PARTS = 16


def measure_e2e(ce, pristine, target, work, flush, loss, kw, stream, steps):
    """ms per step through the public API with host inputs: H2D of the
    targets (pinned), ce_fwd_bwd_from_host (the logits copied from pinned host
    memory in row blocks on a second stream, each block's kernel started when
    its copy lands), D2H of the loss. Calls that need the row pass (softcap,
    z-loss, accuracy) or ask for a variant copy first and call ce_fwd_bwd."""
    import torch
    host_x = pristine.cpu().pin_memory()
    host_t = target.cpu().pin_memory()
    host_loss = torch.empty(1, dtype=torch.float32).pin_memory()
    dev_t = torch.empty_like(target)
    copy_stream = torch.cuda.Stream(device=work.device)
    piped = kw.get("variant", "auto") == "auto" and not kw.get("tune") and not kw.get("cluster") and \
        not kw.get("softcap") and not kw.get("z_loss") and kw.get("accuracy") is None
    fkw = {k: v for k, v in kw.items() if k not in ("variant", "tune", "cluster")}

    def one():
        dev_t.copy_(host_t, non_blocking=True)
        if piped:
            ce.ce_fwd_bwd_from_host(host_x, work, dev_t, copy_stream=copy_stream, n_parts=E2E_PARTS, **fkw)
        else:
            work.copy_(host_x, non_blocking=True)
            ce.ce_fwd_bwd(work, dev_t, **kw)
        host_loss.copy_(loss, non_blocking=True)

    e2e_steps = max(3, min(steps, 10))
    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e2e_ev = []
    for _ in range(e2e_steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        one()
        b.record(stream)
        e2e_ev.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / e2e_steps

    return e2e_ms


def measure_flce(ce, device, steps: int, chunk_rows: int):
    """Fused-linear cross-entropy at hidden 8192 x 4096, W 128256 x 4096 bf16:
    ms per forward + backward step, and each tcgen05 GEMM timed alone on the
    step's chunk shapes (TFLOP/s against the measured bf16 peak)."""
    import torch

    from workloads import FLCE_CONFIGS, make_flce_inputs
    cfg = FLCE_CONFIGS["flce"]
    inp = make_flce_inputs(cfg, device=device)
    h, W, t = inp["hidden"], inp["weight"], inp["target"]
    BT, H, V = cfg.n_rows, cfg.hidden, cfg.vocab
    loss = torch.empty(1, device=device)
    gh = torch.empty(BT, H, dtype=torch.bfloat16, device=device)
    gw = torch.empty(V, H, dtype=torch.float32, device=device)
    ws = torch.empty(ce.flce_workspace_size(BT, H, V, chunk_rows), dtype=torch.uint8, device=device)
    kw = dict(reduction="mean", chunk_rows=chunk_rows, loss=loss, grad_hidden=gh, grad_weight=gw, ws=ws)

    def timed(**variant):
        for _ in range(2):
            ce.flce_fwd_bwd(h, W, t, **variant, **kw)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in ev:
            a.record()
            ce.flce_fwd_bwd(h, W, t, **variant, **kw)
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / steps

    # the default: ignored rows compacted away on the device, chunk cross-entropy
    # from the logits GEMM's row statistics + one streaming map
    step_ms = timed()
    dense_ms = timed(dense=True)            # every row through every GEMM
    cluster_ms = timed(ce_cluster=True)     # chunk cross-entropy by the cluster kernel
    n_valid = int(((t >= 0) & (t < V)).sum().item())
    flop = 3 * 2.0 * BT * V * H
    # the three GEMMs of one chunk, each timed alone
    c = min(chunk_rows, BT)
    dz = torch.randn(c, V, device=device).to(torch.bfloat16)
    z = torch.empty(c, V, device=device)
    ghc = torch.empty(c, H, dtype=torch.bfloat16, device=device)
    gemms = {
        "logits  Z = h W^T": (lambda: ce.ce_gemm_bf16(h[:c], W, out=z), 2.0 * c * V * H),
        "grad_h  dZ W": (lambda: ce.ce_gemm_bf16(dz, W, b_mn_major=True, out=ghc,
                                                 out_kind=ce.CE_GEMM_BF16_STORE), 2.0 * c * V * H),
        "grad_W += dZ^T h": (lambda: ce.ce_gemm_bf16(dz, h[:c], a_mn_major=True, b_mn_major=True, out=gw,
                                                     out_kind=ce.CE_GEMM_F32_ACCUM), 2.0 * c * V * H),
    }
    per = {}
    for name, (fn, fl) in gemms.items():
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 3
        per[name] = {"ms": ms, "tflops": fl / ms / 1e9}
    del dz, z, ghc
    return {"workload": f"flce: hidden [{BT}, {H}] bf16 N(0,1), weight [{V}, {H}] bf16 N(0, 0.02^2), "
                        f"5% ignore_index, mean, chunk_rows={chunk_rows}",
            "ms_per_step": step_ms, "tokens_per_s": BT / (step_ms / 1e3),
            "gemm_tflops_whole_step": flop / step_ms / 1e9,
            "valid_rows": n_valid, "gemm_tflops_executed": 3 * 2.0 * n_valid * V * H / step_ms / 1e9,
            "ms_per_step_dense": dense_ms, "gemm_tflops_dense": flop / dense_ms / 1e9,
            "ms_per_step_ce_cluster": cluster_ms,
            "gemm_chunk": per}


def measure_gemm(ce, device, spec: str, steps: int, warmup: int):
    """One tcgen05 GEMM alone: spec "M,N,K,a_mn,b_mn" (bf16 in, fp32 out)."""
    import torch
    M, N, K, a_mn, b_mn = (int(v) for v in spec.split(","))
    g = torch.Generator(device=device).manual_seed(9)
    A = torch.randn(K, M, generator=g, device=device).to(torch.bfloat16) if a_mn else \
        torch.randn(M, K, generator=g, device=device).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g, device=device).to(torch.bfloat16) if b_mn else \
        torch.randn(N, K, generator=g, device=device).to(torch.bfloat16)
    D = torch.empty(M, N, device=device)
    for _ in range(warmup):
        ce.ce_gemm_bf16(A, B, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn), out=D)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        ce.ce_gemm_bf16(A, B, a_mn_major=bool(a_mn), b_mn_major=bool(b_mn), out=D)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tflops = 2.0 * M * N * K / ms / 1e9
    peak = read_bf16_peak()
    return {"M": M, "N": N, "K": K, "a_mn_major": a_mn, "b_mn_major": b_mn, "ms": ms, "tflops": tflops,
            "peak_tflops": peak, "frac": tflops / peak}


# --------------------------------------------------------------------------- workload timing
class Workload:
    """One CE workload resident on the device: the pristine logits, a working
    copy the call overwrites with the gradient, targets, weights,
    grad_output, workspace and loss, and the keyword arguments of the call."""

    def __init__(self, ce, cfg, device, variant="auto", tune=0, cluster=0, options=None, stream=None):
        import torch
        from workloads import make_ce_inputs
        inp = make_ce_inputs(cfg, device=device)
        self.cfg = cfg
        self.pristine, self.target, self.g = inp["logits"], inp["target"], inp["grad_output"]
        self.weight = inp["weight"]
        self.work = torch.empty_like(self.pristine)
        self.R, self.V = cfg.n_rows, cfg.vocab
        self.ws = ce.workspace(self.R, device)
        self.loss = torch.empty(self.R if cfg.reduction == "none" else 1, dtype=torch.float32, device=device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(device)
        self.options = dict(options or {})
        self.kw = dict(label_smoothing=cfg.label_smoothing, reduction=cfg.reduction, grad_output=self.g,
                       loss=self.loss, ws=self.ws, stream=self.stream, variant=variant, cluster=cluster,
                       weight=self.weight, tune=tune, **self.options)
        self.n_valid = int((self.target >= 0).sum().item())
        self.esz = self.pristine.element_size()
        self.path = variant if variant != "auto" else ce.auto_variant(self.pristine, self.target,
                                                                      weight=self.weight, **self.options)

    def algo_bytes(self) -> int:
        """Algorithmic bytes of one forward + backward: every valid row read
        once (twice on the split path, whose statistics pass reads every row),
        every row written once (ignored rows are only zeroed), the targets
        twice (normaliser kernel and row kernel); with reduction none the
        per-row grad_output and losses; with class weights the weights twice
        (normaliser sum and gradient terms)."""
        cfg, R, V = self.cfg, self.R, self.V
        reads = self.n_valid + (R if self.path == "split" else 0)
        b = (reads + R) * V * self.esz + 2 * R * self.target.element_size()
        if cfg.reduction == "none":
            b += 2 * R * 4
        if self.weight is not None:
            b += 2 * V * 4
        return b

    def launches_per_step(self) -> int:
        # the normaliser kernel (plus its combining kernel with class weights)
        # and the row kernel(s)
        return (3 if self.path == "split" else 2) + (1 if self.weight is not None else 0)

    def step(self, ce):
        return ce.ce_fwd_bwd(self.work, self.target, **self.kw)

    def free(self):
        for k in ("pristine", "work", "target", "g", "weight", "ws", "loss"):
            setattr(self, k, None)


def time_workload(ce, W: Workload, steps: int, warmup: int, flush, clock_gpu=None) -> dict:
    """CUDA-event timing of W's step (normalisers + row kernel) and of the
    row kernel alone (normalisers prepared before its first event), each
    step with the logits restored from the pristine copy and a buffer larger
    than the L2 written beforehand, outside the timed region."""
    import torch
    for _ in range(warmup):
        W.work.copy_(W.pristine)
        W.step(ce)
    torch.cuda.synchronize()
    sampler = ClockSampler(clock_gpu) if clock_gpu is not None else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for k in range(steps):
        W.work.copy_(W.pristine)
        flush.zero_()
        ev[k][0].record(W.stream)
        W.step(ce)
        ev[k][1].record(W.stream)
    torch.cuda.synchronize()
    kev = []
    for _ in range(steps):
        W.work.copy_(W.pristine)
        ce.ce_prepare(W.work, W.target, label_smoothing=W.cfg.label_smoothing, reduction=W.cfg.reduction,
                      ws=W.ws, stream=W.stream, weight=W.weight)
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(W.stream)
        ce.ce_fwd_bwd(W.work, W.target, prepared=True, **W.kw)
        e1.record(W.stream)
        kev.append((e0, e1))
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    return {"step_ms": [a.elapsed_time(b) for a, b in ev], "kernel_ms": [a.elapsed_time(b) for a, b in kev],
            "clocks": clocks}


def workload_entry(W: Workload, t: dict, peak: float) -> dict:
    """The bench-line record of one timed workload."""
    step_ms = statistics.mean(t["step_ms"])
    kern_ms = statistics.mean(t["kernel_ms"])
    ab = W.algo_bytes()
    achieved = ab / (kern_ms / 1e3) / 1e9
    return {"workload": workload_text(W.cfg, W.R, W.V, W.R - W.n_valid), "path": W.path,
            "ms_per_step": step_ms, "tokens_per_s": W.R / (step_ms / 1e3),
            "step_ms_min_median_max": [min(t["step_ms"]), statistics.median(t["step_ms"]), max(t["step_ms"])],
            "kernel_ms": kern_ms, "algorithmic_bytes": ab, "achieved_gbs": achieved, "peak_gbs": peak,
            "frac": achieved / peak, "gpu_launches_per_step": W.launches_per_step(), "clocks": t["clocks"]}


def measure_tiny(ce, device, flush, steps: int = 200) -> dict:
    """The 64 x 1024 fp32 workload: device microseconds per step (CUDA
    events around each call, inputs restored outside), and the host cost of
    one call from API entry to return, taken while a sleep kernel keeps the
    GPU busy so no call waits for the device: through the Python binding
    (argument marshalling included) and through the C ABI alone (ctypes
    with a prepared parameter block)."""
    import ctypes

    import torch
    from workloads import CONFIGS
    cfg = CONFIGS["tiny"]
    W = Workload(ce, cfg, device)
    t = time_workload(ce, W, steps, 20, flush)
    dev_us = [1e3 * v for v in t["step_ms"]]
    # host cost per call
    p = ce.make_params(W.work, W.target, label_smoothing=cfg.label_smoothing, reduction=cfg.reduction)
    st = ce._stream(W.stream)
    args = (ctypes.byref(p), ctypes.c_void_p(W.work.data_ptr()), ctypes.c_void_p(W.target.data_ptr()),
            ctypes.c_void_p(W.loss.data_ptr()), None, ctypes.c_void_p(W.ws.data_ptr()),
            W.ws.numel(), st)
    n = 100
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)
    t0 = time.perf_counter()
    for _ in range(n):
        rc = ce._lib.ce_fwd_bwd(*args)
    c_us = (time.perf_counter() - t0) / n * 1e6
    if rc != 0:
        raise RuntimeError(f"ce_fwd_bwd returned {rc}")
    torch.cuda.synchronize()
    torch.cuda._sleep(100_000_000)
    kw = dict(W.kw)
    t0 = time.perf_counter()
    for _ in range(n):
        ce.ce_fwd_bwd(W.work, W.target, **kw)
    py_us = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize()
    W.free()
    return {"workload": workload_text(cfg, cfg.n_rows, cfg.vocab, 0), "path": "stream",
            "device_us_per_step_min_median_max": [min(dev_us), statistics.median(dev_us), max(dev_us)],
            "kernel_us_median": 1e3 * statistics.median(t["kernel_ms"]),
            "host_us_per_call_c_abi": c_us, "host_us_per_call_python": py_us,
            "gpu_launches_per_step": 2, "bound": "launch (report microseconds)"}


def pages_dxy_table() -> dict:
    """The pages' dx_y error table (H100, bf16, V = 32000), from its cited
    golden file, as context beside the measured errors."""
    with open(os.path.join(ROOT, "tests", "golden", "dxy_error_table_v32000_bf16.json")) as f:
        d = json.load(f)
    cols = d["columns"]
    return {"source": d["source"],
            "softmax_xy": [r[cols.index("softmax_xy")] for r in d["rows"]],
            "before_1268_pct": [r[cols.index("before_1268_pct")] for r in d["rows"]],
            "at_1268_pct": [r[cols.index("at_1268_pct")] for r in d["rows"]],
            "torch_pct": [r[cols.index("torch_pct")] for r in d["rows"]]}


def confident_dxy_report(ce, device, threads: int) -> dict:
    """dx_y accuracy on the confident workload (4096 x 32000 bf16, target
    softmax near 0.9 / 0.99 / 0.999 in thirds, 10% ignored): the max
    relative error of dx_y per third against the fp64 oracle, for this
    library and for torch.nn.functional.cross_entropy's bf16 autograd on the
    same GPU (a comparison column, like the pages' "torch" column), with the
    realised softmax(x_y) range per third. Part of the CPU-baseline leg: the
    oracle run here is also timed as that config's baseline."""
    import torch
    import torch.nn.functional as F

    import oracle
    from workloads import CONFIGS, IGNORE_INDEX, make_ce_inputs
    cfg = CONFIGS["confident"]
    inp = make_ce_inputs(cfg, device=device)
    x, t = inp["logits"], inp["target"]
    R, V = x.shape
    x_host, t_host = x.cpu(), t.cpu()
    n, wy, wall, _ = oracle.normalizers(t_host, V, IGNORE_INDEX, None)
    t0 = time.perf_counter()
    ref = oracle.rows(x_host, t_host, reduction="mean", norm_wy=wy, w_all=wall, want_grad=True, n_threads=threads)
    secs = time.perf_counter() - t0
    valid = (t_host >= 0) & (t_host < V)
    rows = valid.nonzero().flatten()
    want = ref["grad"][rows, t_host[rows]]
    st = ref["stats"][rows]
    e = torch.exp(st[:, 2] - st[:, 0])
    p_y = e / (st[:, 1] + e)
    del ref
    xg = x.clone()
    ce.ce_fwd_bwd(xg, t)
    xt = x.clone().requires_grad_(True)
    F.cross_entropy(xt, t, ignore_index=IGNORE_INDEX, reduction="mean").backward()
    torch.cuda.synchronize()
    ours = xg[rows.to(device), t[rows.to(device)]].double().cpu()
    theirs = xt.grad[rows.to(device), t[rows.to(device)]].double().cpu()
    third = (R + 2) // 3
    out = {"ours_pct": [], "torch_gpu_pct": [], "p_realised_min_max": [], "rows_per_third": []}
    for k in range(3):
        sel = (rows >= k * third) & (rows < (k + 1) * third)
        out["ours_pct"].append(100 * float(((ours[sel] - want[sel]).abs() / want[sel].abs()).max()))
        out["torch_gpu_pct"].append(100 * float(((theirs[sel] - want[sel]).abs() / want[sel].abs()).max()))
        out["p_realised_min_max"].append([float(p_y[sel].min()), float(p_y[sel].max())])
        out["rows_per_third"].append(int(sel.sum()))
    out["nominal_p"] = [0.9, 0.99, 0.999]
    out["pages_h100"] = pages_dxy_table()
    del xg, xt
    return {"dxy": out, "oracle_secs": secs, "oracle_rows": R}


def oracle_config_baseline(cfg, n_rows: int, threads: int) -> dict:
    """The oracle on n_rows rows of a workload (its distribution, weights,
    smoothing, reduction and grad_output), timed on the host cores."""
    import oracle
    from workloads import IGNORE_INDEX, make_grad_output, make_logits, make_targets, make_weights
    r = min(n_rows, cfg.n_rows)
    x = make_logits(r, cfg.vocab, cfg.dtype, cfg.sigma, cfg.seed + 1000)
    t_all = make_targets(cfg.n_rows, cfg.vocab, cfg.ignore_frac, cfg.seed)
    w = make_weights(cfg.vocab, cfg.seed) if cfg.weighted else None
    g = make_grad_output(cfg)
    n, wy, wall, _ = oracle.normalizers(t_all, cfg.vocab, IGNORE_INDEX, w)
    t0 = time.perf_counter()
    oracle.rows(x, t_all[:r], weight=w, label_smoothing=cfg.label_smoothing, reduction=cfg.reduction,
                grad_output=g[:r] if cfg.reduction == "none" else g, norm_wy=wy, w_all=wall, want_grad=True,
                n_threads=threads)
    secs = time.perf_counter() - t0
    return {"value": r / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{r} rows x {cfg.vocab} of the workload, forward + fp64 gradient, {secs:.2f} s"}


# --------------------------------------------------------------------------- GPU arm
def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if args.gemm_only:
        import softmax_cross_entropy_pass_gb300 as ce
        print(json.dumps({"gemm": measure_gemm(ce, device, args.gemm_only, max(1, args.steps), args.warmup)}),
              flush=True)
        return 0
    if args.flce_only:
        import softmax_cross_entropy_pass_gb300 as ce
        flce = measure_flce(ce, device, max(1, args.steps), args.flce_chunk)
        peak_tf = read_bf16_peak()
        flce["peak_tflops"] = peak_tf
        flce["frac_whole_step"] = flce["gemm_tflops_whole_step"] / peak_tf
        flce["frac_executed"] = flce["gemm_tflops_executed"] / peak_tf
        flce["frac_dense"] = flce["gemm_tflops_dense"] / peak_tf
        print(json.dumps({"flce": flce}), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    import softmax_cross_entropy_pass_gb300 as ce
    from workloads import CONFIGS
    cfg = CONFIGS[args.workload]
    if args.rows or args.vocab or args.dtype or args.ignore_frac >= 0 or args.reduction:
        import dataclasses
        cfg = dataclasses.replace(cfg, n_rows=args.rows or cfg.n_rows, vocab=args.vocab or cfg.vocab,
                                  dtype=args.dtype or cfg.dtype,
                                  ignore_frac=args.ignore_frac if args.ignore_frac >= 0 else cfg.ignore_frac,
                                  reduction=args.reduction or cfg.reduction)
    options = {}
    if args.softcap > 0:
        options["softcap"] = args.softcap
    if args.z_loss > 0:
        options["z_loss"] = args.z_loss
    if args.accuracy:
        options["accuracy"] = torch.empty(1, dtype=torch.float32, device=device)
    W = Workload(ce, cfg, device, variant=args.variant, tune=args.tune, cluster=args.cluster, options=options)
    R, V = W.R, W.V
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    plan = ce.ce_fused_plan(R, V, W.pristine.dtype, label_smoothing=cfg.label_smoothing, cluster=args.cluster,
                            weighted=W.weight is not None)
    path, esz = W.path, W.esz
    kernel_name = {"fused": f"ce_fused_kernel<{cfg.dtype}>", "rowpass": f"ce_rowpass_kernel<{cfg.dtype}>",
                   "stream": f"ce_stream_kernel<{cfg.dtype}>",
                   "split": f"ce_stats_kernel + ce_grad_kernel <{cfg.dtype}>"}[path]

    barrier(world)
    t = time_workload(ce, W, args.steps, args.warmup, flush, clock_gpu=local if rank == 0 else None)
    barrier(world)
    clocks = t["clocks"]
    step_ms = t["step_ms"]
    total_ms = sum(step_ms)
    kernel_avg_s = statistics.mean(t["kernel_ms"]) / 1e3

    # end to end through the public API with host buffers: H2D of the logits
    # and targets from pinned memory, the call, D2H of the loss
    e2e_ms = float("nan")
    if not args.no_e2e:
        e2e_ms = measure_e2e(ce, W.pristine, W.target, W.work, flush, W.loss, W.kw, W.stream, args.steps)

    value, ms_per_step = aggregate_throughput(R, args.steps, total_ms, world, device)
    e2e_ms = reduce_max(e2e_ms, world, device)
    kernel_avg_s = reduce_max(kernel_avg_s, world, device)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_kind = read_peaks()
    algo_bytes = W.algo_bytes()
    achieved = algo_bytes / kernel_avg_s / 1e9
    traffic = read_traffic(path, cfg.name)
    n_valid, h2d = W.n_valid, W.pristine.numel() * esz + R * 8
    loss_numel, launches = W.loss.numel(), W.launches_per_step()
    W.free()
    del W
    torch.cuda.empty_cache()

    # the other workloads, one at a time, timed the same way (one GPU only)
    configs = None
    if world == 1 and not args.no_configs and not (args.rows or args.vocab or args.dtype or args.reduction) and \
            args.ignore_frac < 0 and \
            args.workload == WORKLOAD and not options and args.variant == "auto" and not args.tune:
        configs = {"tiny": measure_tiny(ce, device, flush)}
        for name in ("confident", "large_vocab", "large_vocab_none"):
            Wc = Workload(ce, CONFIGS[name], device)
            tc = time_workload(ce, Wc, min(args.steps, 20), 3, flush, clock_gpu=local)
            configs[name] = workload_entry(Wc, tc, peak)
            Wc.free()
            del Wc
            torch.cuda.empty_cache()

    flce = None
    if not args.no_flce:
        flce = measure_flce(ce, device, max(3, min(args.steps, 5)), args.flce_chunk)
        peak_tf = read_bf16_peak()
        flce["peak_tflops"] = peak_tf
        flce["frac_whole_step"] = flce["gemm_tflops_whole_step"] / peak_tf
        flce["frac_executed"] = flce["gemm_tflops_executed"] / peak_tf
        flce["frac_dense"] = flce["gemm_tflops_dense"] / peak_tf
        for v in flce["gemm_chunk"].values():
            v["frac"] = v["tflops"] / peak_tf

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.default_threads()
        secs = oracle_sample_run(cfg, args.cpu_rows, threads)
        one_rows = max(16, args.cpu_rows // 64)
        secs1 = oracle_sample_run(cfg, one_rows, 1)
        cpu = {"value": args.cpu_rows / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{args.cpu_rows} rows x {V} (the whole batch of the workload, in 1024-row "
                         f"blocks), forward + fp64 gradient, {secs:.2f} s on {threads} threads",
               "single_core": {"value": one_rows / secs1, "unit": "tokens/s", "cores": 1,
                               "sample": f"{one_rows} rows, {secs1:.2f} s"}}
        if configs is not None:
            # the oracle on each other workload; on the confident one its
            # gradient also gives the dx_y accuracy report
            rep = confident_dxy_report(ce, device, threads)
            configs["confident"]["dxy_max_rel_err"] = rep["dxy"]
            configs["confident"]["cpu_baseline"] = {
                "value": rep["oracle_rows"] / rep["oracle_secs"], "unit": "tokens/s", "cores": threads,
                "kind": "oracle", "sample": f"the whole batch ({rep['oracle_rows']} rows), forward + fp64 "
                                            f"gradient, {rep['oracle_secs']:.2f} s"}
            configs["tiny"]["cpu_baseline"] = oracle_config_baseline(CONFIGS["tiny"], 64, threads)
            for name in ("large_vocab", "large_vocab_none"):
                configs[name]["cpu_baseline"] = oracle_config_baseline(CONFIGS[name], 256, threads)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        # the arithmetic type: statistics and gradient are formed in fp32 (the
        # logits' storage type is config.logits_dtype)
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_text(cfg, R, V, R - n_valid),
                   "global_batch": R * world, "seq_len": None, "parallelism": f"replicas x{world}",
                   "variant": args.variant, "path": path, "tune": args.tune, "fused_plan": plan,
                   "options": {k: (v if k != "accuracy" else True) for k, v in options.items()} or None,
                   "logits_dtype": cfg.dtype,
                   "l2": f"inputs {R * V * esz / 1e9:.2f} GB {'>' if R * V * esz > 129e6 else '<'} 129 MB L2; "
                         "logits restored and a 256 MB buffer written before every step, outside the timed "
                         "region"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_name, "kernel_ms": kernel_avg_s * 1e3,
                     "algorithmic_bytes": algo_bytes, "peak_source": peak_kind},
        "e2e": None if args.no_e2e else {"value": R * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": loss_numel * 4,
                "ms_per_step": e2e_ms},
        # per step: the normaliser kernel (two with class weights: eight partial
        # blocks, then the kernel combining them) and the row kernel(s)
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "configs": configs,
        "flce": flce,
        "step_ms_min_median_max": [min(step_ms), statistics.median(step_ms), max(step_ms)],
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--variant", choices=["auto", "fused", "split", "rowpass", "stream"], default="auto")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--tune", type=int, default=0, help="stream-kernel tuning bits (see include/ce.h)")
    ap.add_argument("--cpu-rows", type=int, default=8192)
    ap.add_argument("--ref-rows", type=int, default=2048)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-flce", action="store_true", help="skip the fused-linear measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (tiny, confident, large vocabulary sum and none)")
    ap.add_argument("--flce-chunk", type=int, default=4096)
    ap.add_argument("--flce-only", action="store_true", help="only the fused-linear measurement")
    ap.add_argument("--gemm-only", default="", help="only one GEMM: M,N,K,a_mn,b_mn")
    ap.add_argument("--rows", type=int, default=0, help="rows of a smaller case of the workload (profiling)")
    ap.add_argument("--softcap", type=float, default=0.0, help="logit softcap c (0: off)")
    ap.add_argument("--z-loss", type=float, default=0.0, help="z-loss weight lambda (0: off)")
    ap.add_argument("--accuracy", action="store_true", help="also compute the token accuracy")
    ap.add_argument("--dtype", choices=["bf16", "f16", "f32"], default="",
                    help="logits storage type (default: the workload's)")
    ap.add_argument("--reduction", choices=["mean", "sum", "none"], default="",
                    help="another reduction for the workload (profiling)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="another vocabulary size for the workload (e.g. one that leaves rows unaligned)")
    ap.add_argument("--ignore-frac", type=float, default=-1.0,
                    help="share of ignored rows for the workload (default: the workload's own)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="CE workload of workloads.CONFIGS (the default is the headline metric's)")
    ap.add_argument("--print-kernel-hash", action="store_true")
    args = ap.parse_args()
    if args.print_kernel_hash:
        print(kernel_source_hash())
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
