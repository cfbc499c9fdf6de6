#!/usr/bin/env python
"""LoRA linear layer fwd+bwd throughput on GB300: tokens/s and fraction of the layer roofline.

Default workload: the Llama-3.1-8B MLP up-projection shape, m=8192 tokens,
k=4096, n=14336, rank 16, alpha 2, dropout 0.1, bf16 with fp32 accumulation,
synthetic seeded inputs.  One step = lora_fwd + lora_bwd (every kernel of the
hot path).  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference     # the fp64 CPU oracle on the host cores

N > 1 (torchrun): independent replicas, one per GPU, no collective on the data
path (the layer needs none); value = tokens of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from lora_fine_tuning_gb300 import synth  # noqa: E402

METRIC = "LoRA linear fwd+bwd tokens/s on 1 GB300; % of layer roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# shared helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(name, cfg):
    return (f"{name}: LoRA linear m={cfg['m']} tokens, k={cfg['k']}, n={cfg['n']}, r={cfg['r']}, "
            f"alpha={cfg['alpha']}, p={cfg['p']}, seed={cfg['seed']}")


def layer_flops(m, k, n, r):
    """Algorithmic FLOPs of one fwd+bwd: 4mkn + 6mr(k+n) (no dW: W is frozen)."""
    return 4 * m * k * n + 6 * m * r * (k + n)


def layer_bytes(m, k, n, r):
    """Compulsory HBM bytes of one fwd+bwd (bf16): fwd X, W, A, B, Y, S; bwd dY, W, X, S, A, B, dX, dA, dB."""
    fwd = 2 * (m * k + k * n + k * r + r * n + m * n + m * r)
    bwd = 2 * (m * n + k * n + m * k + m * r + k * r + r * n + m * k + k * r + r * n)
    return fwd + bwd


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                pw.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [s for s, p in zip(sm, pw) if p > 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None if
    the kernel sources changed since the capture (or none exists)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    entry = data.get(kernel)
    if not entry:
        return None
    if entry.get("source_digest") != source_digest(entry.get("sources", [])):
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import lora_oracle as O
    name = args.workload
    cfg = synth.WORKLOADS[name]
    m, k, n, r, alpha, p, seed = (cfg[x] for x in ("m", "k", "n", "r", "alpha", "p", "seed"))
    raw = synth.layer_inputs(seed, m, k, n, r)
    W = O.bf16_to_f64(raw["W"])
    A = O.bf16_to_f64(raw["A"])
    B = O.bf16_to_f64(raw["B"])

    def step(rows):
        X = O.bf16_to_f64(raw["X"][rows])
        dY = O.bf16_to_f64(raw["dY"][rows])
        O.lora_forward(X, W, A, B, alpha, p, seed, rows=rows)
        O.lora_backward(dY, X, W, A, B, alpha, p, seed, rows=rows)

    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(m, size=32, replace=False))
    t0 = time.perf_counter()
    step(probe)
    t_probe = time.perf_counter() - t0
    budget = min(args.ref_step_seconds, 150.0 / max(1, args.steps + args.warmup))
    rows_per_step = int(np.clip(32 * budget / max(t_probe, 1e-3), 16, m))
    times = []
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(m, size=rows_per_step, replace=False))
        t0 = time.perf_counter()
        step(rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = rows_per_step * len(times) / total
    cores = os.cpu_count()
    sample = (f"{rows_per_step} random rows of the {m}-row batch per step (Y, S, dX rows and their dA/dB "
              f"contributions; keep mask regenerated), fp64 numpy/BLAS")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(name, cfg), "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_leg(name, cfg, seconds: float):
    """The oracle as it stands on a bounded row sample of the same workload (rank 0, N=1)."""
    from oracle import lora_oracle as O
    m, k, n, r, alpha, p, seed = (cfg[x] for x in ("m", "k", "n", "r", "alpha", "p", "seed"))
    raw = synth.layer_inputs(seed, m, k, n, r)
    W, A, B = (O.bf16_to_f64(raw[x]) for x in ("W", "A", "B"))
    rng = np.random.default_rng(1)

    def step(rows):
        X = O.bf16_to_f64(raw["X"][rows])
        dY = O.bf16_to_f64(raw["dY"][rows])
        O.lora_forward(X, W, A, B, alpha, p, seed, rows=rows)
        O.lora_backward(dY, X, W, A, B, alpha, p, seed, rows=rows)

    probe = np.sort(rng.choice(m, size=32, replace=False))
    t0 = time.perf_counter()
    step(probe)
    tp = time.perf_counter() - t0
    rows_n = int(np.clip(32 * seconds / max(tp, 1e-3), 32, m))
    rows = np.sort(rng.choice(m, size=rows_n, replace=False))
    t0 = time.perf_counter()
    step(rows)
    dt = time.perf_counter() - t0
    return {"value": rows_n / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows_n} of {m} rows, one fwd+bwd pass (fp64 numpy/BLAS), {dt:.1f} s"}


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args):
    import torch
    import torch.distributed as dist

    from lora_fine_tuning_gb300 import api, native

    ws_n, rank, local = dist_env()
    if ws_n > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload
    cfg = synth.WORKLOADS[name]
    m, k, n, r, alpha, p, seed = (cfg[x] for x in ("m", "k", "n", "r", "alpha", "p", "seed"))

    raw = synth.layer_inputs(seed, m, k, n, r)

    def pinned(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()

    Xh, Wh, Ah, Bh, dYh = (pinned(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    X, W, A, B, dY = (t.to(dev) for t in (Xh, Wh, Ah, Bh, dYh))
    Y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    S = torch.empty((m, r), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((k, r), dtype=torch.bfloat16, device=dev)
    dB = torch.empty((r, n), dtype=torch.bfloat16, device=dev)
    wsb = api.workspace(m, k, n, r, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        api.lora_fwd(X, W, A, B, alpha, p, seed, Y=Y, S_saved=S, ws=wsb, stream=stream)
        api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed, dX=dX, dA=dA, dB=dB, ws=wsb, stream=stream)

    def barrier():
        if ws_n > 1:
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        if ws_n == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if api.lora_device_status(wsb, stream) != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")

    # --- timed region (device, inputs resident in HBM; per-kernel events on the launch stream) ---
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize(dev)
        native.timing_begin()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        kernel_times = native.timing_end()
        barrier()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1))
    clk = clocks.summary()
    if api.lora_device_status(wsb, stream) != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")

    ms_per_step = elapsed_ms / args.steps
    tokens = m * args.steps * ws_n
    value = tokens / (elapsed_ms / 1e3)

    # --- end to end through the public API with host buffers ---
    e2e = None
    if not args.no_e2e:
        Yh = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
        dXh = torch.empty((m, k), dtype=torch.bfloat16).pin_memory()
        dAh = torch.empty((k, r), dtype=torch.bfloat16).pin_memory()
        dBh = torch.empty((r, n), dtype=torch.bfloat16).pin_memory()
        e2e_steps = max(3, min(args.steps, 20))

        def e2e_step():
            X.copy_(Xh, non_blocking=True)
            dY.copy_(dYh, non_blocking=True)
            step()
            Yh.copy_(Y, non_blocking=True)
            dXh.copy_(dX, non_blocking=True)
            dAh.copy_(dA, non_blocking=True)
            dBh.copy_(dB, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(f0.elapsed_time(f1))
        h2d = (Xh.numel() + dYh.numel()) * 2
        d2h = (Yh.numel() + dXh.numel() + dAh.numel() + dBh.numel()) * 2
        e2e = {"value": m * e2e_steps * ws_n / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / e2e_steps}

    # --- frozen-layer reference points (overhead of the LoRA branch) ---
    frozen = None
    if not args.no_frozen:
        reps = args.steps   # same length as the timed LoRA loop, so both see the same clock behaviour

        def frozen_ours():
            api.multi_lora_fwd(X, W, [], [], seed, Y=Y, ws=wsb, stream=stream)
            api.multi_lora_bwd(dY, X, W, [], [], seed, None, dX=dX, ws=wsb, stream=stream)

        def frozen_torch():
            torch.matmul(X, W, out=Y)
            torch.matmul(dY, W.t(), out=dX)

        res = {}
        frozen_kernels = {}
        for label, fn in (("ours", frozen_ours), ("torch_matmul", frozen_torch)):
            fn()
            torch.cuda.synchronize(dev)
            if label == "ours":
                native.timing_begin()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(reps):
                fn()
            g1.record(stream)
            torch.cuda.synchronize(dev)
            if label == "ours":
                frozen_kernels = {kname: ms / max(1, cnt) for kname, (ms, cnt) in native.timing_end().items()}
            res[label] = max_over_ranks(g0.elapsed_time(g1)) / reps
        frozen = {"frozen_ms_per_step_ours": res["ours"], "frozen_ms_per_step_torch": res["torch_matmul"],
                  "frozen_ms_per_launch_ours": frozen_kernels,
                  "lora_overhead_vs_ours": ms_per_step / res["ours"],
                  "lora_overhead_vs_torch": ms_per_step / res["torch_matmul"]}

    if rank != 0:
        return

    peaks, peak_kind = load_peaks()
    # dominant kernel: the largest summed device time
    dom = max(kernel_times.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_launches) = dom
    avg_ms = dom_ms / max(1, dom_launches)
    if dom_name == "gemm_bwd":
        dom_flops = 2 * m * n * k + 2 * m * r * k
    elif dom_name == "gemm_fwd":
        dom_flops = 2 * m * k * n + 2 * m * r * n
    else:
        dom_flops = None
    if dom_flops is not None:
        achieved = dom_flops / (avg_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": profiled_traffic(dom_name),
                    "peak_source": f"{peak_kind} (burst bf16)",
                    "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peak)}
    else:
        roofline = {"bound": "hbm", "kernel": dom_name, "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": None, "traffic": None}

    F = layer_flops(m, k, n, r)
    Bc = layer_bytes(m, k, n, r)
    t_roof = max(F / (peaks["bf16_tflops"] * 1e12), Bc / (peaks["hbm_gbs"] * 1e9))
    layer_roof = {"flops": F, "compulsory_bytes": Bc, "roofline_ms": t_roof * 1e3,
                  "frac": t_roof * 1e3 / ms_per_step, "peak_source": peak_kind,
                  "achieved_tflops": F / (ms_per_step / 1e3) / 1e12}

    kernels = {kname: {"ms_per_launch": ms / max(1, cnt), "launches": cnt, "share": ms / max(1e-9, elapsed_ms)}
               for kname, (ms, cnt) in sorted(kernel_times.items(), key=lambda kv: -kv[1][0])}
    gpu_launches = sum(cnt for kname, (ms, cnt) in kernel_times.items() if kname != "memset")

    cpu = None
    if ws_n == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(name, cfg, args.cpu_seconds)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, Llama-shaped)",
            "config": {"workload": workload_desc(name, cfg), "m": m, "k": k, "n": n, "r": r,
                       "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU",
                       "l2": "no flush: inputs larger than L2 (X 67 MB, W 117 MB, dY 235 MB, Y/dX written)"},
            "roofline": roofline, "layer_roofline": layer_roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": gpu_launches, "kernels": kernels, "clocks": clk}
    if frozen:
        line["frozen"] = frozen
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="llama8b_up", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--m", type=int, default=None, help="override the workload's token count (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline leg")
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-frozen", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.m is not None:
        synth.WORKLOADS[args.workload] = dict(synth.WORKLOADS[args.workload], m=args.m)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
