#!/usr/bin/env python
"""LoRA linear layer fwd+bwd throughput on GB300: tokens/s and fraction of the layer roofline.

Default workload: the largest single-GPU layer of the set, the Llama-3.1-70B
MLP up-projection shape, m=16384 tokens, k=8192, n=28672, rank 64, alpha 2,
dropout 0.1, bf16 with fp32 accumulation, synthetic seeded inputs
(`--workload llama8b_up` for the Llama-3.1-8B up-projection, m=8192,
k=4096, n=14336, r=16).  One step = lora_fwd + lora_bwd (every kernel of the
hot path); for the packed workload multi_4ad, multi_lora_fwd + multi_lora_bwd.
Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--m M] [--r R]
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
# Kernels the library runs on its side stream, concurrently with the dX GEMM, when the backward reads the
# forward's keep bits (--saved-mask): their event pair spans from the fork (the GEMM's start) to their own
# end, so their time is not a device duration of their own.  When the backward regenerates the mask (the
# default; every workload here has k % 128 == 0) the dX GEMM hands its bits to dA, which runs after it on
# the caller's stream.
SIDE_STREAM_KINDS_SAVED_MASK = {"da"}
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 datasheet figures (dense bf16, HBM3e), for the fractions of the hardware bound beside the
# fractions of the measured copy / cuBLAS rates
DATASHEET_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
# a timed window at least this long counts as sustained (the power-capped clock has settled)
SUSTAINED_SECONDS = 1.0
DEFAULT_WORKLOAD = "llama70b_up_r64"


# ---------------------------------------------------------------------------
# shared helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


MULTI = "multi_4ad"      # packed batch, four adapters with ranks 16/16/32/64 on one 8192x8192 weight
GREEDY = "multi_4ad_greedy"   # a global batch of the same samples packed into 16384-row microbatches (greedy)
LAYER = "llama8b_layer"  # the seven LoRA projections of one Llama-3.1-8B decoder layer
DORA = "dora8b_up"       # the Llama-3.1-8B up-proj layer as DoRA (magnitude per output column)
MULTI_SQ = "multi_square4096"   # four adapters at one swept rank on a square 4096 weight, packed to --m rows


class Part:
    """One LoRA linear of a workload: its shapes, weight, adapters, inputs and (packed) segments."""

    def __init__(self, label, k, n, specs, seed, X, W, dY, adapters, segments=None, x_key="X", mag=None):
        self.label, self.k, self.n, self.specs, self.seed = label, k, n, specs, seed
        self.X, self.W, self.dY, self.adapters, self.segments, self.x_key = X, W, dY, adapters, segments, x_key
        self.mag = mag          # DoRA: magnitude per output column (fp32), else None

    @property
    def single(self) -> bool:
        return self.segments is None

    @property
    def r_max(self) -> int:
        return max(r for r, _, _ in self.specs)


class Workload:
    """One benchmark problem on the host: the token rows and one or more LoRA linears over them.

    A single-adapter linear runs through lora_fwd / lora_bwd, the packed
    multi-adapter one through multi_lora_fwd / multi_lora_bwd; the decoder
    layer runs its seven linears forward in order, then backward in reverse.
    """

    def __init__(self, name: str, m=None, r=None, packer=None):
        self.name = name
        if name == GREEDY:
            # samples for four microbatches' worth of rows, packed first-fit decreasing into microbatches
            # of 16384 rows; one multi-adapter call per microbatch, all on the same layer
            w = synth.MULTI_WORKLOAD
            specs = [(s.rank, s.alpha, s.p) for s in w["specs"]]
            cap = m or w["total_rows"]
            lengths, ads = synth.sample_stream(w["seed"], 4 * cap, len(specs))
            batches = packer(lengths, ads, cap)
            self.m = cap
            base = synth.multi_inputs(w["seed"], w["k"], w["n"], w["specs"], synth.PackedBatch(m=128))
            self.parts, owners, valid_rows = [], [], []
            for b, mb in enumerate(batches):
                pb = synth.PackedBatch(m=cap, segments=mb["segments"], valid=mb["valid"])
                raw = synth.multi_inputs(w["seed"] + 1000 + b, w["k"], w["n"], w["specs"], pb)
                self.parts.append(Part(f"microbatch{b}", w["k"], w["n"], specs, w["seed"] + b, raw["X"], base["W"],
                                       raw["dY"], base["adapters"], list(mb["segments"]), x_key=f"X{b}"))
            self.n_samples = len(lengths)
            self.n_batches = len(batches)
            self.packed_rows = sum(mb["rows"] for mb in batches)
            self.valid_tokens = int(sum(lengths))
            self.token_count = [(i, lengths[i]) for i in range(len(lengths))]
            self.owner = None
            self.valid_rows = np.arange(self.valid_tokens)   # counts only; per-part rows are in the parts
            self.spec_tokens = [sum(l for l, a in zip(lengths, ads) if a == i) for i in range(len(specs))]
            # the CPU legs run the oracle on rows of the first microbatch
            mb0 = batches[0]
            self.cpu_parts = self.parts[:1]
            self.row_pool = np.concatenate([np.arange(st, st + v) for (st, _r, _a), v in zip(mb0["segments"],
                                                                                               mb0["valid"])])
            self.spec_rows = [sum(-(-l // 128) * 128 for l, a in zip(lengths, ads) if a == i)
                              for i in range(len(specs))]
        elif name in (MULTI, MULTI_SQ):
            if name == MULTI:
                w = synth.MULTI_WORKLOAD
                aspecs, rows = w["specs"], m or w["total_rows"]
            else:
                w = synth.MULTI_SWEEP_WORKLOAD
                aspecs, rows = synth.multi_sweep_specs(r or 16), m or 16384
            specs = [(s.rank, s.alpha, s.p) for s in aspecs]
            batch = synth.packed_batch(w["seed"], rows, len(specs))
            self.m = batch.m
            raw = synth.multi_inputs(w["seed"], w["k"], w["n"], aspecs, batch)
            self.owner = np.full(self.m, -1, dtype=np.int64)
            valid = []
            for (start, rows, a), v in zip(batch.segments, batch.valid):
                self.owner[start:start + rows] = a
                valid.append(np.arange(start, start + v))
            self.valid_rows = np.concatenate(valid) if valid else np.zeros(0, dtype=np.int64)
            self.parts = [Part("packed", w["k"], w["n"], specs, w["seed"], raw["X"], raw["W"], raw["dY"],
                               raw["adapters"], list(batch.segments))]
            self.n_samples = len(batch.segments)
        elif name == LAYER:
            cfg = dict(synth.LAYER_WORKLOAD)
            self.m = m or cfg["m"]
            r = r or cfg["r"]
            raw = synth.decoder_layer_inputs(cfg["seed"], self.m, r)
            self.parts = [Part(q["name"], q["k"], q["n"], [(r, cfg["alpha"], cfg["p"])], cfg["seed"] + i,
                               raw["X"][q["input"]], q["W"], q["dY"], [(q["A"], q["B"])], x_key=q["input"])
                          for i, q in enumerate(raw["parts"])]
            self.owner = np.zeros(self.m, dtype=np.int64)
            self.valid_rows = np.arange(self.m)
        else:
            cfg = dict(synth.WORKLOADS["llama8b_up" if name == DORA else name])
            if m:
                cfg["m"] = m
            if r:
                cfg["r"] = r
            self.m = cfg["m"]
            raw = synth.layer_inputs(cfg["seed"], self.m, cfg["k"], cfg["n"], cfg["r"])
            mag = None
            if name == DORA:
                # magnitudes near their initial values (the column norms of W), seeded
                Wf = (raw["W"].astype(np.uint32) << 16).view(np.float32)
                rng = np.random.Generator(np.random.PCG64(cfg["seed"] + 100))
                mag = (np.sqrt((Wf.astype(np.float64) ** 2).sum(0)) * rng.uniform(0.8, 1.2, cfg["n"])).astype(np.float32)
            self.parts = [Part(name, cfg["k"], cfg["n"], [(cfg["r"], cfg["alpha"], cfg["p"])], cfg["seed"],
                               raw["X"], raw["W"], raw["dY"], [(raw["A"], raw["B"])], mag=mag)]
            self.owner = np.zeros(self.m, dtype=np.int64)
            self.valid_rows = np.arange(self.m)

    @property
    def tokens(self) -> int:
        return int(self.valid_rows.size)

    @property
    def sample_pool(self):
        """Global rows the CPU legs sample from."""
        return getattr(self, "row_pool", self.valid_rows)

    def tokens_of(self, i: int) -> int:
        if self.name == GREEDY:
            return self.spec_tokens[i]
        return int(np.count_nonzero(self.owner[self.valid_rows] == i))

    def rows_of(self, i: int) -> int:
        """Rows (padding included) the kernels run adapter i on."""
        if self.name == GREEDY:
            return self.spec_rows[i]
        return int(np.count_nonzero(self.owner == i))

    def describe(self) -> str:
        if self.name == GREEDY:
            q = self.parts[0]
            ads = ", ".join(f"(r={r}, alpha={a}, p={p})" for r, a, p in q.specs)
            return (f"{self.name}: {self.n_samples} samples (lognormal lengths, {self.valid_tokens} tokens) packed "
                    f"first-fit decreasing into {self.n_batches} microbatches of {self.m} rows "
                    f"({self.packed_rows} rows used by tiles), k={q.k}, n={q.n}, adapters {ads}")
        if self.name in (MULTI, MULTI_SQ):
            q = self.parts[0]
            ads = ", ".join(f"(r={r}, alpha={a}, p={p})" for r, a, p in q.specs)
            return (f"{self.name}: packed multi-adapter LoRA linear, {self.m} padded rows ({self.n_samples} samples, "
                    f"lognormal lengths, {self.tokens} valid tokens), k={q.k}, n={q.n}, adapters {ads}, "
                    f"seed={q.seed}")
        if self.name == LAYER:
            r, alpha, p = self.parts[0].specs[0]
            shapes = ", ".join(f"{q.label} {q.k}x{q.n}" for q in self.parts)
            return (f"{self.name}: the seven LoRA linears of a Llama-3.1-8B decoder layer ({shapes}), m={self.m} "
                    f"tokens, r={r}, alpha={alpha}, p={p}; attention, norms and activations not included")
        q = self.parts[0]
        r, alpha, p = q.specs[0]
        kind = "DoRA linear (column magnitudes, norm held constant in the backward)" if q.mag is not None else "LoRA linear"
        return f"{self.name}: {kind} m={self.m} tokens, k={q.k}, n={q.n}, r={r}, alpha={alpha}, p={p}, seed={q.seed}"

    def layer_flops(self) -> int:
        """Algorithmic FLOPs of one fwd+bwd over the valid tokens: per linear 4Tkn + sum_i 6 T_i r_i (k+n)
        (W is frozen: no weight gradient).  Microbatches of one layer count as one linear."""
        F = 0
        for q in (self.parts[:1] if self.name == GREEDY else self.parts):
            F += 4 * self.tokens * q.k * q.n
            F += sum(6 * self.tokens_of(i) * r * (q.k + q.n) for i, (r, _, _) in enumerate(q.specs))
            if q.mag is not None:   # DoRA's column norm: U = W^T A (2knr) and G = A^T A (2kr^2)
                r = q.specs[0][0]
                F += 2 * q.k * q.n * r + 2 * q.k * r * r
        return F

    def layer_bytes(self) -> int:
        """Compulsory bf16 HBM bytes of one fwd+bwd over the valid tokens.

        Per linear, fwd: X, W, Y and per adapter A_i, B_i, S_i; bwd: dY, W, X,
        dX and per adapter S_i, A_i, B_i, dA_i, dB_i.
        """
        T = self.tokens
        total = 0
        for q in (self.parts[:1] if self.name == GREEDY else self.parts):
            k, n = q.k, q.n
            fwd = T * k + k * n + T * n
            bwd = T * n + k * n + 2 * T * k
            for i, (r, _, _) in enumerate(q.specs):
                Ti = self.tokens_of(i)
                fwd += k * r + r * n + Ti * r
                bwd += Ti * r + 2 * (k * r + r * n)
            if q.mag is not None:   # DoRA: W again for U; bwd reads Y and writes + reads dZ = dY * g
                fwd += k * n
                bwd += 3 * T * n
            total += fwd + bwd
        return 2 * total

    def gemm_flops_per_step(self, kind: str):
        """Algorithmic FLOPs of the frozen-weight GEMM launches of one kind (with their rank-r tails) in
        one step, over the rows they run."""
        if kind not in ("gemm_fwd", "gemm_bwd"):
            return None
        F = 0
        for j, q in enumerate(self.parts):
            out = q.n if kind == "gemm_fwd" else q.k
            F += 2 * self.m * q.k * q.n
            if self.name != GREEDY or j == 0:   # a packed global batch: the tails of all its rows, once
                F += sum(2 * self.rows_of(i) * r * out for i, (r, _, _) in enumerate(q.specs))
        return F

    def rank_bytes_per_step(self, kind: str, saved_mask: bool = False, deterministic: bool = False):
        """Algorithmic HBM bytes of one step's launches of a rank-r pass, over the rows they run (bf16 tensors;
        keep bits one bit an element): down_proj reads X and A_i and writes S' (and the keep bits when the
        forward keeps them); ds_db reads dY, S' and B_i (dY twice in the deterministic mode); da reads X, the
        keep bits (handed over by the dX GEMM, or the forward's) and dSq, and writes dA_i."""
        if kind not in ("down_proj", "ds_db", "da"):
            return None
        B = 0
        for q in (self.parts[:1] if self.name == GREEDY else self.parts):
            rows_i = [self.rows_of(i) for i in range(len(q.specs))]
            rows = sum(rows_i)
            ranks = [r for r, _, _ in q.specs]
            if kind == "down_proj":
                B += 2 * rows * q.k + sum(2 * q.k * r + 2 * t * r for t, r in zip(rows_i, ranks))
                B += rows * q.k // 8 if saved_mask else 0
            elif kind == "ds_db":
                B += 2 * rows * q.n * (2 if deterministic else 1)
                B += sum(2 * t * r + 2 * r * q.n for t, r in zip(rows_i, ranks))
            else:
                B += 2 * rows * q.k + rows * q.k // 8 + sum(2 * t * r + 2 * q.k * r for t, r in zip(rows_i, ranks))
        return B

    def resident_bytes(self) -> int:
        """Bytes of X, W, dY, Y and dX over all linears: what one step streams through L2."""
        m = self.m
        return sum(2 * (2 * m * q.k + q.k * q.n + 2 * m * q.n) for q in self.parts)


def oracle_step(wl: Workload):
    """fwd + bwd of the oracle on a sample of global rows of the workload (CPU legs only)."""
    from oracle import lora_oracle as O
    prepared = []
    for q in getattr(wl, "cpu_parts", wl.parts):
        ads = [dict(A=O.bf16_to_f64(A), B=O.bf16_to_f64(B), alpha=a, p=p)
               for (A, B), (_, a, p) in zip(q.adapters, q.specs)]
        prepared.append((q, O.bf16_to_f64(q.W), ads))

    def step(rows):
        for q, W, ads in prepared:
            X = O.bf16_to_f64(q.X[rows])
            dY = O.bf16_to_f64(q.dY[rows])
            if q.mag is not None:
                ad = ads[0]
                O.dora_forward(X, W, ad["A"], ad["B"], q.mag, ad["alpha"], ad["p"], q.seed, rows=rows)
                O.dora_backward(dY, X, W, ad["A"], ad["B"], q.mag, ad["alpha"], ad["p"], q.seed, rows=rows)
            elif q.single:
                ad = ads[0]
                O.lora_forward(X, W, ad["A"], ad["B"], ad["alpha"], ad["p"], q.seed, rows=rows)
                O.lora_backward(dY, X, W, ad["A"], ad["B"], ad["alpha"], ad["p"], q.seed, rows=rows)
            else:
                O.multi_lora_forward(X, W, ads, q.segments, q.seed, rows=rows)
                O.multi_lora_backward(dY, X, W, ads, q.segments, q.seed, rows=rows)

    return step


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Replicas:
    """The ranks of a replicas-only run: one process per GPU, each running the whole layer on its own
    tokens, with no collective on the data path.  The process group only lines the ranks up around a
    timed region and takes the slowest rank's time (tensors live on `device`: the GPU under NCCL, the
    CPU under gloo)."""

    def __init__(self, world: int, device):
        self.world, self.device = world, device

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())


def job_throughput(tokens_per_rank_step: int, steps: int, world: int, max_rank_ms: float) -> float:
    """Whole-job tokens/s: the tokens every rank processed over the slowest rank's time (weak scaling)."""
    return tokens_per_rank_step * steps * world / (max_rank_ms / 1e3)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
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
                                          "--format=csv,noheader,nounits", "-lms", "20"],
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

    def mark(self, what: str):
        """Wall-clock bounds of the timed region: samples outside them are not summarised."""
        setattr(self, what, time.time())

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
        import datetime
        t0, t1 = getattr(self, "start", None), getattr(self, "stop", None)
        sm, mx, pw, reasons, inside = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                vals = (float(parts[1]), float(parts[2]), float(parts[3]))
            except ValueError:
                continue
            if t0 is not None and t1 is not None and not (t0 - 0.025 <= ts <= t1 + 0.025):
                continue
            inside += 1
            sm.append(vals[0])
            mx.append(vals[1])
            pw.append(vals[2])
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample fell inside the timed region"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": inside, "power_w_max": max(pw), "sampling": "nvidia-smi every 20 ms, timed region only"}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` on `workload` from the committed ncu summary, or None if
    the kernel sources changed since the capture (or none exists)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    entry = data.get(workload, {}).get(kernel)
    if not entry:
        return None
    if entry.get("source_digest") != source_digest(entry.get("sources", [])):
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_packer(lengths, adapters, capacity):
    """The oracle's greedy packing, in the layout native.pack_microbatches returns (CPU legs only)."""
    from oracle import lora_oracle as O
    batch, row, nb = O.greedy_pack(lengths, capacity)
    out = [{"segments": [], "samples": [], "valid": [], "rows": 0} for _ in range(nb)]
    for i in sorted(range(len(lengths)), key=lambda i: (batch[i], row[i])):
        b = out[batch[i]]
        rows = O.padded_rows(lengths[i])
        b["segments"].append((row[i], rows, int(adapters[i])))
        b["samples"].append(i)
        b["valid"].append(int(lengths[i]))
        b["rows"] = row[i] + rows
    return out


def sample_rows(wl: Workload, rng, count: int):
    pool = wl.sample_pool
    count = int(np.clip(count, 1, pool.size))
    return np.sort(rng.choice(pool, size=count, replace=False))


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    wl = Workload(args.workload, args.m, args.r, packer=oracle_packer)
    step = oracle_step(wl)
    rng = np.random.default_rng(0)
    probe = sample_rows(wl, rng, 32)
    t0 = time.perf_counter()
    step(probe)
    t_probe = time.perf_counter() - t0
    budget = min(args.ref_step_seconds, 150.0 / max(1, args.steps + args.warmup))
    rows_per_step = int(np.clip(probe.size * budget / max(t_probe, 1e-3), 16, wl.tokens))
    times = []
    for i in range(args.warmup + args.steps):
        rows = sample_rows(wl, rng, rows_per_step)
        t0 = time.perf_counter()
        step(rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = rows_per_step * len(times) / total
    cores = os.cpu_count()
    sample = (f"{rows_per_step} random valid rows of the {wl.m}-row batch per step (Y, S, dX rows and their "
              f"dA/dB contributions; keep mask regenerated), fp64 numpy/BLAS")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.describe(), "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_leg(wl: Workload, seconds: float):
    """The oracle as it stands on a bounded row sample of the same workload (rank 0, N=1)."""
    step = oracle_step(wl)
    rng = np.random.default_rng(1)
    probe = sample_rows(wl, rng, 32)
    t0 = time.perf_counter()
    step(probe)
    tp = time.perf_counter() - t0
    rows = sample_rows(wl, rng, int(probe.size * seconds / max(tp, 1e-3)))
    t0 = time.perf_counter()
    step(rows)
    dt = time.perf_counter() - t0
    return {"value": rows.size / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows.size} of {wl.tokens} valid rows, one fwd+bwd pass (fp64 numpy/BLAS), {dt:.1f} s"}


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

class DeviceProblem:
    """The workload's tensors on the GPU plus pinned host copies, and one step through the C ABI."""

    def __init__(self, wl: Workload, dev, stream, saved_mask: bool = False):
        import torch

        from lora_fine_tuning_gb300 import api
        self.wl, self.dev, self.stream, self.api = wl, dev, stream, api
        bf = torch.bfloat16

        def pinned(a):
            return torch.from_numpy(a.view(np.int16)).view(bf).pin_memory()

        m = wl.m
        self.inputs = {}   # name -> (pinned host, device); shared inputs appear once
        self.parts = []
        shared = {}        # one device copy of a weight that several linears (microbatches) use

        def weight(a):
            if id(a) not in shared:
                shared[id(a)] = pinned(a).to(dev)
            return shared[id(a)]

        ws_need = (0, None)
        for q in wl.parts:
            if q.x_key not in self.inputs:
                h = pinned(q.X)
                self.inputs[q.x_key] = (h, h.to(dev))
            dYh = pinned(q.dY)
            self.inputs["dY:" + q.label] = (dYh, dYh.to(dev))
            d = dict(part=q, X=self.inputs[q.x_key][1], dY=self.inputs["dY:" + q.label][1],
                     W=weight(q.W), Y=torch.empty((m, q.n), dtype=bf, device=dev),
                     dX=torch.empty((m, q.k), dtype=bf, device=dev),
                     S=torch.empty((m, q.r_max), dtype=bf, device=dev),
                     # keep bits written by the forward and read by the backward (saved-mask mode only;
                     # otherwise the backward regenerates the mask from the seed)
                     M=torch.empty((m, q.k // 8), dtype=torch.uint8, device=dev) if saved_mask else None,
                     adapters=[api.Adapter(A=weight(A), B=weight(B), alpha=a, p=p,
                                           dA=torch.empty((q.k, r), dtype=bf, device=dev),
                                           dB=torch.empty((r, q.n), dtype=bf, device=dev))
                               for (A, B), (r, a, p) in zip(q.adapters, q.specs)])
            if q.mag is not None:
                d["mag"] = torch.from_numpy(q.mag).to(dev)
                d["wn2"] = api.dora_weight_norm2(d["W"])          # W is frozen: once, outside any timed region
                d["g"] = torch.empty(q.n, dtype=torch.float32, device=dev)
                d["dmag"] = torch.empty(q.n, dtype=torch.float32, device=dev)
                d["dZ"] = torch.empty((m, q.n), dtype=bf, device=dev)
            self.parts.append(d)
            size = api.lora_workspace_size(m, q.k, q.n, max(8, q.r_max), len(q.adapters))
            if size > ws_need[0]:
                ws_need = (size, (m, q.k, q.n, max(8, q.r_max), len(q.adapters)))
        if any(q.mag is not None for q in wl.parts):
            q = wl.parts[0]
            self.ws = api.dora_workspace(m, q.k, q.n, q.r_max, device=dev)
        else:
            self.ws = api.workspace(*ws_need[1], device=dev)

    def _fwd(self, d):
        api, q, s = self.api, d["part"], self.stream
        if q.mag is not None:
            a = d["adapters"][0]
            api.dora_fwd(d["X"], d["W"], a.A, a.B, d["mag"], d["wn2"], a.alpha, a.p, q.seed, Y=d["Y"],
                         S_saved=d["S"], g_saved=d["g"], mask_bits=d["M"], ws=self.ws, stream=s)
        elif q.single:
            a = d["adapters"][0]
            api.lora_fwd(d["X"], d["W"], a.A, a.B, a.alpha, a.p, q.seed, Y=d["Y"], S_saved=d["S"],
                         mask_bits=d["M"], ws=self.ws, stream=s)
        else:
            api.multi_lora_fwd(d["X"], d["W"], d["adapters"], q.segments, q.seed, Y=d["Y"], S_saved=d["S"],
                               mask_bits=d["M"], ws=self.ws, stream=s)

    def _bwd(self, d):
        api, q, s = self.api, d["part"], self.stream
        if q.mag is not None:
            a = d["adapters"][0]
            api.dora_bwd(d["dY"], d["X"], d["W"], a.A, a.B, d["S"], d["Y"], d["mag"], d["g"], a.alpha, a.p, q.seed,
                         dX=d["dX"], dA=a.dA, dB=a.dB, dmag=d["dmag"], dZ=d["dZ"], ws=self.ws, stream=s,
                         mask_bits=d["M"])
        elif q.single:
            a = d["adapters"][0]
            api.lora_bwd(d["dY"], d["X"], d["W"], a.A, a.B, d["S"], a.alpha, a.p, q.seed, dX=d["dX"], dA=a.dA,
                         dB=a.dB, ws=self.ws, stream=s, mask_bits=d["M"])
        else:
            api.multi_lora_bwd(d["dY"], d["X"], d["W"], d["adapters"], q.segments, q.seed, d["S"], dX=d["dX"],
                               ws=self.ws, stream=s, mask_bits=d["M"])

    def step(self):
        for d in self.parts:
            self._fwd(d)
        for d in reversed(self.parts):
            self._bwd(d)

    def part_step(self, d):
        self._fwd(d)
        self._bwd(d)

    def part_frozen(self, d):
        api, s = self.api, self.stream
        api.multi_lora_fwd(d["X"], d["W"], [], [], 0, Y=d["Y"], ws=self.ws, stream=s)
        api.multi_lora_bwd(d["dY"], d["X"], d["W"], [], [], 0, None, dX=d["dX"], ws=self.ws, stream=s)

    def part_torch(self, d):
        import torch
        torch.matmul(d["X"], d["W"], out=d["Y"])
        torch.matmul(d["dY"], d["W"].t(), out=d["dX"])

    def frozen_step(self):
        """The same linears with no adapter: Y = X W and dX = dY W^T through the same GEMM kernels."""
        api, s = self.api, self.stream
        for d in self.parts:
            api.multi_lora_fwd(d["X"], d["W"], [], [], 0, Y=d["Y"], ws=self.ws, stream=s)
        for d in reversed(self.parts):
            api.multi_lora_bwd(d["dY"], d["X"], d["W"], [], [], 0, None, dX=d["dX"], ws=self.ws, stream=s)

    def torch_frozen_step(self):
        import torch
        for d in self.parts:
            torch.matmul(d["X"], d["W"], out=d["Y"])
        for d in reversed(self.parts):
            torch.matmul(d["dY"], d["W"].t(), out=d["dX"])

    def outputs(self):
        out = []
        for d in self.parts:
            out += [d["Y"], d["dX"]]
            for a in d["adapters"]:
                out += [a.dA, a.dB]
            if "dmag" in d:
                out.append(d["dmag"])
        return out

    def status(self) -> int:
        return self.api.lora_device_status(self.ws, self.stream)


WAIT_KERNELS = {1: "down_proj", 2: "gemm_fwd", 3: "gemm_bwd", 4: "ds_db", 5: "da", 6: "debug"}


def check_status(prob, where: str) -> None:
    """Raise if a kernel gave up a bounded wait (the workspace status word: kernel id << 8 | wait site)."""
    code = prob.status()
    if code != 0:
        raise RuntimeError(f"a kernel reported a bounded-wait timeout {where}: status 0x{code:x} "
                           f"({WAIT_KERNELS.get(code >> 8, 'unknown kernel')}, wait site {code & 0xFF})")


def timed_loop(fn, steps, stream, flush=None):
    """Device milliseconds of `steps` calls of fn, on `stream`.  With `flush`, L2 is overwritten
    before every call and only the calls themselves are timed (per-call event pairs)."""
    import torch
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    pairs = []
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.add_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs)


def e2e_leg(prob_a, prob_b, wl, dev, stream, steps, barrier, max_over_ranks, ws_n):
    """Steps through the public API with every step's inputs copied in from pinned host memory and its
    results copied back, all inside the timed region.

    Two buffer sets alternate between steps.  A host-to-device stream prefetches the inputs of step
    i+1, and a device-to-host stream drains the outputs of step i-1, while step i computes on the
    launch stream.  Events order each copy after the compute that frees its buffers.  A serial
    variant (copy in, compute, copy out, one stream) is timed too.
    """
    import torch
    sets = [prob_a, prob_b]
    outs = [p.outputs() for p in sets]
    hosts = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o] for o in outs]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def copy_in(b):
        with torch.cuda.stream(h2d_s):
            for h, t in sets[b].inputs.values():
                t.copy_(h, non_blocking=True)
        ev_in[b].record(h2d_s)

    def pipelined(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)
        copy_in(0)
        if n > 1:
            copy_in(1)
        for i in range(n):
            b = i & 1
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])      # outputs of step i-2 are on the host
            sets[b].step()
            ev_comp[b].record(stream)
            d2h_s.wait_event(ev_comp[b])
            with torch.cuda.stream(d2h_s):
                for h, t in zip(hosts[b], outs[b]):
                    h.copy_(t, non_blocking=True)
            ev_out[b].record(d2h_s)
            if i + 2 < n:
                h2d_s.wait_event(ev_comp[b])      # step i no longer reads buffer set b
                copy_in(b)
        stream.wait_event(ev_out[(n - 1) & 1])
        if n > 1:
            stream.wait_event(ev_out[n & 1])
        end.record(stream)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end)

    def serial():
        for h, t in sets[0].inputs.values():
            t.copy_(h, non_blocking=True)
        sets[0].step()
        for h, t in zip(hosts[0], outs[0]):
            h.copy_(t, non_blocking=True)

    pipelined(2)
    serial()
    torch.cuda.synchronize(dev)
    barrier()
    ms = max_over_ranks(pipelined(steps))
    barrier()
    ms_serial = max_over_ranks(timed_loop(serial, steps, stream))
    for p in sets:
        check_status(p, "in the end-to-end leg")
    h2d = sum(h.numel() * h.element_size() for h, _ in sets[0].inputs.values())
    d2h = sum(h.numel() * h.element_size() for h in hosts[0])
    return {"value": job_throughput(wl.tokens, steps, ws_n, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / steps, "steps": steps,
            "overlap": "inputs of step i+1 and outputs of step i-1 copied on two copy streams while step i runs",
            "serial_ms_per_step": ms_serial / steps,
            "serial_value": job_throughput(wl.tokens, steps, ws_n, ms_serial)}


def run_native(args):
    import torch
    import torch.distributed as dist

    from lora_fine_tuning_gb300 import native

    ws_n, rank, local = dist_env()
    if ws_n > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = Workload(args.workload, args.m, args.r, packer=native.pack_microbatches)
    stream = torch.cuda.current_stream(dev)
    from lora_fine_tuning_gb300 import api
    api.lora_set_deterministic(args.deterministic)   # before any workspace is sized
    prob = DeviceProblem(wl, dev, stream, args.saved_mask)

    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if wl.resident_bytes() < 2 * l2_bytes:
        flush = torch.empty(max(2 * l2_bytes, 256 << 20) // 4, dtype=torch.int32, device=dev)
        l2_note = (f"L2 flushed before every step (write of a {flush.numel() * 4 >> 20} MiB buffer, outside the "
                   f"timed events): X/W/dY/Y/dX total {wl.resident_bytes() / 1e6:.0f} MB")
    else:
        l2_note = (f"no flush: X/W/dY/Y/dX total {wl.resident_bytes() / 1e6:.0f} MB, larger than twice L2 "
                   f"({l2_bytes >> 20} MiB)")

    replicas = Replicas(ws_n, dev)
    barrier, max_over_ranks = replicas.barrier, replicas.max

    for _ in range(args.warmup):
        prob.step()
    torch.cuda.synchronize(dev)
    check_status(prob, "during warm-up")

    # --- timed region (device, inputs resident in HBM, nothing between the library's launches) ---
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize(dev)
        clocks.mark("start")
        elapsed_ms = timed_loop(prob.step, args.steps, stream, flush)
        clocks.mark("stop")
        barrier()
    elapsed_ms = max_over_ranks(elapsed_ms)
    clk = clocks.summary()
    check_status(prob, "in the timed region")

    # --- sustained: the same step repeated for at least --sustained-seconds, so that the clock has settled
    # under the power cap; its own clock summary ---
    sustained = None
    if not args.no_sustained:
        sus_steps = max(args.steps, math.ceil(args.sustained_seconds * 1e3 * args.steps / max(elapsed_ms, 1e-6)))
        with ClockSampler(local) as sclocks:
            barrier()
            torch.cuda.synchronize(dev)
            sclocks.mark("start")
            sus_ms = timed_loop(prob.step, sus_steps, stream, flush)
            sclocks.mark("stop")
            barrier()
        sus_ms = max_over_ranks(sus_ms)
        check_status(prob, "in the sustained region")
        sustained = {"steps": sus_steps, "seconds": sus_ms / 1e3, "ms_per_step": sus_ms / sus_steps,
                     "value": job_throughput(wl.tokens, sus_steps, ws_n, sus_ms), "unit": UNIT,
                     "clocks": sclocks.summary()}

    # --- per-kernel breakdown: a second timed region of the same steps with an event pair around every
    # launch (on the launch stream); the events also keep consecutive kernels from overlapping ---
    torch.cuda.synchronize(dev)
    native.timing_begin()
    instrumented_ms = timed_loop(prob.step, args.steps, stream, flush)
    kernel_times = native.timing_end()
    check_status(prob, "in the instrumented region")

    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(wl.tokens, args.steps, ws_n, elapsed_ms)

    # --- end to end through the public API with host buffers ---
    e2e = None
    if not args.no_e2e:
        e2e = e2e_leg(prob, DeviceProblem(wl, dev, stream, args.saved_mask), wl, dev, stream, max(4, min(args.steps, 20)),
                      barrier, max_over_ranks, ws_n)

    # --- frozen-layer reference points (overhead of the LoRA branch) ---
    frozen = None
    if not args.no_frozen:
        reps = args.steps   # same length as the timed LoRA loop, so both see the same clock behaviour
        res = {}
        frozen_kernels = {}
        for label, fn in (("ours", prob.frozen_step), ("torch_matmul", prob.torch_frozen_step)):
            fn()
            torch.cuda.synchronize(dev)
            res[label] = max_over_ranks(timed_loop(fn, reps, stream, flush)) / reps
        # per-launch times from a separate loop: the events between launches would otherwise be in the
        # frozen step's own time (they also keep consecutive kernels from overlapping)
        native.timing_begin()
        timed_loop(prob.frozen_step, min(reps, 20), stream, flush)
        frozen_kernels = {kname: t / max(1, cnt) for kname, (t, cnt) in native.timing_end().items()}
        frozen = {"frozen_ms_per_step_ours": res["ours"], "frozen_ms_per_step_torch": res["torch_matmul"],
                  "frozen_ms_per_launch_ours": frozen_kernels,
                  "lora_overhead_vs_ours": ms_per_step / res["ours"],
                  "lora_overhead_vs_torch": ms_per_step / res["torch_matmul"]}

    # --- per projection (workloads of several linears): each one's fwd+bwd alone, its frozen GEMMs alone ---
    per_projection = None
    if wl.name == LAYER and not args.no_frozen:
        peaks_pp, _ = load_peaks()
        per_projection = []
        for d in prob.parts:
            q = d["part"]
            t = {}
            for label, fn in (("lora", prob.part_step), ("frozen_ours", prob.part_frozen),
                              ("frozen_torch", prob.part_torch)):
                fn(d)
                torch.cuda.synchronize(dev)
                t[label] = max_over_ranks(timed_loop(lambda: fn(d), args.steps, stream, flush)) / args.steps
            r = q.specs[0][0]
            flops = 4 * wl.tokens * q.k * q.n + 6 * wl.tokens * r * (q.k + q.n)
            per_projection.append({
                "projection": q.label, "k": q.k, "n": q.n, "r": r, "ms_lora": t["lora"],
                "ms_frozen_ours": t["frozen_ours"], "ms_frozen_torch": t["frozen_torch"],
                "overhead_vs_ours": t["lora"] / t["frozen_ours"], "overhead_vs_torch": t["lora"] / t["frozen_torch"],
                "tflops": flops / (t["lora"] / 1e3) / 1e12,
                "frac_of_measured_peak": flops / (t["lora"] / 1e3) / 1e12 / peaks_pp["bf16_tflops"]})

    if rank != 0:
        return

    peaks, peak_kind = load_peaks()
    side_kinds = SIDE_STREAM_KINDS_SAVED_MASK if args.saved_mask else set()
    # the instrumented window's length decides which measured peak applies: the burst figure for a
    # short window, the seconds-long (power-capped) figure for a long one
    long_window = instrumented_ms / 1e3 >= SUSTAINED_SECONDS
    tensor_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) if long_window else peaks["bf16_tflops"]
    # dominant kernel: the largest summed device time among the kernels on the launch stream
    dom_name, (dom_ms, dom_launches) = max(((kn, tc) for kn, tc in kernel_times.items()
                                            if kn not in side_kinds), key=lambda kv: kv[1][0])
    dom_flops = wl.gemm_flops_per_step(dom_name)
    if dom_flops is not None:
        # FLOPs of all its launches over their summed device time (one launch per step for one linear)
        achieved = dom_flops * args.steps / (dom_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": achieved / tensor_peak, "traffic": profiled_traffic(dom_name, wl.name),
                    "peak_source": (f"{peak_kind} bf16, "
                                    f"{'sustained (seconds-long window)' if long_window else 'burst (short window)'}"),
                    "window_s": instrumented_ms / 1e3,
                    "frac_of_datasheet": achieved / DATASHEET_PEAKS["bf16_tflops"],
                    "datasheet_peak": DATASHEET_PEAKS["bf16_tflops"]}
    else:
        roofline = {"bound": "hbm", "kernel": dom_name, "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": None, "traffic": None}

    F, Bc = wl.layer_flops(), wl.layer_bytes()
    t_roof = max(F / (peaks["bf16_tflops"] * 1e12), Bc / (peaks["hbm_gbs"] * 1e9))
    t_sheet = max(F / (DATASHEET_PEAKS["bf16_tflops"] * 1e12), Bc / (DATASHEET_PEAKS["hbm_gbs"] * 1e9))
    layer_roof = {"flops": F, "compulsory_bytes": Bc, "roofline_ms": t_roof * 1e3,
                  "frac": t_roof * 1e3 / ms_per_step,
                  "peak_source": f"{peak_kind} (burst bf16 {peaks['bf16_tflops']} TFLOP/s, copy {peaks['hbm_gbs']} GB/s)",
                  "achieved_tflops": F / (ms_per_step / 1e3) / 1e12,
                  "roofline_ms_datasheet": t_sheet * 1e3, "frac_of_datasheet": t_sheet * 1e3 / ms_per_step,
                  "datasheet_peaks": dict(DATASHEET_PEAKS)}
    if sustained is not None:
        t_sus = max(F / (peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12),
                    Bc / (peaks["hbm_gbs"] * 1e9))
        sustained["layer_roofline_frac"] = t_sus * 1e3 / sustained["ms_per_step"]
        sustained["layer_roofline_frac_of_datasheet"] = t_sheet * 1e3 / sustained["ms_per_step"]
        sustained["peak_source"] = f"{peak_kind} sustained bf16 {peaks.get('bf16_tflops_sustained')} TFLOP/s"

    kernels = {}
    for kname, (t, cnt) in sorted(kernel_times.items(), key=lambda kv: -kv[1][0]):
        if kname in side_kinds:
            kernels[kname] = {"ms_fork_to_end": t / max(1, cnt), "launches": cnt,
                              "stream": "side stream, concurrent with gemm_bwd"}
        else:
            kernels[kname] = {"ms_per_launch": t / max(1, cnt), "launches": cnt,
                              "share": t / max(1e-9, instrumented_ms)}
            nbytes = wl.rank_bytes_per_step(kname, args.saved_mask, args.deterministic)
            if nbytes is not None and t > 0:
                gbs = nbytes * args.steps / (t / 1e3) / 1e9
                kernels[kname].update({"algorithmic_bytes_per_step": nbytes, "achieved_gbs": gbs,
                                       "frac_of_hbm": gbs / peaks["hbm_gbs"]})
    gpu_launches = sum(cnt for kname, (t, cnt) in kernel_times.items() if kname != "memset")

    cpu = None
    if ws_n == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_leg(wl, args.cpu_seconds)

    config = {"workload": wl.describe(), "m": wl.m, "k": [q.k for q in wl.parts], "n": [q.n for q in wl.parts],
              "r": [[r for r, _, _ in q.specs] for q in wl.parts], "tokens_per_step": wl.tokens,
              "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU", "l2": l2_note,
              "saved_for_backward": ("S_saved and the keep bits (m x k/8 bytes) written by the forward"
                                     if args.saved_mask else "S_saved; the backward regenerates the keep mask from the seed"),
              "reductions": ("deterministic: fixed-order sums of per-CTA partials, dY read twice" if args.deterministic
                             else "fp32 atomic reductions of per-CTA partials")}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, Llama-shaped)", "config": config,
            "roofline": roofline, "layer_roofline": layer_roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": gpu_launches, "kernels": kernels,
            "kernel_timing": {"ms_per_step_instrumented": instrumented_ms / args.steps,
                              "how": "second run of the same steps with CUDA events around each launch"},
            "clocks": clk}
    if sustained:
        line["sustained"] = sustained
    if frozen:
        line["frozen"] = frozen
    if per_projection:
        line["per_projection"] = per_projection
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(synth.WORKLOADS) + [MULTI, MULTI_SQ, GREEDY, LAYER, DORA])
    ap.add_argument("--m", type=int, default=None,
                    help="override the workload's token count (padded rows for the packed workload)")
    ap.add_argument("--r", type=int, default=None,
                    help="override the rank of a single-adapter workload (multi_square4096: every adapter's rank)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline leg")
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-frozen", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sustained", action="store_true", help="skip the seconds-long sustained leg")
    ap.add_argument("--sustained-seconds", type=float, default=SUSTAINED_SECONDS,
                    help="minimum length of the sustained leg's timed window")
    ap.add_argument("--saved-mask", action="store_true",
                    help="the forward writes the keep bits and the backward reads them (default: regenerated)")
    ap.add_argument("--deterministic", action="store_true",
                    help="bit-reproducible reductions (lora_set_deterministic(1)): fixed-order sums, a second dY read")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
