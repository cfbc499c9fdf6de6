"""Seeded synthetic inputs for the LoRA linear layer.

This module only draws numbers and lays out packed batches. It holds none of
the layer's arithmetic (no dropout, no products, no routing): both the CUDA
path and the CPU oracle consume what it returns.

Value distributions follow the workloads the LoRAFusion write-ups benchmark
(Llama-shaped linear layers, rank 16..128, several adapters sharing one
frozen weight, variable-length summarisation samples packed into
microbatches):

* X, dY ~ N(0, 1)
* W ~ N(0, 1/k)           (frozen base weight, k x n, row-major)
* A ~ U(-1/sqrt(k), 1/sqrt(k))   (k x r)
* B ~ N(0, 0.02^2)        (r x n; nonzero so the branch is exercised)

Everything is returned as bf16 bit patterns (numpy uint16), rounded from
float32 to nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

TILE_ROWS = 128


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x)


def _uniform(rng: np.random.Generator, shape, bound: float) -> np.ndarray:
    x = rng.random(size=shape, dtype=np.float32)
    x = (x * np.float32(2.0) - np.float32(1.0)) * np.float32(bound)
    return f32_to_bf16_bits(x)


def adapter_weights(rng: np.random.Generator, k: int, n: int, r: int):
    """LoRA factors A (k x r) and B (r x n) as bf16 bits."""
    A = _uniform(rng, (k, r), 1.0 / math.sqrt(k))
    B = _normal(rng, (r, n), 0.02)
    return A, B


def layer_inputs(seed: int, m: int, k: int, n: int, r: int, *, with_grad: bool = True):
    """X (m x k), W (k x n), A (k x r), B (r x n) and optionally dY (m x n)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {}
    out["W"] = _normal(rng, (k, n), 1.0 / math.sqrt(k))
    out["A"], out["B"] = adapter_weights(rng, k, n, r)
    out["X"] = _normal(rng, (m, k), 1.0)
    if with_grad:
        out["dY"] = _normal(rng, (m, n), 1.0)
    return out


@dataclass
class AdapterSpec:
    rank: int
    alpha: float
    p: float


@dataclass
class PackedBatch:
    """A packed multi-adapter microbatch.

    segments: list of (row_start, rows, adapter); each sample is one segment
    whose rows are the sample length rounded up to whole 128-row tiles.
    valid: the unpadded sample length of each segment.
    Rows of a segment beyond its valid length are padding and hold zeros in X
    and dY.
    """
    m: int
    segments: list = field(default_factory=list)
    valid: list = field(default_factory=list)

    @property
    def valid_tokens(self) -> int:
        return int(sum(self.valid))


def packed_batch(seed: int, total_rows: int, n_adapters: int, *, mu: float = 6.2, sigma: float = 0.6,
                 lo: int = 64, hi: int = 2048) -> PackedBatch:
    """Sample lengths ~ lognormal(mu, sigma) clipped to [lo, hi], adapter ids uniform.

    Samples are packed in draw order, each padded to whole 128-row tiles, until
    `total_rows` rows are filled; the last sample is truncated to fit.
    """
    if total_rows % TILE_ROWS:
        raise ValueError("total_rows must be a multiple of 128")
    rng = np.random.Generator(np.random.PCG64(seed))
    batch = PackedBatch(m=total_rows)
    row = 0
    while row < total_rows:
        length = int(np.clip(np.round(rng.lognormal(mu, sigma)), lo, hi))
        adapter = int(rng.integers(0, n_adapters))
        rows = -(-length // TILE_ROWS) * TILE_ROWS
        rows = min(rows, total_rows - row)
        length = min(length, rows)
        batch.segments.append((row, rows, adapter))
        batch.valid.append(length)
        row += rows
    return batch


def sample_stream(seed: int, target_rows: int, n_adapters: int, *, mu: float = 6.2, sigma: float = 0.6,
                  lo: int = 64, hi: int = 2048):
    """Samples of a global batch: lengths ~ lognormal(mu, sigma) clipped to [lo, hi] and uniform adapter
    ids, drawn until their tile-padded rows reach target_rows.  Returns (lengths, adapters)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths, adapters, rows = [], [], 0
    while rows < target_rows:
        length = int(np.clip(np.round(rng.lognormal(mu, sigma)), lo, hi))
        lengths.append(length)
        adapters.append(int(rng.integers(0, n_adapters)))
        rows += -(-length // TILE_ROWS) * TILE_ROWS
    return lengths, adapters


def multi_inputs(seed: int, k: int, n: int, specs: list, batch: PackedBatch, *, with_grad: bool = True):
    """Shared W, per-adapter (A_i, B_i), and X / dY with zero padding rows."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = batch.m
    out = {"W": _normal(rng, (k, n), 1.0 / math.sqrt(k))}
    out["adapters"] = [adapter_weights(rng, k, n, s.rank) for s in specs]
    X = _normal(rng, (m, k), 1.0)
    dY = _normal(rng, (m, n), 1.0) if with_grad else None
    for (start, rows, _a), v in zip(batch.segments, batch.valid):
        X[start + v:start + rows] = 0
        if dY is not None:
            dY[start + v:start + rows] = 0
    out["X"] = X
    if with_grad:
        out["dY"] = dY
    return out


# Workloads of the benchmark suite for this layer, by name.
WORKLOADS = {
    "tiny": dict(m=256, k=512, n=512, r=16, alpha=2.0, p=0.1, seed=0),
    "llama8b_up": dict(m=8192, k=4096, n=14336, r=16, alpha=2.0, p=0.1, seed=1),
    "llama70b_o_r16": dict(m=16384, k=8192, n=8192, r=16, alpha=2.0, p=0.1, seed=2),
    "llama70b_o_r64": dict(m=16384, k=8192, n=8192, r=64, alpha=2.0, p=0.1, seed=2),
    "llama70b_up_r16": dict(m=16384, k=8192, n=28672, r=16, alpha=2.0, p=0.1, seed=2),
    "llama70b_up_r64": dict(m=16384, k=8192, n=28672, r=64, alpha=2.0, p=0.1, seed=2),
    # the Llama-3.1-8B MLP down-projection alone (k > n: the backward GEMM's K is n = 4096)
    "llama8b_down": dict(m=8192, k=14336, n=4096, r=16, alpha=2.0, p=0.1, seed=11),
    # square 4096 layer for sweeps over the token count and the rank
    "square4096": dict(m=4096, k=4096, n=4096, r=16, alpha=2.0, p=0.1, seed=4),
}

# all seven projections of a Llama-3.1-8B decoder layer, one adapter each
LAYER_WORKLOAD = dict(m=8192, r=16, alpha=2.0, p=0.1, seed=5)

# The seven projections of one Llama-3.1-8B decoder layer (hidden 4096, MLP 14336,
# 32 query heads and 8 key/value heads of width 128): (name, k, n, input).  The
# projections that read the same activation share it: q/k/v the attention input,
# gate/up the MLP input.
LLAMA8B_LAYER = [("q_proj", 4096, 4096, "attn_in"), ("k_proj", 4096, 1024, "attn_in"),
                 ("v_proj", 4096, 1024, "attn_in"), ("o_proj", 4096, 4096, "attn_out"),
                 ("gate_proj", 4096, 14336, "mlp_in"), ("up_proj", 4096, 14336, "mlp_in"),
                 ("down_proj", 14336, 4096, "mlp_act")]


def decoder_layer_inputs(seed: int, m: int, r: int):
    """Inputs of the seven LoRA linears of one decoder layer for m tokens.

    Returns {"X": {input name: m x k}, "parts": [dict(name, k, n, input, W, A, B, dY)]},
    every tensor seeded from `seed` and the projection's position.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    xs = {}
    for _name, k, _n, src in LLAMA8B_LAYER:
        if src not in xs:
            xs[src] = _normal(rng, (m, k), 1.0)
    parts = []
    for name, k, n, src in LLAMA8B_LAYER:
        W = _normal(rng, (k, n), 1.0 / math.sqrt(k))
        A, B = adapter_weights(rng, k, n, r)
        parts.append(dict(name=name, k=k, n=n, input=src, W=W, A=A, B=B, dY=_normal(rng, (m, n), 1.0)))
    return {"X": xs, "parts": parts}


MULTI_WORKLOAD = dict(k=8192, n=8192, total_rows=16384, seed=3,
                      specs=[AdapterSpec(16, 1.0, 0.0), AdapterSpec(16, 2.0, 0.1),
                             AdapterSpec(32, 2.0, 0.1), AdapterSpec(64, 4.0, 0.05)])


# The rank sweep on a square 4096 layer in its four-adapter form: every adapter at the swept rank, the
# multi-adapter workload's scales {1, 2, 2, 4}, drop rate 0.1 for all, lognormal sample lengths packed to
# the swept token count.
MULTI_SWEEP_WORKLOAD = dict(k=4096, n=4096, seed=4, alphas=(1.0, 2.0, 2.0, 4.0), p=0.1)


def multi_sweep_specs(r: int) -> list:
    """Adapter settings of the four-adapter sweep at rank r."""
    return [AdapterSpec(r, a, MULTI_SWEEP_WORKLOAD["p"]) for a in MULTI_SWEEP_WORKLOAD["alphas"]]
