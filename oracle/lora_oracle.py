"""fp64 CPU oracle for the LoRA linear layer, forward and backward, one or many adapters.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this module. It shares no code with the CUDA
library (it never imports `lora_fine_tuning_gb300` beyond what callers hand
it as plain arrays) and it is never on the product path.

What it computes, and where each step comes from:

* The layer (Eurosys26 LoRAFusion article, juhe.plus, section 2 "background":
  the LoRA formula):  Y = X W + alpha * (X A) B = X W + alpha * S B, with
  W (k x n) frozen and only A (k x r), B (r x n) trained.
* Dropout sits on the branch input only (LoRAFusion notes, papers.chlience.com,
  section 3 "thinking path" and section 5 "FusedLoRA": S = X_hat A, dropout fused
  with the down-projection).  The pages fix neither the random source nor the
  scaling; the readings taken here are: inverted dropout (kept elements scaled
  by q = 1/(1-p)); keep decisions drawn from Philox4x32-10 (Salmon, Moraes,
  Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) keyed by
  the 64-bit seed, with counter (row, feature // 8, 0, 0); the four 32-bit
  output words give eight 16-bit lanes, lane e (low half first) deciding
  feature 8*g + e, kept iff lane >= T with T = floor(p * 65536 + 0.5).
* Gradients are those of the definition with W frozen (the same notes,
  section 5: dS/dB share dY, the base-gradient path and the LoRA path are
  fused; "reading goals and judgement boundary": the kernels are designed to
  be lossless, i.e. they compute exactly these gradients up to rounding):
      dS = alpha dY B^T,  dB = alpha S^T dY,  dA = X_hat^T dS,
      dX = dY W^T + (D q) * (dS A^T).
* Multi-adapter (LoRAFusion notes, section 5 "FusedMultiLoRA"; the article,
  section 4.1): every 128-row tile carries one adapter id and that adapter's
  rank, scale and dropout rate; the frozen product is shared by all rows and
  gradients are routed back to each tile's own adapter.  A row that no
  segment covers uses no adapter.

Everything is float64; bf16 inputs are widened exactly.  Matrix products use
numpy's matmul as a library primitive, with no blocking or reordering beyond
the formulas above.
"""
from __future__ import annotations

import math

import numpy as np

TILE_ROWS = 128

# ---------------------------------------------------------------------------
# bf16 handling
# ---------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of an IEEE float32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# Philox-4xW (Salmon et al., SC'11): counter-based bijection, 10 rounds
# ---------------------------------------------------------------------------

# Round multipliers and Weyl key increments published with the generator for
# word widths 32 and 64.  The increments are the golden ratio and sqrt(3)-1
# scaled to the word width (the tests recompute them from those closed forms).
PHILOX = {
    32: dict(M0=0xD2511F53, M1=0xCD9E8D57, W0=0x9E3779B9, W1=0xBB67AE85),
    64: dict(M0=0xD2E7470EE14C6C93, M1=0xCA5A826395121157,
             W0=0x9E3779B97F4A7C15, W1=0xBB67AE8584CAA73B),
}


def philox4_scalar(counter, key, width: int = 32, rounds: int = 10):
    """Philox-4xW on Python integers, for any word width in PHILOX.

    One round: the words are paired as (x0, x3) under multiplier M0 and key
    word 1, and (x2, x1) under M1 and key word 0; each pair (L, R) becomes
    (hi(M L) xor R xor key, lo(M L)), and the results are placed as
    (hi1^x1^k0, lo1, hi0^x3^k1, lo0).  Between rounds the key is bumped by
    the Weyl increments.
    """
    c = PHILOX[width]
    mask = (1 << width) - 1
    x0, x1, x2, x3 = (int(v) & mask for v in counter)
    k0, k1 = (int(v) & mask for v in key)
    for rnd in range(rounds):
        if rnd:
            k0 = (k0 + c["W0"]) & mask
            k1 = (k1 + c["W1"]) & mask
        p0 = c["M0"] * x0
        p1 = c["M1"] * x2
        x0, x1, x2, x3 = ((p1 >> width) ^ x1 ^ k0) & mask, p1 & mask, ((p0 >> width) ^ x3 ^ k1) & mask, p0 & mask
    return x0, x1, x2, x3


def philox4x32(c0, c1, c2, c3, k0: int, k1: int, rounds: int = 10):
    """Philox-4x32 over numpy uint32 arrays (broadcasting), same rounds as philox4_scalar."""
    c = PHILOX[32]
    lo32 = np.uint64(0xFFFFFFFF)
    sh = np.uint64(32)
    x0, x1, x2, x3 = (np.asarray(v, dtype=np.uint64) for v in (c0, c1, c2, c3))
    x0, x1, x2, x3 = np.broadcast_arrays(x0, x1, x2, x3)
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    M0 = np.uint64(c["M0"])
    M1 = np.uint64(c["M1"])
    for rnd in range(rounds):
        if rnd:
            k0 = (k0 + c["W0"]) & 0xFFFFFFFF
            k1 = (k1 + c["W1"]) & 0xFFFFFFFF
        p0 = M0 * x0          # exact: both factors < 2^32
        p1 = M1 * x2
        x0, x1, x2, x3 = ((p1 >> sh) ^ x1 ^ np.uint64(k0)), (p1 & lo32), ((p0 >> sh) ^ x3 ^ np.uint64(k1)), (p0 & lo32)
    return tuple(v.astype(np.uint32) for v in (x0, x1, x2, x3))


# ---------------------------------------------------------------------------
# Dropout on the branch input
# ---------------------------------------------------------------------------


def dropout_threshold(p: float) -> int:
    """Integer keep threshold T for drop rate p: a 16-bit lane u keeps its element iff u >= T."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout rate must satisfy 0 <= p < 1")
    return int(math.floor(p * 65536.0 + 0.5))


def dropout_scale(p: float) -> float:
    """Inverted-dropout scale q = 1/(1-p) applied to kept elements."""
    return 1.0 / (1.0 - p)


def keep_mask(seed: int, rows, k: int, T: int) -> np.ndarray:
    """Keep decisions D[t, j] (bool) for the given global row indices and features 0..k-1.

    Counter (t, j // 8, 0, 0), key (seed low 32 bits, seed high 32 bits);
    feature j reads 16-bit lane j % 8 of the output (word (j%8)//2, low half
    for even j%8).
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    n_groups = -(-k // 8)
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    t = (rows & 0xFFFFFFFF).astype(np.uint32)[:, None]
    g = np.arange(n_groups, dtype=np.uint32)[None, :]
    w = philox4x32(t, g, 0, 0, seed & 0xFFFFFFFF, seed >> 32)
    lanes = np.empty((rows.size, n_groups, 8), dtype=np.uint32)
    for word in range(4):
        lanes[:, :, 2 * word] = w[word] & np.uint32(0xFFFF)
        lanes[:, :, 2 * word + 1] = w[word] >> np.uint32(16)
    return (lanes.reshape(rows.size, n_groups * 8)[:, :k] >= np.uint32(T))


def pack_mask_bits(D: np.ndarray) -> np.ndarray:
    """Bit j%8 of byte (t, j//8) is the keep decision of feature j (k a multiple of 8)."""
    m, k = D.shape
    weights = (1 << np.arange(8, dtype=np.uint32))
    return (D.reshape(m, k // 8, 8).astype(np.uint32) * weights).sum(axis=2).astype(np.uint8)


# ---------------------------------------------------------------------------
# Single adapter
# ---------------------------------------------------------------------------


def lora_branch(X, A, B, alpha: float, p: float, seed: int, rows):
    """The adapter branch alone: returns (alpha * S B, S, D) with S = X_hat A.

    X holds the global rows `rows` of the layer input; the keep mask of a row
    depends on its global index, not on its position in X.
    """
    D = keep_mask(seed, rows, X.shape[1], dropout_threshold(p))
    q = dropout_scale(p)
    X_hat = X * D * q
    S = X_hat @ A
    return alpha * (S @ B), S, D


def lora_forward(X, W, A, B, alpha: float, p: float, seed: int, rows=None):
    """Y = X W + alpha * (dropout(X) A) B.  Returns (Y, S, D).

    X holds the rows `rows` (global row indices; default 0..len(X)-1) of the
    layer input; S = X_hat A is the rank-r intermediate kept for backward.
    """
    X = np.asarray(X, dtype=np.float64)
    if rows is None:
        rows = np.arange(X.shape[0])
    branch, S, D = lora_branch(X, A, B, alpha, p, seed, rows)
    Y = X @ W + branch
    return Y, S, D


def lora_branch_backward(dY, X, A, B, alpha: float, p: float, seed: int, rows):
    """Gradients through the branch: returns (dX_branch, dA, dB, dS).

    dS = alpha dY B^T, dB = alpha S^T dY, dA = X_hat^T dS and the branch's
    share of dX, (D q) * (dS A^T).  The keep mask is regenerated from the seed.
    """
    D = keep_mask(seed, rows, X.shape[1], dropout_threshold(p))
    q = dropout_scale(p)
    X_hat = X * D * q
    S = X_hat @ A
    dS = alpha * (dY @ B.T)
    dB = alpha * (S.T @ dY)
    dA = X_hat.T @ dS
    dX_branch = (D * q) * (dS @ A.T)
    return dX_branch, dA, dB, dS


def lora_backward(dY, X, W, A, B, alpha: float, p: float, seed: int, rows=None):
    """Gradients of the layer with W frozen.  Returns (dX, dA, dB, dS).

    dX = dY W^T + (D q) * (dS A^T); the base weight gets no gradient.
    """
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    if rows is None:
        rows = np.arange(X.shape[0])
    dX_branch, dA, dB, dS = lora_branch_backward(dY, X, A, B, alpha, p, seed, rows)
    dX = dY @ W.T + dX_branch
    return dX, dA, dB, dS


# ---------------------------------------------------------------------------
# Many adapters: segment table -> per-row / per-tile adapter
# ---------------------------------------------------------------------------


def row_adapters(segments, m: int, n_adapters: int) -> np.ndarray:
    """Adapter id of every row (-1 where no segment covers the row).

    Segments are (row_start, rows, adapter).  Each starts on a 128-row tile
    boundary and spans whole tiles, except that the last tile of the batch may
    be partial; segments do not overlap.
    """
    owner = np.full(m, -1, dtype=np.int64)
    for start, rows, adapter in segments:
        start, rows, adapter = int(start), int(rows), int(adapter)
        if rows == 0:
            continue
        if start < 0 or rows < 0 or start + rows > m:
            raise ValueError("segment outside the batch")
        if start % TILE_ROWS or (rows % TILE_ROWS and start + rows != m):
            raise ValueError("segment not aligned to 128-row tiles")
        if not (0 <= adapter < n_adapters):
            raise ValueError("segment names an unknown adapter")
        if np.any(owner[start:start + rows] != -1):
            raise ValueError("segments overlap")
        owner[start:start + rows] = adapter
    return owner


def tile_adapters(segments, m: int, n_adapters: int) -> np.ndarray:
    """Adapter id of every 128-row tile (the routing table), -1 for none."""
    owner = row_adapters(segments, m, n_adapters)
    return owner[::TILE_ROWS].copy()


def multi_lora_forward(X, W, adapters, segments, seed: int, rows=None):
    """Packed multi-adapter forward.  adapters: list of dicts with A, B, alpha, p.

    Returns (Y, S_list, owner) where S_list[i] holds adapter i's S rows in row
    order (an array of shape (rows_i, r_i)) and owner is the per-row adapter.
    `rows` restricts the computation to those global rows.
    """
    X = np.asarray(X, dtype=np.float64)
    m_total = None
    if rows is None:
        rows = np.arange(X.shape[0])
        m_total = X.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    if m_total is None:
        m_total = int(rows.max()) + 1 if rows.size else 0
        m_total = max(m_total, max((s + r for s, r, _ in segments), default=0))
    owner = row_adapters(segments, m_total, len(adapters))[rows]
    Y = X @ W
    S_list = []
    for i, ad in enumerate(adapters):
        sel = np.nonzero(owner == i)[0]
        if sel.size == 0:
            S_list.append(np.zeros((0, ad["A"].shape[1])))
            continue
        Yi, Si, _ = lora_branch(X[sel], ad["A"], ad["B"], ad["alpha"], ad["p"], seed, rows[sel])
        Y[sel] += Yi
        S_list.append(Si)
    return Y, S_list, owner


def multi_lora_backward(dY, X, W, adapters, segments, seed: int, rows=None):
    """Packed multi-adapter backward.  Returns (dX, dA_list, dB_list, dS_list, owner).

    dA_i and dB_i sum over the rows of adapter i only; an adapter with no rows
    gets zero gradients.  `rows` restricts the computation to those global rows
    (dX for them, and their share of each dA_i / dB_i), as in the forward.
    """
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    m_total = None
    if rows is None:
        rows = np.arange(X.shape[0])
        m_total = X.shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    if m_total is None:
        m_total = int(rows.max()) + 1 if rows.size else 0
        m_total = max(m_total, max((s + r for s, r, _ in segments), default=0))
    owner = row_adapters(segments, m_total, len(adapters))[rows]
    dX = dY @ W.T
    dA_list, dB_list, dS_list = [], [], []
    for i, ad in enumerate(adapters):
        A, B = ad["A"], ad["B"]
        sel = np.nonzero(owner == i)[0]
        if sel.size == 0:
            dA_list.append(np.zeros_like(A, dtype=np.float64))
            dB_list.append(np.zeros_like(B, dtype=np.float64))
            dS_list.append(np.zeros((0, A.shape[1])))
            continue
        dXi, dAi, dBi, dSi = lora_branch_backward(dY[sel], X[sel], A, B, ad["alpha"], ad["p"], seed, rows[sel])
        dX[sel] += dXi
        dA_list.append(dAi)
        dB_list.append(dBi)
        dS_list.append(dSi)
    return dX, dA_list, dB_list, dS_list, owner


# ---------------------------------------------------------------------------
# Greedy token-capacity packing of samples into microbatches
# ---------------------------------------------------------------------------
#
# The multi-adapter scheduler (LoRAFusion notes, papers.chlience.com, section 5
# "Multi-LoRA scheduler"; the article, juhe.plus, section 4.2 step 2) packs the
# samples of a group into microbatches that each hold at most a token capacity,
# solving a two-stage MILP and falling back to greedy packing when the solver
# times out.  The pages do not spell the greedy algorithm out; the reading taken
# here is the textbook greedy for bin packing, first-fit decreasing.  A sample
# occupies its length rounded up to whole 128-row tiles, because the
# multi-adapter kernels route whole tiles.


def padded_rows(length: int) -> int:
    """Rows a sample of `length` tokens occupies: whole 128-row tiles."""
    return -(-int(length) // TILE_ROWS) * TILE_ROWS


def greedy_pack(lengths, capacity: int):
    """First-fit decreasing packing.  Returns (batch_of_sample, row_of_sample, n_batches).

    Samples are taken in order of decreasing padded size (equal sizes: lower
    sample index first).  Each goes into the first microbatch, in the order the
    microbatches were opened, whose remaining rows can hold it; if none can, a
    new microbatch is opened.  Inside a microbatch the samples lie one after
    another in the order they were placed, so row_of_sample is where the sample
    starts.  Raises ValueError for a sample longer than the capacity, a length
    below 1, or a capacity that is not a positive multiple of 128.
    """
    if capacity <= 0 or capacity % TILE_ROWS:
        raise ValueError("capacity must be a positive multiple of 128 rows")
    sizes = []
    for length in lengths:
        if int(length) < 1:
            raise ValueError("sample lengths must be at least 1")
        size = padded_rows(length)
        if size > capacity:
            raise ValueError("a sample does not fit in one microbatch")
        sizes.append(size)
    order = sorted(range(len(sizes)), key=lambda i: (-sizes[i], i))
    used = []                                   # rows filled in each open microbatch
    batch = [0] * len(sizes)
    row = [0] * len(sizes)
    for i in order:
        for b, filled in enumerate(used):
            if filled + sizes[i] <= capacity:
                break
        else:
            b = len(used)
            used.append(0)
        batch[i] = b
        row[i] = used[b]
        used[b] += sizes[i]
    return batch, row, len(used)


# ---------------------------------------------------------------------------
# DoRA: the LoRA layer with a learned magnitude per output feature
# ---------------------------------------------------------------------------
#
# "Scaling DoRA" (paper.rainbus.top), background and method: the adapted
# weight is split into a magnitude vector and a direction,
#     W' = mag * (W + s B A) / ||W + s B A||   (norm over each output feature).
# In this layer's orientation (Y = X W, W is k x n, the adapter adds
# alpha * A B with A k x r, B r x n) the output features are the n columns, so
#     g_j = mag_j / ||W[:, j] + alpha (A B)[:, j]||,
#     Y   = g * (X W + alpha (dropout(X) A) B)      (g scales column j).
# The pages say nothing about dropout here; the branch keeps the LoRA path's
# dropout, so with p = 0 this is exactly X W'.  The pages do not fix the
# backward either; the reading taken is that of DoRA's own training recipe:
# the column norm is treated as a constant (no gradient flows through it), so
#     dZ = dY * g,  (dX, dA, dB) = the LoRA backward of dZ,
#     dmag_j = sum_t dY[t, j] Z[t, j] / ||W[:, j] + alpha (A B)[:, j]||,
# with Z = X W + alpha S B the output before the column scale.


def dora_column_norms(W, A, B, alpha: float) -> np.ndarray:
    """||W[:, j] + alpha (A B)[:, j]||_2 for every output column j (the dense definition)."""
    V = np.asarray(W, dtype=np.float64) + alpha * (np.asarray(A, dtype=np.float64) @ np.asarray(B, dtype=np.float64))
    return np.sqrt((V * V).sum(axis=0))


def dora_forward(X, W, A, B, mag, alpha: float, p: float, seed: int, rows=None):
    """Returns (Y, S, D, g, Z): Y = g * Z with Z the LoRA output and g = mag / column norms."""
    Z, S, D = lora_forward(X, W, A, B, alpha, p, seed, rows)
    g = np.asarray(mag, dtype=np.float64) / dora_column_norms(W, A, B, alpha)
    return Z * g, S, D, g, Z


def dora_backward(dY, X, W, A, B, mag, alpha: float, p: float, seed: int, rows=None):
    """Gradients with the column norm held constant.  Returns (dX, dA, dB, dmag)."""
    norms = dora_column_norms(W, A, B, alpha)
    g = np.asarray(mag, dtype=np.float64) / norms
    Z, _, _ = lora_forward(X, W, A, B, alpha, p, seed, rows)
    dY = np.asarray(dY, dtype=np.float64)
    dX, dA, dB, _ = lora_backward(dY * g, X, W, A, B, alpha, p, seed, rows)
    dmag = (dY * Z).sum(axis=0) / norms
    return dX, dA, dB, dmag
