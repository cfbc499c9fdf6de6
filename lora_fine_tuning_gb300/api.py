"""Tensor-level API of the LoRA linear layer (torch tensors in, torch tensors out).

The functions carry the C ABI's names and pass raw device pointers and the
current CUDA stream to it; PyTorch only allocates outputs and workspace.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import native

_WS_CACHE: dict = {}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_bf16(name: str, t: torch.Tensor, shape) -> None:
    if t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def lora_workspace_size(m: int, k: int, n: int, r_max: int, n_adapters: int = 1) -> int:
    return int(native.lib().lora_workspace_size(m, k, n, r_max, n_adapters))


def lora_set_deterministic(on: bool) -> None:
    """Bit-reproducible reductions for every later call (see include/lora.h); sizes workspaces anew."""
    native.check("lora_set_deterministic", native.lib().lora_set_deterministic(1 if on else 0))


def lora_get_deterministic() -> bool:
    return bool(native.lib().lora_get_deterministic())


def workspace(m: int, k: int, n: int, r_max: int, n_adapters: int = 1, device=None) -> torch.Tensor:
    """A cached, zero-initialised workspace large enough for these sizes."""
    device = torch.device(device or torch.cuda.current_device())
    size = lora_workspace_size(m, k, n, r_max, n_adapters)
    key = device.index
    ws = _WS_CACHE.get(key)
    if ws is None or ws.numel() < size:
        ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=device)
        _WS_CACHE[key] = ws
    return ws


def lora_fwd(X, W, A, B, alpha: float, p: float, seed: int, *, Y=None, S_saved=None, mask_bits=None,
             want_mask: bool = False, ws=None, stream=None):
    """Y = X W + alpha * (dropout(X) A) B.  Returns (Y, S_saved, mask_bits or None)."""
    m, k = X.shape
    n = W.shape[1]
    r = A.shape[1]
    _check_bf16("X", X, (m, k))
    _check_bf16("W", W, (k, n))
    _check_bf16("A", A, (k, r))
    _check_bf16("B", B, (r, n))
    Y = Y if Y is not None else torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    S_saved = S_saved if S_saved is not None else torch.empty((m, r), dtype=torch.bfloat16, device=X.device)
    if want_mask and mask_bits is None:
        mask_bits = torch.empty((m, k // 8), dtype=torch.uint8, device=X.device)
    ws = ws if ws is not None else workspace(m, k, n, r)
    st = native.lib().lora_fwd(_ptr(X), _ptr(W), _ptr(A), _ptr(B), float(alpha), float(p), int(seed) & (2**64 - 1),
                               m, k, n, r, _ptr(Y), _ptr(S_saved), _ptr(mask_bits), _ptr(ws), ws.numel(),
                               _stream(stream))
    native.check("lora_fwd", st)
    return Y, S_saved, mask_bits


def lora_bwd(dY, X, W, A, B, S_saved, alpha: float, p: float, seed: int, *, dX=None, dA=None, dB=None, ws=None,
             stream=None, mask_bits=None):
    """Gradients of lora_fwd with W frozen.  Returns (dX, dA, dB).  mask_bits: optional, the keep bits
    lora_fwd wrote for the same inputs (read instead of regenerating the mask)."""
    m, k = X.shape
    n = W.shape[1]
    r = A.shape[1]
    for name, t, shp in (("dY", dY, (m, n)), ("X", X, (m, k)), ("W", W, (k, n)), ("A", A, (k, r)),
                         ("B", B, (r, n)), ("S_saved", S_saved, (m, r))):
        _check_bf16(name, t, shp)
    dX = dX if dX is not None else torch.empty((m, k), dtype=torch.bfloat16, device=X.device)
    dA = dA if dA is not None else torch.empty((k, r), dtype=torch.bfloat16, device=X.device)
    dB = dB if dB is not None else torch.empty((r, n), dtype=torch.bfloat16, device=X.device)
    _check_bits(mask_bits, m, k)
    ws = ws if ws is not None else workspace(m, k, n, r)
    st = native.lib().lora_bwd(_ptr(dY), _ptr(X), _ptr(W), _ptr(A), _ptr(B), _ptr(S_saved), _ptr(mask_bits),
                               float(alpha), float(p),
                               int(seed) & (2**64 - 1), m, k, n, r, _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws),
                               ws.numel(), _stream(stream))
    native.check("lora_bwd", st)
    return dX, dA, dB


@dataclass
class Adapter:
    """One adapter of a packed multi-adapter batch (A: k x r, B: r x n, bf16 on the device)."""
    A: torch.Tensor
    B: torch.Tensor
    alpha: float
    p: float
    dA: Optional[torch.Tensor] = None
    dB: Optional[torch.Tensor] = None

    @property
    def rank(self) -> int:
        return self.A.shape[1]


def _adapter_array(adapters: Sequence[Adapter], with_grads: bool):
    arr = (native.LoraAdapter * max(1, len(adapters)))()
    for i, a in enumerate(adapters):
        arr[i].rank = a.rank
        arr[i].alpha = a.alpha
        arr[i].p = a.p
        arr[i].A = _ptr(a.A)
        arr[i].B = _ptr(a.B)
        arr[i].dA = _ptr(a.dA) if with_grads else None
        arr[i].dB = _ptr(a.dB) if with_grads else None
    return arr


def saved_width(adapters: Sequence[Adapter]) -> int:
    return max((a.rank for a in adapters), default=0)


def multi_lora_fwd(X, W, adapters: Sequence[Adapter], segments, seed: int, *, Y=None, S_saved=None, mask_bits=None,
                   want_mask: bool = False, ws=None, stream=None):
    """Packed multi-adapter forward; segments are (row_start, rows, adapter).  Returns (Y, S_saved, mask_bits)."""
    m, k = X.shape
    n = W.shape[1]
    _check_bf16("X", X, (m, k))
    _check_bf16("W", W, (k, n))
    s_ld = saved_width(adapters)
    Y = Y if Y is not None else torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    if S_saved is None and adapters:
        S_saved = torch.empty((m, s_ld), dtype=torch.bfloat16, device=X.device)
    if want_mask and mask_bits is None:
        mask_bits = torch.zeros((m, k // 8), dtype=torch.uint8, device=X.device)
    ws = ws if ws is not None else workspace(m, k, n, max(s_ld, 8), max(1, len(adapters)))
    seg = native.segments_array(segments)
    ad = _adapter_array(adapters, False)
    st = native.lib().multi_lora_fwd(_ptr(X), _ptr(W), ad, len(adapters), seg, len(segments), int(seed) & (2**64 - 1),
                                     m, k, n, _ptr(Y), _ptr(S_saved), _ptr(mask_bits), _ptr(ws), ws.numel(),
                                     _stream(stream))
    native.check("multi_lora_fwd", st)
    return Y, S_saved, mask_bits


def multi_lora_bwd(dY, X, W, adapters: Sequence[Adapter], segments, seed: int, S_saved, *, dX=None, ws=None,
                   stream=None, mask_bits=None):
    """Packed multi-adapter backward.  Fills each adapter's dA / dB (allocated if missing); returns dX.
    mask_bits: optional, the keep bits multi_lora_fwd wrote for the same batch."""
    m, k = X.shape
    n = W.shape[1]
    _check_bf16("dY", dY, (m, n))
    _check_bf16("X", X, (m, k))
    _check_bf16("W", W, (k, n))
    for a in adapters:
        if a.dA is None:
            a.dA = torch.empty_like(a.A)
        if a.dB is None:
            a.dB = torch.empty_like(a.B)
    s_ld = saved_width(adapters)
    dX = dX if dX is not None else torch.empty((m, k), dtype=torch.bfloat16, device=X.device)
    ws = ws if ws is not None else workspace(m, k, n, max(s_ld, 8), max(1, len(adapters)))
    seg = native.segments_array(segments)
    ad = _adapter_array(adapters, True)
    _check_bits(mask_bits, m, k)
    st = native.lib().multi_lora_bwd(_ptr(dY), _ptr(X), _ptr(W), ad, len(adapters), seg, len(segments),
                                     int(seed) & (2**64 - 1), m, k, n, _ptr(S_saved), _ptr(mask_bits), _ptr(dX),
                                     _ptr(ws), ws.numel(), _stream(stream))
    native.check("multi_lora_bwd", st)
    return dX


_DORA_WS: dict = {}


def dora_workspace(m: int, k: int, n: int, r: int, device=None) -> torch.Tensor:
    """A cached, zero-initialised workspace for dora_fwd / dora_bwd with these sizes."""
    device = torch.device(device or torch.cuda.current_device())
    size = int(native.lib().dora_workspace_size(m, k, n, r))
    ws = _DORA_WS.get(device.index)
    if ws is None or ws.numel() < size:
        ws = torch.zeros(max(size, 256), dtype=torch.uint8, device=device)
        _DORA_WS[device.index] = ws
    return ws


def _check_bits(t, m: int, k: int) -> None:
    """The forward's keep bits handed to a backward: m x k/8 bytes, contiguous, on the device."""
    if t is None:
        return
    if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (m, k // 8):
        raise ValueError(f"mask_bits must be a contiguous CUDA uint8 tensor of shape {(m, k // 8)}")


def _check_f32(name: str, t: torch.Tensor, n: int) -> None:
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{name} must be a contiguous CUDA float32 vector of {n}")


def dora_weight_norm2(W, stream=None):
    """Column norms squared of the frozen weight, fp32 (computed once per weight)."""
    k, n = W.shape
    _check_bf16("W", W, (k, n))
    out = torch.empty(n, dtype=torch.float32, device=W.device)
    native.check("dora_weight_norm2", native.lib().dora_weight_norm2(_ptr(W), k, n, _ptr(out), _stream(stream)))
    return out


def dora_fwd(X, W, A, B, mag, w_norm2, alpha: float, p: float, seed: int, *, Y=None, S_saved=None, g_saved=None,
             mask_bits=None, want_mask: bool = False, ws=None, stream=None):
    """DoRA forward: Y = g * (X W + alpha (dropout(X) A) B) with g = mag / column norms of W + alpha A B.
    Returns (Y, S_saved, g_saved, mask_bits or None)."""
    m, k = X.shape
    n = W.shape[1]
    r = A.shape[1]
    for name, t, shp in (("X", X, (m, k)), ("W", W, (k, n)), ("A", A, (k, r)), ("B", B, (r, n))):
        _check_bf16(name, t, shp)
    _check_f32("mag", mag, n)
    _check_f32("w_norm2", w_norm2, n)
    Y = Y if Y is not None else torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    S_saved = S_saved if S_saved is not None else torch.empty((m, r), dtype=torch.bfloat16, device=X.device)
    g_saved = g_saved if g_saved is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    if want_mask and mask_bits is None:
        mask_bits = torch.empty((m, k // 8), dtype=torch.uint8, device=X.device)
    ws = ws if ws is not None else dora_workspace(m, k, n, r)
    st = native.lib().dora_fwd(_ptr(X), _ptr(W), _ptr(A), _ptr(B), _ptr(mag), _ptr(w_norm2), float(alpha), float(p),
                               int(seed) & (2**64 - 1), m, k, n, r, _ptr(Y), _ptr(S_saved), _ptr(g_saved),
                               _ptr(mask_bits), _ptr(ws), ws.numel(), _stream(stream))
    native.check("dora_fwd", st)
    return Y, S_saved, g_saved, mask_bits


def dora_bwd(dY, X, W, A, B, S_saved, Y, mag, g_saved, alpha: float, p: float, seed: int, *, dX=None, dA=None,
             dB=None, dmag=None, dZ=None, ws=None, stream=None, mask_bits=None):
    """DoRA backward with the column norm held constant.  Returns (dX, dA, dB, dmag).
    dZ: m x n bf16 scratch (allocated if not given).  mask_bits: optional, the keep bits dora_fwd wrote."""
    m, k = X.shape
    n = W.shape[1]
    r = A.shape[1]
    for name, t, shp in (("dY", dY, (m, n)), ("X", X, (m, k)), ("W", W, (k, n)), ("A", A, (k, r)),
                         ("B", B, (r, n)), ("S_saved", S_saved, (m, r)), ("Y", Y, (m, n))):
        _check_bf16(name, t, shp)
    _check_f32("mag", mag, n)
    _check_f32("g_saved", g_saved, n)
    dX = dX if dX is not None else torch.empty((m, k), dtype=torch.bfloat16, device=X.device)
    dA = dA if dA is not None else torch.empty((k, r), dtype=torch.bfloat16, device=X.device)
    dB = dB if dB is not None else torch.empty((r, n), dtype=torch.bfloat16, device=X.device)
    dmag = dmag if dmag is not None else torch.empty(n, dtype=torch.float32, device=X.device)
    dZ = dZ if dZ is not None else torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    _check_bf16("dZ", dZ, (m, n))
    _check_bits(mask_bits, m, k)
    ws = ws if ws is not None else dora_workspace(m, k, n, r)
    st = native.lib().dora_bwd(_ptr(dY), _ptr(X), _ptr(W), _ptr(A), _ptr(B), _ptr(S_saved), _ptr(mask_bits),
                               _ptr(Y), _ptr(mag),
                               _ptr(g_saved), float(alpha), float(p), int(seed) & (2**64 - 1), m, k, n, r, _ptr(dX),
                               _ptr(dA), _ptr(dB), _ptr(dmag), _ptr(dZ), _ptr(ws), ws.numel(), _stream(stream))
    native.check("dora_bwd", st)
    return dX, dA, dB, dmag


def lora_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream; returns the raw device status code of the workspace (0 = fine) and clears it."""
    code = ctypes.c_int32(0)
    native.lib().lora_device_status(_ptr(ws), _stream(stream), ctypes.byref(code))
    return code.value


def lora_set_wait_limit_ns(ns: int) -> None:
    native.lib().lora_set_wait_limit_ns(int(ns))


def lora_debug_stuck_wait(ws: torch.Tensor, stream=None) -> None:
    native.check("lora_debug_stuck_wait", native.lib().lora_debug_stuck_wait(_ptr(ws), ws.numel(), _stream(stream)))
