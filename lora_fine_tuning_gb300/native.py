"""ctypes binding of liblora_gb300.so (the C ABI declared in include/lora.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblora_gb300.so")

LORA_OK = 0
LORA_EDEVICE_TIMEOUT = 7
STATUS_NAMES = {0: "LORA_OK", 1: "LORA_EINVAL", 2: "LORA_EALIGN", 3: "LORA_ESHAPE", 4: "LORA_EARCH",
                5: "LORA_ECUDA", 6: "LORA_EWORKSPACE", 7: "LORA_EDEVICE_TIMEOUT", 8: "LORA_ETABLE"}

# Symbols include/lora.h declares, in declaration order.
EXPORTED = ["lora_workspace_size", "lora_set_deterministic", "lora_get_deterministic", "lora_fwd", "lora_bwd", "multi_lora_fwd", "multi_lora_bwd",
            "dora_workspace_size", "dora_weight_norm2", "dora_fwd", "dora_bwd",
            "lora_fwd_static_scratch", "lora_tile_table",
            "lora_keep_threshold", "lora_pack_greedy", "lora_device_status", "lora_set_wait_limit_ns", "lora_debug_stuck_wait",
            "lora_debug_gemm_runs",
            "lora_status_string", "lora_timing_begin", "lora_timing_end", "lora_kernel_name",
            "lora_last_error_string"]


class LoraAdapter(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("alpha", ctypes.c_float), ("p", ctypes.c_float),
                ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("dA", ctypes.c_void_p), ("dB", ctypes.c_void_p)]


class LoraSegment(ctypes.Structure):
    _fields_ = [("row_start", ctypes.c_int64), ("rows", ctypes.c_int64), ("adapter", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class LoraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = ""
        if status == 5:
            try:
                detail = f" ({lib().lora_last_error_string().decode()})"
            except Exception:
                pass
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: {status_string(status)}{detail}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (or python -m lora_fine_tuning_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                      ctypes.c_float, ctypes.c_size_t)
        sig = {
            "lora_workspace_size": (sz, [i64, i64, i64, i32, i32]),
            "lora_set_deterministic": (i32, [i32]),
            "lora_get_deterministic": (i32, []),
            "lora_fwd": (i32, [vp, vp, vp, vp, f32, f32, u64, i64, i64, i64, i32, vp, vp, vp, vp, sz, vp]),
            "lora_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, f32, f32, u64, i64, i64, i64, i32, vp, vp, vp, vp, sz, vp]),
            "multi_lora_fwd": (i32, [vp, vp, ctypes.POINTER(LoraAdapter), i32, ctypes.POINTER(LoraSegment), i32, u64,
                                     i64, i64, i64, vp, vp, vp, vp, sz, vp]),
            "multi_lora_bwd": (i32, [vp, vp, vp, ctypes.POINTER(LoraAdapter), i32, ctypes.POINTER(LoraSegment), i32,
                                     u64, i64, i64, i64, vp, vp, vp, vp, sz, vp]),
            "dora_workspace_size": (sz, [i64, i64, i64, i32]),
            "dora_weight_norm2": (i32, [vp, i64, i64, vp, vp]),
            "dora_fwd": (i32, [vp, vp, vp, vp, vp, vp, f32, f32, u64, i64, i64, i64, i32, vp, vp, vp, vp, vp, sz,
                               vp]),
            "dora_bwd": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, f32, u64, i64, i64, i64, i32, vp, vp,
                               vp, vp, vp, vp, sz, vp]),
            "lora_fwd_static_scratch": (i32, [vp, vp, vp, vp, f32, f32, u64, i64, i64, i64, i32, vp, vp, vp, vp]),
            "lora_tile_table": (i32, [ctypes.POINTER(LoraSegment), i32, i32, i64, ctypes.POINTER(ctypes.c_int32),
                                      i64]),
            "lora_keep_threshold": (i32, [f32, ctypes.POINTER(ctypes.c_uint32)]),
            "lora_pack_greedy": (i32, [ctypes.POINTER(ctypes.c_int64), i32, i64, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)]),
            "lora_device_status": (i32, [vp, vp, ctypes.POINTER(ctypes.c_int32)]),
            "lora_set_wait_limit_ns": (None, [u64]),
            "lora_debug_stuck_wait": (i32, [vp, sz, vp]),
            "lora_debug_gemm_runs": (i32, [i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32), i64,
                                           ctypes.POINTER(ctypes.c_int64)]),
            "lora_status_string": (ctypes.c_char_p, [i32]),
            "lora_last_error_string": (ctypes.c_char_p, []),
            "lora_timing_begin": (i32, []),
            "lora_timing_end": (i32, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int32), i32]),
            "lora_kernel_name": (ctypes.c_char_p, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().lora_status_string(int(status)).decode()
    except Exception:  # library missing: still give a readable name
        return STATUS_NAMES.get(status, str(status))


def check(fn: str, status: int) -> None:
    if status != LORA_OK:
        raise LoraError(fn, status)


def segments_array(segments):
    """(row_start, rows, adapter) triples -> ctypes array of LoraSegment."""
    arr = (LoraSegment * max(1, len(segments)))()
    for i, (s, r, a) in enumerate(segments):
        arr[i].row_start, arr[i].rows, arr[i].adapter, arr[i].reserved = int(s), int(r), int(a), 0
    return arr


def tile_table(segments, n_adapters: int, m: int):
    """Host-only routing table from the library: adapter id per 128-row tile (-1 = none)."""
    n_tiles = -(-m // 128)
    out = (ctypes.c_int32 * max(1, n_tiles))()
    seg = segments_array(segments)
    st = lib().lora_tile_table(seg, len(segments), n_adapters, m, out, n_tiles)
    check("lora_tile_table", st)
    return [out[i] for i in range(n_tiles)]


def keep_threshold(p: float) -> int:
    T = ctypes.c_uint32(0)
    check("lora_keep_threshold", lib().lora_keep_threshold(ctypes.c_float(p), ctypes.byref(T)))
    return T.value


def pack_greedy(lengths, capacity: int):
    """Host-only greedy packing (first-fit decreasing) from the library.

    Returns (batch_of_sample, row_of_sample, n_batches) as Python lists / int."""
    n = len(lengths)
    L = (ctypes.c_int64 * max(1, n))(*[int(x) for x in lengths])
    B = (ctypes.c_int32 * max(1, n))()
    R = (ctypes.c_int64 * max(1, n))()
    nb = ctypes.c_int32(0)
    check("lora_pack_greedy", lib().lora_pack_greedy(L, n, int(capacity), B, R, ctypes.byref(nb)))
    return [B[i] for i in range(n)], [R[i] for i in range(n)], nb.value


def pack_microbatches(lengths, adapters, capacity: int):
    """Packs samples (token lengths and adapter ids) into microbatches of `capacity` rows.

    Returns one dict per microbatch: "segments" [(row_start, rows, adapter)] in row order (the table
    multi_lora_fwd / multi_lora_bwd take), "samples" (sample index per segment), "valid" (tokens per
    segment) and "rows" (rows in use; the rest of the microbatch is free)."""
    batch, row, nb = pack_greedy(lengths, capacity)
    out = [{"segments": [], "samples": [], "valid": [], "rows": 0} for _ in range(nb)]
    for i in sorted(range(len(lengths)), key=lambda i: (batch[i], row[i])):
        b = out[batch[i]]
        rows = -(-int(lengths[i]) // 128) * 128
        b["segments"].append((row[i], rows, int(adapters[i])))
        b["samples"].append(i)
        b["valid"].append(int(lengths[i]))
        b["rows"] = row[i] + rows
    return out


def gemm_runs(M: int, N: int, bn: int, stages: int, max_pairs: int, allow_split: bool = True,
              single_acc: bool = False):
    """The pair GEMM's schedule from the library (host only).

    Returns (pairs, split_tiles, runs), runs a list of (pair, tile, first stage, end stage) in the order
    each pair works through them."""
    pairs, split, n = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int64(0)
    args = (M, N, bn, stages, max_pairs, int(allow_split), int(single_acc), ctypes.byref(pairs), ctypes.byref(split))
    check("lora_debug_gemm_runs", lib().lora_debug_gemm_runs(*args, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_int32 * (4 * max(1, n.value)))()
    check("lora_debug_gemm_runs", lib().lora_debug_gemm_runs(*args, buf, n.value, ctypes.byref(n)))
    runs = [tuple(buf[4 * i:4 * i + 4]) for i in range(n.value)]
    return pairs.value, split.value, runs


KERNEL_KINDS = 13


def timing_begin() -> None:
    check("lora_timing_begin", lib().lora_timing_begin())


def timing_end() -> dict:
    """{kernel name: (total device ms, launches)} for the launches since timing_begin()."""
    ms = (ctypes.c_float * KERNEL_KINDS)()
    n = (ctypes.c_int32 * KERNEL_KINDS)()
    check("lora_timing_end", lib().lora_timing_end(ms, n, KERNEL_KINDS))
    return {lib().lora_kernel_name(i).decode(): (float(ms[i]), int(n[i])) for i in range(KERNEL_KINDS) if n[i]}
