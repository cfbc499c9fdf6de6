"""Shared helpers for the GPU parity tests (device transfer and error metrics)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import lora_oracle as O  # noqa: E402

TOL = 1e-2  # max|err| / max|ref| per tensor, bf16 storage with fp32 accumulation


def gpu_available() -> bool:
    return torch.cuda.is_available()


def to_dev(bits: np.ndarray) -> "torch.Tensor":
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def host_f64(t) -> np.ndarray:
    return O.bf16_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = np.abs(ref).max()
    if scale == 0.0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def assert_close(name, got, ref, tol=TOL):
    e = rel_err(got, ref)
    assert e <= tol, f"{name}: max|err|/max|ref| = {e:.3e} > {tol:g}"
    return e
