"""bench.py's roofline denominators and the loud failure without the library (CPU only).

The layer roofline divides by F = 4mkn + 6mr(k + n) FLOPs and by the compulsory bf16 bytes of one fwd+bwd;
DoRA adds its column-norm work.  These tests write the sums out by hand for the Llama-3.1-8B up-proj
shape, so a dropped or doubled term in bench.py's accounting shows up.
"""
import importlib
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

m, k, n, r = 8192, 4096, 14336, 16


@pytest.fixture(scope="module")
def bench():
    b = importlib.import_module("bench")
    # the accounting needs only the shapes: hand the workloads zero-filled bf16 arrays instead of seeded data
    real = b.synth.layer_inputs

    def zeros(seed, m_, k_, n_, r_, **kw):
        z = lambda *shape: np.zeros(shape, dtype=np.uint16)  # noqa: E731
        return {"X": z(m_, k_), "W": z(k_, n_), "A": z(k_, r_), "B": z(r_, n_), "dY": z(m_, n_)}

    b.synth.layer_inputs = zeros
    yield b
    b.synth.layer_inputs = real


def test_layer_flops_and_bytes_8b_up(bench):
    wl = bench.Workload("llama8b_up")
    assert wl.layer_flops() == 4 * m * k * n + 6 * m * r * (k + n) == 1_938_640_863_232
    fwd = m * k + k * n + m * n + k * r + r * n + m * r          # X, W, Y, A, B, S'
    bwd = m * n + k * n + 2 * m * k + m * r + 2 * (k * r + r * n)  # dY, W, X, dX, S', A, B, dA, dB
    assert wl.layer_bytes() == 2 * (fwd + bwd) == 908_263_424


def test_gemm_flops_per_launch_8b_up(bench):
    wl = bench.Workload("llama8b_up")
    assert wl.gemm_flops_per_step("gemm_fwd") == 2 * m * k * n + 2 * m * r * n
    assert wl.gemm_flops_per_step("gemm_bwd") == 2 * m * n * k + 2 * m * r * k
    assert wl.gemm_flops_per_step("ds_db") is None


def test_dora_adds_its_norm_work(bench):
    lora, dora = bench.Workload("llama8b_up"), bench.Workload(bench.DORA)
    assert dora.layer_flops() - lora.layer_flops() == 2 * k * n * r + 2 * k * r * r
    assert dora.layer_bytes() - lora.layer_bytes() == 2 * (k * n + 3 * m * n)


def test_product_path_fails_loudly_without_the_library(tmp_path):
    """With the shared library absent the binding raises; nothing falls back to another implementation."""
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from lora_fine_tuning_gb300 import native\n"
            "native.LIB_PATH = %r\n"
            "native._lib = None\n"
            "try:\n"
            "    native.lib()\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'missing' in str(e))\n") % (ROOT, str(tmp_path / "absent.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.stdout.strip() == "raised True", r.stdout + r.stderr


def test_default_workload_is_the_70b_up_proj_rank_64(bench):
    # the largest single-GPU layer of the set is the headline: m=16384, k=8192, n=28672, r=64
    assert bench.DEFAULT_WORKLOAD == "llama70b_up_r64"
    wl = bench.Workload(bench.DEFAULT_WORKLOAD)
    M, K, N, R = 16384, 8192, 28672, 64
    assert (wl.m, wl.parts[0].k, wl.parts[0].n, wl.parts[0].r_max) == (M, K, N, R)
    assert wl.layer_flops() == 4 * M * K * N + 6 * M * R * (K + N)
    fwd = M * K + K * N + M * N + K * R + R * N + M * R
    bwd = M * N + K * N + 2 * M * K + M * R + 2 * (K * R + R * N)
    assert wl.layer_bytes() == 2 * (fwd + bwd)


def test_rank_pass_bytes_8b_up(bench):
    """Algorithmic bytes behind the rank-r passes' HBM fractions: down_proj reads X, A and writes S'; ds_db
    reads dY, S', B (dY twice in the deterministic mode); da reads X, the keep bits (one bit an element), dSq
    and writes dA."""
    wl = bench.Workload("llama8b_up")
    assert wl.rank_bytes_per_step("down_proj") == 2 * m * k + 2 * k * r + 2 * m * r == 67_502_080
    assert wl.rank_bytes_per_step("down_proj", saved_mask=True) == 67_502_080 + m * k // 8
    assert wl.rank_bytes_per_step("ds_db") == 2 * m * n + 2 * m * r + 2 * r * n == 235_601_920
    assert wl.rank_bytes_per_step("ds_db", deterministic=True) == 235_601_920 + 2 * m * n
    assert wl.rank_bytes_per_step("da") == 2 * m * k + m * k // 8 + 2 * m * r + 2 * k * r == 71_696_384
    assert wl.rank_bytes_per_step("gemm_fwd") is None
