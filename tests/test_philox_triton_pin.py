"""Pin of the oracle's Philox-4x32-10 against an independent implementation.

Triton ships its own Philox-4x32 (the generator behind its random-number
functions), written from the same published definition: multipliers
0xD2511F53 / 0xCD9E8D57, Weyl key increments 0x9E3779B9 / 0xBB67AE85, key
(seed low 32 bits, seed high 32 bits).  Triton's interpreter runs its kernels
on the CPU with numpy, so the oracle's 32-bit generator, multipliers
included, can be checked word for word against it without a GPU.  The
counters are the ones the keep mask uses: (token row, feature group, 0, 0).
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import lora_oracle as O

pytest.importorskip("triton")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SEEDS = [0, 1, 0x9E3779B9, 2**32 + 5, 123456789012345, 2**64 - 1]

# Runs in a child process: the interpreter is chosen when triton is imported.
CHILD = r"""
import json, sys
import numpy as np
import torch
import triton
import triton.language as tl

@triton.jit
def words(seed, c0_ptr, c1_ptr, out_ptr, N: tl.constexpr):
    offs = tl.arange(0, N)
    c0 = tl.load(c0_ptr + offs)
    c1 = tl.load(c1_ptr + offs)
    z = tl.zeros_like(c0)
    r0, r1, r2, r3 = tl.philox(seed, c0, c1, z, z, 10)
    tl.store(out_ptr + offs * 4 + 0, r0)
    tl.store(out_ptr + offs * 4 + 1, r1)
    tl.store(out_ptr + offs * 4 + 2, r2)
    tl.store(out_ptr + offs * 4 + 3, r3)

req = json.loads(sys.stdin.read())
c0 = torch.tensor(np.array(req["c0"], dtype=np.uint32).view(np.int32))
c1 = torch.tensor(np.array(req["c1"], dtype=np.uint32).view(np.int32))
res = {}
for seed in req["seeds"]:
    out = torch.zeros(4 * len(req["c0"]), dtype=torch.int32)
    # the kernel's seed argument is a 64-bit integer: pass the same bits as a signed value
    s = seed - 2**64 if seed >= 2**63 else seed
    words[(1,)](s, c0, c1, out, N=len(req["c0"]))
    res[str(seed)] = out.numpy().view(np.uint32).reshape(-1, 4).tolist()
print(json.dumps(res))
"""


def test_philox4x32_matches_triton():
    rng = np.random.default_rng(5)
    n = 64
    # token rows and feature groups as the keep mask uses them, plus the extremes of the 32-bit range
    c0 = np.concatenate([[0, 1, 2**31 - 1, 2**32 - 1], rng.integers(0, 2**32, n - 4)]).astype(np.uint64)
    c1 = np.concatenate([[0, 2**32 - 1, 7, 2**28], rng.integers(0, 2**32, n - 4)]).astype(np.uint64)
    req = {"c0": [int(v) for v in c0], "c1": [int(v) for v in c1], "seeds": SEEDS}
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, "-c", CHILD], input=json.dumps(req), capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=600)
    if r.returncode != 0:
        pytest.skip(f"triton interpreter unavailable here: {r.stderr.strip().splitlines()[-1] if r.stderr else ''}")
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for seed in SEEDS:
        k0, k1 = seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF
        ours = np.stack(O.philox4x32(c0, c1, 0, 0, k0, k1), axis=1)
        np.testing.assert_array_equal(ours, np.array(got[str(seed)], dtype=np.uint32), err_msg=f"seed {seed}")


def test_keep_mask_words_come_from_triton_philox_too():
    """The oracle's keep mask for a few rows equals the 16-bit-lane test applied to Triton's words."""
    seed, T, k = 2**33 + 77, O.dropout_threshold(0.3), 64
    rows = np.array([0, 5, 1023, 2**20 + 3])
    D = O.keep_mask(seed, rows, k, T)
    c0 = np.repeat(rows, k // 8).astype(np.uint64)
    c1 = np.tile(np.arange(k // 8), len(rows)).astype(np.uint64)
    req = {"c0": [int(v) for v in c0], "c1": [int(v) for v in c1], "seeds": [seed]}
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, "-c", CHILD], input=json.dumps(req), capture_output=True, text=True,
                       env=env, cwd=ROOT, timeout=600)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable here")
    w = np.array(json.loads(r.stdout.strip().splitlines()[-1])[str(seed)], dtype=np.uint32)   # (rows * groups, 4)
    lanes = np.stack([w & 0xFFFF, w >> 16], axis=2).reshape(len(rows), k // 8, 8)   # low half first
    expect = (lanes >= T).reshape(len(rows), k)
    np.testing.assert_array_equal(D, expect)
