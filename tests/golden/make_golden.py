"""Write tests/golden/oracle_tiny.json: a digest of the oracle on the tiny workload.

Calls only the oracle (and the seeded input generator).  The stored values
guard the oracle against accidental edits; they are not taken from any other
implementation.  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from lora_fine_tuning_gb300 import synth  # noqa: E402
from oracle import lora_oracle as O  # noqa: E402


def digest():
    cfg = synth.WORKLOADS["tiny"]
    raw = synth.layer_inputs(cfg["seed"], cfg["m"], cfg["k"], cfg["n"], cfg["r"])
    X, W, A, B, dY = (O.bf16_to_f64(raw[k]) for k in ("X", "W", "A", "B", "dY"))
    a, p, s = cfg["alpha"], cfg["p"], cfg["seed"]
    Y, S, D = O.lora_forward(X, W, A, B, a, p, s)
    dX, dA, dB, dS = O.lora_backward(dY, X, W, A, B, a, p, s)
    out = {"workload": "tiny", "config": cfg, "mask_kept": int(D.sum()),
           "mask_bits_first_row": O.pack_mask_bits(D)[0, :8].tolist()}
    for name, v in (("Y", Y), ("S", S), ("dX", dX), ("dA", dA), ("dB", dB), ("dS", dS)):
        out[name] = {"sum": float(v.sum()), "abs_sum": float(abs(v).sum()), "corner": v[:2, :3].tolist(),
                     "last": v[-1, -3:].tolist()}
    return out


if __name__ == "__main__":
    path = os.path.join(HERE, "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(digest(), f, indent=1)
    print("wrote", path)
