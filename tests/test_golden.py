"""The oracle still reproduces the digest written by tests/golden/make_golden.py."""
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_stored_digest():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as f:
        stored = json.load(f)
    now = mod.digest()
    assert now["mask_kept"] == stored["mask_kept"]
    assert now["mask_bits_first_row"] == stored["mask_bits_first_row"]
    for name in ("Y", "S", "dX", "dA", "dB", "dS"):
        for key in ("sum", "abs_sum", "corner", "last"):
            np.testing.assert_allclose(np.array(now[name][key]), np.array(stored[name][key]), rtol=1e-9, atol=1e-9)
