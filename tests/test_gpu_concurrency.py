"""Calls from several host threads on several streams at once.

Each entry point prepares its launches in per-thread storage and takes no lock
while it enqueues, and each caller stream has its own side stream for a forked
dA pass.  Two threads run forward + backward steps of different layers on their
own streams and workspaces at the same time; every result must match the same
step run alone (keep masks bit-exact, values within the parity tolerance).
"""
import threading

import pytest

from tests.gpu_helpers import TOL, assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402

# k % 128 != 0 in both layers: each backward forks its dA pass onto its own stream's side stream (with
# k % 128 == 0 the dA pass reads the dX GEMM's keep bits on the caller's stream and nothing is shared)
CASES = [(512, 1032, 768, 16, 2.0, 0.1, 91), (384, 776, 1024, 64, 1.0, 0.2, 92)]


def make(case):
    m, k, n, r, alpha, p, seed = case
    raw = synth.layer_inputs(seed, m, k, n, r)
    return {x: to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY")}


def step(case, t, ws, stream):
    m, k, n, r, alpha, p, seed = case
    Y, S, mask = api.lora_fwd(t["X"], t["W"], t["A"], t["B"], alpha, p, seed, want_mask=True, ws=ws, stream=stream)
    dX, dA, dB = api.lora_bwd(t["dY"], t["X"], t["W"], t["A"], t["B"], S, alpha, p, seed, ws=ws, stream=stream)
    return dict(Y=Y, S=S, mask=mask, dX=dX, dA=dA, dB=dB)


def test_two_threads_on_two_streams_match_single_calls():
    inputs = [make(c) for c in CASES]
    # the reference: each step alone on the current stream
    refs = []
    for case, t in zip(CASES, inputs):
        m, k, n, r = case[:4]
        ws = torch.zeros(api.lora_workspace_size(m, k, n, r), dtype=torch.uint8, device="cuda")
        refs.append(step(case, t, ws, None))
    torch.cuda.synchronize()

    results = [None, None]
    errors = []

    def worker(i):
        try:
            case, t = CASES[i], inputs[i]
            m, k, n, r = case[:4]
            stream = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(stream):
                ws = torch.zeros(api.lora_workspace_size(m, k, n, r), dtype=torch.uint8, device="cuda")
                for _ in range(6):
                    outs.append(step(case, t, ws, stream))
            stream.synchronize()
            code = api.lora_device_status(ws, stream)
            results[i] = (outs, code)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (outs, code), ref in zip(results, refs):
        assert code == 0
        for out in outs:
            assert torch.equal(out["mask"], ref["mask"])
            for name in ("Y", "S", "dX", "dA", "dB"):
                assert_close(name, host_f64(out[name]), host_f64(ref[name]), TOL)
