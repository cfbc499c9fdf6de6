"""Deterministic mode (lora_set_deterministic(1)): every output bit-identical from call to call.

In the default mode the split sums (S over features, dS over n, dA and dB over tokens) are reduced
with fp32 atomics, so their low bits depend on the order in which CTAs finish.  In mode 1 the partials
go to per-(item, CTA) slots that the finalize passes add in CTA order, and dB comes from a second pass
in which each element is the sum of at most two partials.  The shapes below have fewer 128-row tiles
than CTAs, so every tile's sums are split over three or more CTAs (the case atomics cannot order).
Each case also checks the mode against the fp64 oracle (same bar as the other parity tests) and
against the default mode.
"""
import numpy as np
import pytest

from tests.gpu_helpers import TOL, assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import synth
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402
from tests.test_gpu_parity import MULTI_SPECS, check_multi, multi_case  # noqa: E402


@pytest.fixture
def deterministic():
    api.lora_set_deterministic(True)
    try:
        yield
    finally:
        api.lora_set_deterministic(False)


def single_step(raw, alpha, p, seed):
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Y, S, mask = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
    dX, dA, dB = api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed)
    torch.cuda.synchronize()
    m, k = X.shape
    assert api.lora_device_status(api.workspace(m, k, W.shape[1], A.shape[1])) == 0
    return dict(Y=Y, S=S, mask=mask, dX=dX, dA=dA, dB=dB)


def assert_bit_identical(a, b, names):
    for name in names:
        assert torch.equal(a[name].view(torch.int16), b[name].view(torch.int16)), f"{name} differs between calls"


@pytest.mark.parametrize("m,k,n,r,p", [
    (1000, 4096, 768, 16, 0.1),      # 8 tiles, 32 feature blocks: each tile's S split over many CTAs
    (2048, 2048, 4096, 64, 0.1),     # strip-order rank: dS pass in tile order, dB pass on one-block strips
    (300, 1024, 512, 128, 0.05),     # largest rank, ragged rows
    (512, 4096, 2048, 32, 0.1),      # both GEMMs split tiles by K: partials added in pair order
    (512, 1024, 4096, 16, 0.1),      # eight backward tiles, each split in two by K
])
def test_single_adapter_bit_identical_and_correct(deterministic, m, k, n, r, p):
    alpha, seed = 2.0, 41
    raw = synth.layer_inputs(seed, m, k, n, r)
    runs = [single_step(raw, alpha, p, seed) for _ in range(3)]
    for other in runs[1:]:
        assert_bit_identical(runs[0], other, ("Y", "S", "mask", "dX", "dA", "dB"))
    out = runs[0]
    Xo, Wo, Ao, Bo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Yr, Sr, Dr = O.lora_forward(Xo, Wo, Ao, Bo, alpha, p, seed)
    dXr, dAr, dBr, _ = O.lora_backward(dYo, Xo, Wo, Ao, Bo, alpha, p, seed)
    np.testing.assert_array_equal(out["mask"].cpu().numpy(), O.pack_mask_bits(Dr))
    assert_close("Y", host_f64(out["Y"]), Yr)
    assert_close("S", host_f64(out["S"]), alpha * Sr)
    assert_close("dX", host_f64(out["dX"]), dXr)
    assert_close("dA", host_f64(out["dA"]), dAr)
    assert_close("dB", host_f64(out["dB"]), dBr)


def test_matches_default_mode_within_rounding():
    m, k, n, r, alpha, p, seed = 1000, 4096, 768, 16, 2.0, 0.1, 43
    raw = synth.layer_inputs(seed, m, k, n, r)
    default = single_step(raw, alpha, p, seed)
    api.lora_set_deterministic(True)
    try:
        assert api.lora_get_deterministic()
        det = single_step(raw, alpha, p, seed)
    finally:
        api.lora_set_deterministic(False)
    assert not api.lora_get_deterministic()
    assert torch.equal(default["mask"], det["mask"])
    for name in ("Y", "S", "dX", "dA", "dB"):
        assert_close(name, host_f64(det[name]), host_f64(default[name]), TOL)


def test_multi_adapter_bit_identical_and_correct(deterministic):
    k, n, rows, seed = 1024, 768, 4096, 47
    batch, segments, raw = multi_case(k, n, rows, MULTI_SPECS, seed, extra_gap=True)
    X, W, dY = (to_dev(raw[x]) for x in ("X", "W", "dY"))
    runs = []
    for _ in range(3):
        adapters = [api.Adapter(A=to_dev(A), B=to_dev(B), alpha=s.alpha, p=s.p)
                    for (A, B), s in zip(raw["adapters"], MULTI_SPECS)]
        Y, S, mask = api.multi_lora_fwd(X, W, adapters, segments, seed, want_mask=True)
        dX = api.multi_lora_bwd(dY, X, W, adapters, segments, seed, S)
        torch.cuda.synchronize()
        runs.append((adapters, Y, S, mask, dX))
    a0, Y0, S0, m0, dX0 = runs[0]
    # S_saved and keep-bit rows of tiles without an adapter are not written (torch.empty leaves them arbitrary)
    covered = torch.zeros(X.shape[0], dtype=torch.bool, device=X.device)
    for start, count, _ in segments:
        covered[start:start + count] = True
    for a1, Y1, S1, m1, dX1 in runs[1:]:
        for t0, t1, name in ((Y0, Y1, "Y"), (S0[covered], S1[covered], "S"), (dX0, dX1, "dX")):
            assert torch.equal(t0.view(torch.int16), t1.view(torch.int16)), f"{name} differs between calls"
        assert torch.equal(m0[covered], m1[covered])
        for i, (x, y) in enumerate(zip(a0, a1)):
            assert torch.equal(x.dA.view(torch.int16), y.dA.view(torch.int16)), f"dA[{i}] differs between calls"
            assert torch.equal(x.dB.view(torch.int16), y.dB.view(torch.int16)), f"dB[{i}] differs between calls"
    check_multi(k, n, segments, raw, MULTI_SPECS, seed, a0, Y0, S0, m0, dX0)


def test_workspace_grows_and_rejects_bad_mode():
    small = api.lora_workspace_size(4096, 4096, 4096, 64)
    api.lora_set_deterministic(True)
    try:
        big = api.lora_workspace_size(4096, 4096, 4096, 64)
    finally:
        api.lora_set_deterministic(False)
    assert big > small
    from lora_fine_tuning_gb300 import native
    assert native.lib().lora_set_deterministic(2) == 1   # LORA_EINVAL
    assert not api.lora_get_deterministic()


@pytest.mark.parametrize("m,k,n,r", [(1000, 4096, 768, 16), (640, 1024, 512, 64)])
def test_workspace_is_left_zeroed(deterministic, m, k, n, r):
    """The slot region is cleared by the passes that read it, so the whole workspace (slots included) is
    zero after every call and calls of any shape can share it, as in the default mode."""
    raw = synth.layer_inputs(53, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    ws = torch.zeros(api.lora_workspace_size(m, k, n, r), dtype=torch.uint8, device="cuda")
    Y, S, _ = api.lora_fwd(X, W, A, B, 1.0, 0.2, 53, ws=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    api.lora_bwd(dY, X, W, A, B, S, 1.0, 0.2, 53, ws=ws)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
