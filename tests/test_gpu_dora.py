"""GPU parity of the DoRA entry points (factored column norm, column-scaled GEMM epilogue, backward with
the norm held constant) against the oracle's dense definition."""
import numpy as np
import pytest

from tests.gpu_helpers import TOL, assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import synth
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402


def run(m, k, n, r, alpha, p, seed):
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Wo, Ao, Bo = (O.bf16_to_f64(raw[x]) for x in ("W", "A", "B"))
    rng = np.random.default_rng(seed)
    mag_np = O.dora_column_norms(Wo, Ao, Bo, alpha) * rng.uniform(0.7, 1.4, n)   # near the initial magnitudes
    mag = torch.tensor(mag_np, dtype=torch.float32, device="cuda")
    mag_np = mag.cpu().numpy().astype(np.float64)          # what the kernels see (fp32)
    wn2 = api.dora_weight_norm2(W)
    Y, S, g, mask = api.dora_fwd(X, W, A, B, mag, wn2, alpha, p, seed, want_mask=True)
    dX, dA, dB, dmag = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, alpha, p, seed)
    torch.cuda.synchronize()
    return raw, mag_np, dict(wn2=wn2, Y=Y, S=S, g=g, mask=mask, dX=dX, dA=dA, dB=dB, dmag=dmag)


def check(raw, mag, out, alpha, p, seed):
    Xo, Wo, Ao, Bo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    np.testing.assert_allclose(out["wn2"].cpu().numpy(), (Wo * Wo).sum(0), rtol=1e-5)
    Yr, Sr, Dr, gr, _ = O.dora_forward(Xo, Wo, Ao, Bo, mag, alpha, p, seed)
    np.testing.assert_allclose(out["g"].cpu().numpy(), gr, rtol=1e-4)
    if Xo.shape[0]:
        np.testing.assert_array_equal(out["mask"].cpu().numpy(), O.pack_mask_bits(Dr))
    assert_close("Y", host_f64(out["Y"]), Yr)
    assert_close("S_saved", host_f64(out["S"]), alpha * Sr)
    dXr, dAr, dBr, dmagr = O.dora_backward(dYo, Xo, Wo, Ao, Bo, mag, alpha, p, seed)
    assert_close("dX", host_f64(out["dX"]), dXr)
    assert_close("dA", host_f64(out["dA"]), dAr)
    assert_close("dB", host_f64(out["dB"]), dBr)
    assert_close("dmag", out["dmag"].cpu().numpy().astype(np.float64), dmagr)


@pytest.mark.parametrize("m,k,n,r,alpha,p,seed", [
    (256, 512, 512, 16, 2.0, 0.1, 70),
    (200, 264, 392, 8, 1.5, 0.2, 71),          # ragged m, k, n; rank 8 (padded 16)
    (384, 512, 768, 64, 2.0, 0.05, 72),
    (130, 1024, 256, 128, 0.5, 0.0, 73),      # rank 128, no dropout
    (256, 2048, 512, 16, 2.0, 0.1, 74),       # forward tiles split by K: the column scale after the partials' sum
])
def test_dora_matches_oracle(m, k, n, r, alpha, p, seed):
    raw, mag, out = run(m, k, n, r, alpha, p, seed)
    check(raw, mag, out, alpha, p, seed)


def test_dora_at_initialisation_is_the_frozen_layer():
    """mag = ||W||_col and B = 0: Y = X W, and dX = dY W^T."""
    m, k, n, r = 256, 256, 384, 16
    raw = synth.layer_inputs(74, m, k, n, r)
    raw["B"] = np.zeros_like(raw["B"])
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    wn2 = api.dora_weight_norm2(W)
    mag = torch.sqrt(wn2)
    Y, S, g, _ = api.dora_fwd(X, W, A, B, mag, wn2, 2.0, 0.1, 5)
    dX, dA, dB, dmag = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, 2.0, 0.1, 5)
    torch.cuda.synchronize()
    Xo, Wo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "dY"))
    np.testing.assert_allclose(g.cpu().numpy(), 1.0, rtol=1e-5)
    assert_close("Y", host_f64(Y), Xo @ Wo)
    assert_close("dX", host_f64(dX), dYo @ Wo.T)


def test_dora_empty_batch():
    k, n, r = 128, 256, 16
    raw = synth.layer_inputs(75, 1, k, n, r)
    W, A, B = (to_dev(raw[x]) for x in ("W", "A", "B"))
    X = torch.empty((0, k), dtype=torch.bfloat16, device="cuda")
    dY = torch.empty((0, n), dtype=torch.bfloat16, device="cuda")
    wn2 = api.dora_weight_norm2(W)
    mag = torch.ones(n, dtype=torch.float32, device="cuda")
    Y, S, g, _ = api.dora_fwd(X, W, A, B, mag, wn2, 1.0, 0.1, 0)
    dX, dA, dB, dmag = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, 1.0, 0.1, 0)
    torch.cuda.synchronize()
    Wo, Ao, Bo = (O.bf16_to_f64(raw[x]) for x in ("W", "A", "B"))
    np.testing.assert_allclose(g.cpu().numpy(), 1.0 / O.dora_column_norms(Wo, Ao, Bo, 1.0), rtol=1e-4)
    assert not dmag.abs().sum().item()
    assert not dA.float().abs().sum().item() and not dB.float().abs().sum().item()


def test_dora_leaves_the_workspace_zero():
    """Calls of different sizes share one workspace: every DoRA call must leave it all zeros."""
    for (m, k, n, r) in [(256, 1024, 256, 128), (130, 256, 512, 64), (200, 264, 392, 8)]:
        raw, mag, out = run(m, k, n, r, 1.0, 0.1, 76)
        ws = api.dora_workspace(m, k, n, r)
        torch.cuda.synchronize()
        assert api.lora_device_status(ws) == 0
        assert not ws.any().item(), f"workspace not zero after the call with {(m, k, n, r)}"
