"""GPU parity at the benchmark sizes, in the launch configuration the benchmark times.

As in bench.py, one workspace serves both calls (its status word is checked
after); the backward regenerates the keep mask from the seed, as bench.py does
by default, and the 8B case also runs the saved-mask mode (bench.py
--saved-mask: the forward writes the keep bits and the backward reads them).  The
oracle computes, in fp64 on the host: the full keep mask, S, dS-derived dA and
dB (all O(m r (k + n))), and Y / dX on a sample of rows (256 random rows plus
two whole 128-row tiles), which it computes one row at a time.  The cases are
every single-adapter layer of the benchmark set, two decoder-layer projections
whose shapes the set lacks, the packed four-adapter batch and the largest
point of the four-adapter rank sweep.
"""
import numpy as np
import pytest

from tests.gpu_helpers import assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import synth
from oracle import lora_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402


def sample_rows(m, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(m, size=min(256, m), replace=False).tolist())
    rows.update(range(0, min(128, m)))                    # first tile
    rows.update(range(max(0, m - 128), m))                # last tile
    return np.array(sorted(rows))


@pytest.mark.parametrize("name,saved", [("llama8b_up", False), ("llama8b_up", True), ("llama70b_o_r16", False),
                                        ("llama70b_o_r64", False), ("llama70b_up_r16", False),
                                        ("llama70b_up_r64", False)])   # the largest layer of the benchmark set
def test_single_adapter_full_size(name, saved):
    cfg = synth.WORKLOADS[name]
    check_single(*(cfg[x] for x in ("m", "k", "n", "r", "alpha", "p", "seed")), saved)


# two projections of the Llama-3.1-8B decoder layer whose shapes no other case covers: down_proj (k > n, the
# backward GEMM's K is only 4096 while its N is 14336) and k_proj (n = 1024: eight column blocks)
@pytest.mark.parametrize("label,k,n,seed", [("down_proj", 14336, 4096, 11), ("k_proj", 4096, 1024, 6)])
def test_decoder_layer_projection_full_size(label, k, n, seed):
    cfg = synth.LAYER_WORKLOAD
    check_single(cfg["m"], k, n, cfg["r"], cfg["alpha"], cfg["p"], seed, False)


def check_single(m, k, n, r, alpha, p, seed, saved):
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    ws = api.workspace(m, k, n, r)
    Y, S, mask = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True, ws=ws)
    dX, dA, dB = api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed, ws=ws, mask_bits=mask if saved else None)
    torch.cuda.synchronize()
    assert api.lora_device_status(ws) == 0

    Xo = O.bf16_to_f64(raw["X"])
    Ao, Bo = O.bf16_to_f64(raw["A"]), O.bf16_to_f64(raw["B"])
    T, q = O.dropout_threshold(p), O.dropout_scale(p)
    D = O.keep_mask(seed, np.arange(m), k, T)
    np.testing.assert_array_equal(mask.cpu().numpy(), O.pack_mask_bits(D))
    Xhat = Xo * D * q
    del D
    Sr = Xhat @ Ao
    assert_close("S_saved", host_f64(S), alpha * Sr)
    dYo = O.bf16_to_f64(raw["dY"])
    dSr = alpha * (dYo @ Bo.T)
    assert_close("dB", host_f64(dB), alpha * (Sr.T @ dYo))
    assert_close("dA", host_f64(dA), Xhat.T @ dSr)
    del Xhat

    rows = sample_rows(m, seed)
    Wo = O.bf16_to_f64(raw["W"])
    Yr, _, _ = O.lora_forward(Xo[rows], Wo, Ao, Bo, alpha, p, seed, rows=rows)
    assert_close("Y[rows]", host_f64(Y[torch.from_numpy(rows).cuda()]), Yr)
    dXr, _, _, _ = O.lora_backward(dYo[rows], Xo[rows], Wo, Ao, Bo, alpha, p, seed, rows=rows)
    assert_close("dX[rows]", host_f64(dX[torch.from_numpy(rows).cuda()]), dXr)


def test_multi_adapter_full_size():
    w = synth.MULTI_WORKLOAD
    check_multi(w["k"], w["n"], w["seed"], w["specs"], w["total_rows"])


def test_multi_adapter_sweep_point_full_size():
    """The four-adapter sweep at its largest point: 32768 packed rows, every adapter at rank 128, k = n = 4096."""
    w = synth.MULTI_SWEEP_WORKLOAD
    check_multi(w["k"], w["n"], w["seed"], synth.multi_sweep_specs(128), 32768)


def check_multi(k, n, seed, specs, total_rows):
    batch = synth.packed_batch(seed, total_rows, len(specs))
    raw = synth.multi_inputs(seed, k, n, specs, batch)
    X, W, dY = (to_dev(raw[x]) for x in ("X", "W", "dY"))
    adapters = [api.Adapter(A=to_dev(A), B=to_dev(B), alpha=s.alpha, p=s.p) for (A, B), s in zip(raw["adapters"], specs)]
    ws = api.workspace(batch.m, k, n, max(s.rank for s in specs), len(specs))
    Y, S, mask = api.multi_lora_fwd(X, W, adapters, batch.segments, seed, want_mask=True, ws=ws)
    dX = api.multi_lora_bwd(dY, X, W, adapters, batch.segments, seed, S, ws=ws)
    torch.cuda.synchronize()
    assert api.lora_device_status(ws) == 0

    m = batch.m
    Xo, dYo = O.bf16_to_f64(raw["X"]), O.bf16_to_f64(raw["dY"])
    owner = O.row_adapters(batch.segments, m, len(specs))
    mbits = mask.cpu().numpy()
    S_host = host_f64(S)
    for i, ((A, B), s) in enumerate(zip(raw["adapters"], specs)):
        sel = np.nonzero(owner == i)[0]
        Ao, Bo = O.bf16_to_f64(A), O.bf16_to_f64(B)
        if sel.size == 0:
            assert not host_f64(adapters[i].dA).any() and not host_f64(adapters[i].dB).any()
            continue
        D = O.keep_mask(seed, sel, k, O.dropout_threshold(s.p))
        np.testing.assert_array_equal(mbits[sel], O.pack_mask_bits(D))
        Xhat = Xo[sel] * D * O.dropout_scale(s.p)
        Sr = Xhat @ Ao
        assert_close(f"S[{i}]", S_host[sel, :s.rank], s.alpha * Sr)
        dSr = s.alpha * (dYo[sel] @ Bo.T)
        assert_close(f"dB[{i}]", host_f64(adapters[i].dB), s.alpha * (Sr.T @ dYo[sel]))
        assert_close(f"dA[{i}]", host_f64(adapters[i].dA), Xhat.T @ dSr)

    rows = sample_rows(m, seed)
    Wo = O.bf16_to_f64(raw["W"])
    ads_o = [dict(A=O.bf16_to_f64(A), B=O.bf16_to_f64(B), alpha=s.alpha, p=s.p)
             for (A, B), s in zip(raw["adapters"], specs)]
    Yr, _, _ = O.multi_lora_forward(Xo[rows], Wo, ads_o, batch.segments, seed, rows=rows)
    assert_close("Y[rows]", host_f64(Y[torch.from_numpy(rows).cuda()]), Yr)
    # dX on the sampled rows: base part plus each row's own adapter branch
    dXr = dYo[rows] @ Wo.T
    for i, ad in enumerate(ads_o):
        pick = np.nonzero(owner[rows] == i)[0]
        if pick.size:
            dXb, _, _, _ = O.lora_branch_backward(dYo[rows[pick]], Xo[rows[pick]], ad["A"], ad["B"], ad["alpha"],
                                                  ad["p"], seed, rows[pick])
            dXr[pick] += dXb
    assert_close("dX[rows]", host_f64(dX[torch.from_numpy(rows).cuda()]), dXr)


def test_dora_full_size():
    """The Llama-3.1-8B up-proj as DoRA, as bench.py's DoRA workload runs it."""
    cfg = synth.WORKLOADS["llama8b_up"]
    m, k, n, r, alpha, p, seed = (cfg[x] for x in ("m", "k", "n", "r", "alpha", "p", "seed"))
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Wo, Ao, Bo = (O.bf16_to_f64(raw[x]) for x in ("W", "A", "B"))
    rng = np.random.default_rng(seed + 100)
    mag_h = (np.sqrt((Wo ** 2).sum(0)) * rng.uniform(0.8, 1.2, n)).astype(np.float32)
    mag = torch.from_numpy(mag_h).cuda()
    ws = api.dora_workspace(m, k, n, r)
    wn2 = api.dora_weight_norm2(W)
    Y, S, g, mask = api.dora_fwd(X, W, A, B, mag, wn2, alpha, p, seed, want_mask=True, ws=ws)
    dX, dA, dB, dmag = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, alpha, p, seed, ws=ws)
    torch.cuda.synchronize()
    assert api.lora_device_status(ws) == 0

    norms = O.dora_column_norms(Wo, Ao, Bo, alpha)
    gr = mag_h.astype(np.float64) / norms
    assert_close("g", g.double().cpu().numpy(), gr, 1e-4)
    Xo, dYo = O.bf16_to_f64(raw["X"]), O.bf16_to_f64(raw["dY"])
    T, q = O.dropout_threshold(p), O.dropout_scale(p)
    D = O.keep_mask(seed, np.arange(m), k, T)
    np.testing.assert_array_equal(mask.cpu().numpy(), O.pack_mask_bits(D))
    Xhat = Xo * D * q
    del D
    Sr = Xhat @ Ao
    assert_close("S_saved", host_f64(S), alpha * Sr)
    dZ = dYo * gr                                   # the norm is held constant in the backward
    dSr = alpha * (dZ @ Bo.T)
    assert_close("dB", host_f64(dB), alpha * (Sr.T @ dZ))
    assert_close("dA", host_f64(dA), Xhat.T @ dSr)
    del Xhat, dZ

    rows = sample_rows(m, seed)
    Yr, _, _, _, _ = O.dora_forward(Xo[rows], Wo, Ao, Bo, mag_h, alpha, p, seed, rows=rows)
    assert_close("Y[rows]", host_f64(Y[torch.from_numpy(rows).cuda()]), Yr)
    dXr, _, _, _ = O.dora_backward(dYo[rows], Xo[rows], Wo, Ao, Bo, mag_h, alpha, p, seed, rows=rows)
    assert_close("dX[rows]", host_f64(dX[torch.from_numpy(rows).cuda()]), dXr)
    # dmag on a sample of columns: sum over all m rows of dY Z / norm, Z from the definition
    cols = np.sort(rng.choice(n, size=64, replace=False))
    Zc = Xo @ Wo[:, cols] + alpha * (Sr @ Bo[:, cols])
    dmag_r = (dYo[:, cols] * Zc).sum(0) / norms[cols]
    assert_close("dmag[cols]", dmag.double().cpu().numpy()[cols], dmag_r)
