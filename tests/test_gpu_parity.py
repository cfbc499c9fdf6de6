"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: keep masks and routing bit-exact; every bf16 output within
max|err| / max|ref| <= 1e-2 of the oracle (fp32 accumulation, bf16 storage).
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


def run_single(m, k, n, r, alpha, p, seed, *, input_seed=None):
    raw = synth.layer_inputs(seed if input_seed is None else input_seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Y, S, mask = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
    dX, dA, dB = api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed)
    ws = api.workspace(m, k, n, r)
    assert api.lora_device_status(ws) == 0
    return raw, dict(Y=Y, S=S, mask=mask, dX=dX, dA=dA, dB=dB)


def check_single_full(raw, out, alpha, p, seed):
    Xo, Wo, Ao, Bo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Yr, Sr, Dr = O.lora_forward(Xo, Wo, Ao, Bo, alpha, p, seed)
    dXr, dAr, dBr, _ = O.lora_backward(dYo, Xo, Wo, Ao, Bo, alpha, p, seed)
    if Xo.shape[0]:
        np.testing.assert_array_equal(out["mask"].cpu().numpy(), O.pack_mask_bits(Dr))
    errs = {}
    errs["Y"] = assert_close("Y", host_f64(out["Y"]), Yr)
    errs["S"] = assert_close("S_saved", host_f64(out["S"]), alpha * Sr)
    errs["dX"] = assert_close("dX", host_f64(out["dX"]), dXr)
    errs["dA"] = assert_close("dA", host_f64(out["dA"]), dAr)
    errs["dB"] = assert_close("dB", host_f64(out["dB"]), dBr)
    return errs


def test_tiny_workload():
    cfg = synth.WORKLOADS["tiny"]
    raw, out = run_single(cfg["m"], cfg["k"], cfg["n"], cfg["r"], cfg["alpha"], cfg["p"], cfg["seed"])
    check_single_full(raw, out, cfg["alpha"], cfg["p"], cfg["seed"])


@pytest.mark.parametrize("m,k,n,r,alpha,p,seed", [
    (200, 264, 392, 8, 1.5, 0.2, 11),        # ragged m, k, n; rank padded 8 -> 16
    (384, 512, 768, 64, 2.0, 0.1, 12),       # three tiles, rank 64
    (130, 128, 256, 128, 0.5, 0.3, 13),      # rank 128: two swizzle atoms; 2-row tail tile
    (1000, 1032, 520, 24, 1.0, 0.05, 14),    # rank 24 padded to 32
    (256, 4096, 320, 16, 2.0, 0.1, 2**33 + 5),  # many k blocks: a tile split over CTAs; seed above 2^32
    (640, 192, 2048, 32, 4.0, 0.5, 15),      # many n blocks in the dS/dB pass
    (1, 64, 64, 16, 1.0, 0.1, 16),           # one row
    (2048, 8192, 64, 16, 2.0, 0.1, 17),      # short dX GEMM (K = 64); the dA pass then reads the bits it wrote
    (2048, 8184, 64, 16, 2.0, 0.1, 18),      # k % 128 != 0: a long dA pass forked beside the short GEMM, the join must wait
])
def test_single_shapes(m, k, n, r, alpha, p, seed):
    raw, out = run_single(m, k, n, r, alpha, p, seed)
    check_single_full(raw, out, alpha, p, seed)


# Shapes whose GEMMs leave CTA pairs idle: fewer tiles than pairs, and full waves plus a partial one, at
# larger k and n than the other cases (the square 4096 sweep's small-m points), with rank-r tails.  Where
# the last wave leaves most of the 76 pairs idle the GEMMs split tiles by K (stream-K runs whose partial
# sums the run holding stage 0 adds): those cases check the split path, the branch tail in a run that does
# not start its tile, and the keep bits it hands to the dA pass.
@pytest.mark.parametrize("m,k,n,r,alpha,p,seed", [
    (1024, 4096, 4096, 16, 2.0, 0.1, 61),     # 64 tiles in each GEMM (whole tiles)
    (768, 2048, 3072, 64, 1.0, 0.2, 62),      # 36 forward tiles, 24 backward tiles: each split in two
    (4096, 4096, 4096, 32, 2.0, 0.1, 63),     # 256 tiles: three full waves + 28; the forward splits 104
    (1280, 4096, 2048, 16, 2.0, 0.1, 64),     # backward 80 tiles (one wave + 4): all split; keep bits to dA
    (2560, 2048, 4096, 32, 1.0, 0.1, 65),     # forward 160 tiles (two waves + 8): the first 84 split;
                                              # backward 80 tiles, all split
    (640, 2048, 8192, 64, 2.0, 0.2, 66),      # rank 64, 128 K stages in the backward
    (384, 1032, 3072, 8, 1.0, 0.1, 67),       # rank 8; k % 128 != 0 (dA regenerates the mask), a ragged column tile
])
def test_partial_wave_shapes(m, k, n, r, alpha, p, seed):
    raw, out = run_single(m, k, n, r, alpha, p, seed)
    check_single_full(raw, out, alpha, p, seed)


def test_partial_wave_multi_adapter():
    """Four adapters on a 1024-row packed batch at k = n = 4096: fewer GEMM tiles than CTA pairs, and tiles
    whose two 128-row halves carry different adapters' tails."""
    k, n, seed = 4096, 4096, 64
    batch, segments, raw = multi_case(k, n, 1024, MULTI_SPECS, seed)
    adapters, Y, S, mask, dX = run_multi(k, n, segments, raw, MULTI_SPECS, seed)
    check_multi(k, n, segments, raw, MULTI_SPECS, seed, adapters, Y, S, mask, dX)


def test_no_dropout_is_merged_weight():
    """p = 0: Y = X (W + alpha A B), masks all ones."""
    m, k, n, r, alpha = 256, 256, 512, 16, 2.0
    raw, out = run_single(m, k, n, r, alpha, 0.0, 3)
    assert (out["mask"].cpu().numpy() == 255).all()
    Xo, Wo, Ao, Bo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "A", "B"))
    assert_close("Y", host_f64(out["Y"]), Xo @ (Wo + alpha * (Ao @ Bo)))


def test_alpha_zero_is_frozen_layer():
    m, k, n, r = 256, 320, 256, 16
    raw, out = run_single(m, k, n, r, 0.0, 0.1, 4)
    Xo, Wo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "dY"))
    assert_close("Y", host_f64(out["Y"]), Xo @ Wo)
    assert_close("dX", host_f64(out["dX"]), dYo @ Wo.T)
    assert not host_f64(out["dA"]).any()
    assert not host_f64(out["dB"]).any()


def test_empty_batch():
    k, n, r = 128, 128, 16
    raw = synth.layer_inputs(5, 1, k, n, r)
    X = torch.empty((0, k), dtype=torch.bfloat16, device="cuda")
    dY = torch.empty((0, n), dtype=torch.bfloat16, device="cuda")
    W, A, B = (to_dev(raw[x]) for x in ("W", "A", "B"))
    Y, S, _ = api.lora_fwd(X, W, A, B, 1.0, 0.1, 0)
    dA = torch.full((k, r), 7.0, dtype=torch.bfloat16, device="cuda")
    dB = torch.full((r, n), 7.0, dtype=torch.bfloat16, device="cuda")
    dX, dA, dB = api.lora_bwd(dY, X, W, A, B, S, 1.0, 0.1, 0, dA=dA, dB=dB)
    torch.cuda.synchronize()
    assert Y.shape == (0, n) and dX.shape == (0, k)
    assert not dA.float().abs().sum().item() and not dB.float().abs().sum().item()


def test_repeat_calls_are_deterministic_in_mask_and_close_in_values():
    """Masks are bit-identical across calls; S', dA, dB are reduced across CTAs with fp32
    atomics, so values (and Y, dX through S', dSq) agree up to rounding order."""
    m, k, n, r = 384, 4096, 512, 16
    raw, out1 = run_single(m, k, n, r, 2.0, 0.1, 21)
    raw, out2 = run_single(m, k, n, r, 2.0, 0.1, 21)
    assert torch.equal(out1["mask"], out2["mask"])
    for name in ("Y", "S", "dX", "dA", "dB"):
        assert_close(name, host_f64(out1[name]), host_f64(out2[name]), TOL)


# ---------------------------------------------------------------------------
# multi-adapter
# ---------------------------------------------------------------------------

def multi_case(k, n, total_rows, specs, seed, extra_gap=False, unused_adapter=False):
    batch = synth.packed_batch(seed, total_rows, len(specs))
    segments = list(batch.segments)
    if extra_gap and len(segments) > 2:
        segments = [s for i, s in enumerate(segments) if i != 1]     # leave a segment's tiles without adapter
    if unused_adapter:
        segments = [(s, r, a if a != len(specs) - 1 else 0) for s, r, a in segments]
    raw = synth.multi_inputs(seed, k, n, specs, batch)
    return batch, segments, raw


def run_multi(k, n, segments, raw, specs, seed):
    X, W, dY = (to_dev(raw[x]) for x in ("X", "W", "dY"))
    adapters = [api.Adapter(A=to_dev(A), B=to_dev(B), alpha=s.alpha, p=s.p) for (A, B), s in zip(raw["adapters"], specs)]
    Y, S, mask = api.multi_lora_fwd(X, W, adapters, segments, seed, want_mask=True)
    dX = api.multi_lora_bwd(dY, X, W, adapters, segments, seed, S)
    torch.cuda.synchronize()
    return adapters, Y, S, mask, dX


def check_multi(k, n, segments, raw, specs, seed, adapters, Y, S, mask, dX, rows=None):
    Xo, Wo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "dY"))
    ads_o = [dict(A=O.bf16_to_f64(A), B=O.bf16_to_f64(B), alpha=s.alpha, p=s.p)
             for (A, B), s in zip(raw["adapters"], specs)]
    m = Xo.shape[0]
    Yr, S_list, owner = O.multi_lora_forward(Xo, Wo, ads_o, segments, seed)
    dXr, dA_list, dB_list, _, _ = O.multi_lora_backward(dYo, Xo, Wo, ads_o, segments, seed)
    assert_close("Y", host_f64(Y), Yr)
    assert_close("dX", host_f64(dX), dXr)
    s_ld = S.shape[1]
    S_ref = np.zeros((m, s_ld))
    for i, ad in enumerate(ads_o):
        sel = np.nonzero(owner == i)[0]
        S_ref[sel, :ad["A"].shape[1]] = ad["alpha"] * S_list[i]
    rows = owner >= 0          # rows without an adapter are not written (their bytes are whatever was there)
    S_host = host_f64(S[torch.from_numpy(np.nonzero(rows)[0]).to(S.device)])
    assert_close("S_saved", S_host, S_ref[rows])
    # keep masks bit-exact on rows that have an adapter
    mbits = mask.cpu().numpy()
    for i, ad in enumerate(ads_o):
        sel = np.nonzero(owner == i)[0]
        if sel.size:
            D = O.keep_mask(seed, sel, k, O.dropout_threshold(ad["p"]))
            np.testing.assert_array_equal(mbits[sel], O.pack_mask_bits(D))
    for i, a in enumerate(adapters):
        if not (owner == i).any():
            assert not host_f64(a.dA).any() and not host_f64(a.dB).any()
            continue
        assert_close(f"dA[{i}]", host_f64(a.dA), dA_list[i])
        assert_close(f"dB[{i}]", host_f64(a.dB), dB_list[i])


MULTI_SPECS = [synth.AdapterSpec(16, 1.0, 0.0), synth.AdapterSpec(16, 2.0, 0.1), synth.AdapterSpec(32, 2.0, 0.1),
               synth.AdapterSpec(64, 4.0, 0.05)]


@pytest.mark.parametrize("k,n,rows,gap,unused", [(512, 512, 2048, False, False), (256, 768, 3072, True, True)])
def test_multi_adapter_packed_batch(k, n, rows, gap, unused):
    seed = 31
    batch, segments, raw = multi_case(k, n, rows, MULTI_SPECS, seed, gap, unused)
    adapters, Y, S, mask, dX = run_multi(k, n, segments, raw, MULTI_SPECS, seed)
    check_multi(k, n, segments, raw, MULTI_SPECS, seed, adapters, Y, S, mask, dX)


def test_maximum_rows_and_adapters():
    """The row limit (262144 rows = 2048 tiles) with every adapter slot in use, ranks 8 to 128 (the limit), and
    ragged k and n: masks bit-exact and every output against the oracle."""
    specs = [synth.AdapterSpec(8 * (i + 1), (1.0, 2.0, 0.5, 4.0)[i % 4], (0.0, 0.1, 0.25, 0.5)[i % 4])
             for i in range(16)]
    k, n, m, seed = 136, 200, 262144, 71
    batch, segments, raw = multi_case(k, n, m, specs, seed)
    assert batch.m == m and len({s[2] for s in segments}) == 16
    adapters, Y, S, mask, dX = run_multi(k, n, segments, raw, specs, seed)
    check_multi(k, n, segments, raw, specs, seed, adapters, Y, S, mask, dX)


@pytest.mark.parametrize("tiles", [(1, 2, 1, 3), (1, 1, 1, 1, 2, 1, 3, 1)])
def test_adapters_with_few_tiles(tiles):
    """Adapters that own one to three tiles and many 128-feature blocks: the dA pass then runs many short
    runs of mixed lengths, so consecutive runs end on different mask groups; each run's partial must
    still be read after its own MMAs only.  Adapters alternate in row order."""
    k, n, seed = 2048, 256, 43
    specs = [synth.AdapterSpec((16, 32, 16, 64)[i % 4], (1.0, 2.0, 0.5, 4.0)[i % 4], (0.1, 0.05, 0.2, 0.1)[i % 4])
             for i in range(len(tiles))]
    segments, row = [], 0
    for a, t in enumerate(tiles):
        segments.append((row, 128 * t, a))
        row += 128 * t
    batch = synth.PackedBatch(m=row, segments=segments, valid=[rows for _, rows, _ in segments])
    raw = synth.multi_inputs(seed, k, n, specs, batch)
    for _ in range(3):     # the race it guards against depends on timing: run it a few times
        adapters, Y, S, mask, dX = run_multi(k, n, segments, raw, specs, seed)
        check_multi(k, n, segments, raw, specs, seed, adapters, Y, S, mask, dX)


def test_routing_table_matches_oracle():
    batch = synth.packed_batch(3, 16384, 4)
    from lora_fine_tuning_gb300 import native
    assert native.tile_table(batch.segments, 4, 16384) == O.tile_adapters(batch.segments, 16384, 4).tolist()


def test_multi_with_one_adapter_equals_single():
    m, k, n, r, alpha, p, seed = 384, 256, 512, 32, 2.0, 0.1, 41
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    Y1, S1, M1 = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
    dX1, dA1, dB1 = api.lora_bwd(dY, X, W, A, B, S1, alpha, p, seed)
    ad = [api.Adapter(A=A, B=B, alpha=alpha, p=p)]
    Y2, S2, M2 = api.multi_lora_fwd(X, W, ad, [(0, m, 0)], seed, want_mask=True)
    dX2 = api.multi_lora_bwd(dY, X, W, ad, [(0, m, 0)], seed, S2)
    torch.cuda.synchronize()
    assert torch.equal(M1, M2)
    # same kernels and routing; values agree up to the order of the fp32 split-K reductions, which
    # can move a bf16 rounding of S (and through it of Y, dX) by one unit: 2^-8 of the value
    assert_close("Y", host_f64(Y2), host_f64(Y1), 4e-3)
    assert_close("S", host_f64(S2), host_f64(S1), 4e-3)
    assert_close("dX", host_f64(dX2), host_f64(dX1), 4e-3)
    # dA, dB pass through dSq (bf16, reduced with atomics): agreement within the parity tolerance
    assert_close("dA", host_f64(ad[0].dA), host_f64(dA1), TOL)
    assert_close("dB", host_f64(ad[0].dB), host_f64(dB1), TOL)


def test_no_segments_is_frozen_layer():
    m, k, n = 256, 256, 512
    raw = synth.layer_inputs(7, m, k, n, 16)
    X, W, dY = (to_dev(raw[x]) for x in ("X", "W", "dY"))
    Y, S, _ = api.multi_lora_fwd(X, W, [], [], 0)
    dX = api.multi_lora_bwd(dY, X, W, [], [], 0, S)
    torch.cuda.synchronize()
    Xo, Wo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "dY"))
    assert_close("Y", host_f64(Y), Xo @ Wo)
    assert_close("dX", host_f64(dX), dYo @ Wo.T)


# ---------------------------------------------------------------------------
# bounded waits
# ---------------------------------------------------------------------------

def test_stuck_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    api.lora_set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        api.lora_debug_stuck_wait(ws)
        code = api.lora_device_status(ws)
    finally:
        api.lora_set_wait_limit_ns(2_000_000_000)
    assert code == (6 << 8) | 1
    assert api.lora_device_status(ws) == 0  # cleared by the read
    raw, out = run_single(128, 128, 128, 16, 1.0, 0.1, 5)
    check_single_full(raw, out, 1.0, 0.1, 5)


@pytest.mark.parametrize("m,k,n,r,saved_bits", [(640, 1032, 392, 24, False), (640, 1024, 392, 24, True),
                                                  (640, 1024, 392, 24, False)])
def test_workspace_is_left_zeroed(m, k, n, r, saved_bits):
    """Each call leaves the workspace all zeros, so calls of any shape can share it: with k % 128 != 0 (the dA
    pass regenerates the mask beside the dX GEMM), with the forward's keep bits, and with the keep bits the
    dX GEMM hands to the dA pass in the workspace (k % 128 == 0, none given)."""
    raw = synth.layer_inputs(51, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    ws = torch.zeros(api.lora_workspace_size(m, k, n, r), dtype=torch.uint8, device="cuda")
    Y, S, bits = api.lora_fwd(X, W, A, B, 1.0, 0.2, 51, ws=ws, want_mask=saved_bits)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0
    api.lora_bwd(dY, X, W, A, B, S, 1.0, 0.2, 51, ws=ws, mask_bits=bits)
    torch.cuda.synchronize()
    assert int(ws.count_nonzero()) == 0


def test_greedy_packed_microbatches():
    """A global batch packed by the library's greedy packer; every microbatch through the multi-adapter path."""
    from lora_fine_tuning_gb300 import native
    specs = MULTI_SPECS[:3]
    k, n, cap, seed = 256, 384, 1024, 61
    lengths, ads = synth.sample_stream(seed, 3 * cap, len(specs), mu=5.0, sigma=0.7, lo=16, hi=1000)
    batches = native.pack_microbatches(lengths, ads, cap)
    assert sum(len(b["samples"]) for b in batches) == len(lengths)
    for b, mb in enumerate(batches):
        pb = synth.PackedBatch(m=cap, segments=mb["segments"], valid=mb["valid"])
        raw = synth.multi_inputs(seed + b, k, n, specs, pb)
        adapters, Y, S, mask, dX = run_multi(k, n, mb["segments"], raw, specs, seed + b)
        check_multi(k, n, mb["segments"], raw, specs, seed + b, adapters, Y, S, mask, dX)
