"""GPU: the backward reading the forward's keep bits instead of regenerating them.

The bits are the same decisions the Philox generator makes, so the gradients
must match the backward that regenerates the mask (up to the order of the
fp32 split-K reductions, which is free) and the fp64 oracle.  Shapes cover
k % 128 == 0 (the dX GEMM and the dA pass both read the bits), k % 32 == 0
only (the GEMM reads them, dA regenerates) and k % 8 == 0 only (neither).
"""
import pytest

from tests.gpu_helpers import assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import synth
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402

# two backwards on the same inputs: only the reduction order of dS, dA, dB may differ
SAME = 4e-3


@pytest.mark.parametrize("m,k,n,r,alpha,p,seed", [
    (384, 512, 768, 16, 2.0, 0.1, 81),       # k % 128 == 0: GEMM and dA read the bits
    (200, 288, 392, 32, 1.5, 0.2, 82),       # k % 32 == 0 only; ragged m
    (130, 264, 256, 8, 1.0, 0.3, 83),        # k % 8 only: both regenerate
    (256, 4096, 320, 64, 2.0, 0.5, 84),      # many k blocks
    (384, 1024, 2048, 16, 2.0, 0.1, 85),     # backward tiles split by K: the run holding the tail reads the bits
])
def test_single_backward_with_saved_bits(m, k, n, r, alpha, p, seed):
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    _, S, bits = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
    dX0, dA0, dB0 = api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed)
    dX1, dA1, dB1 = api.lora_bwd(dY, X, W, A, B, S, alpha, p, seed, mask_bits=bits)
    torch.cuda.synchronize()
    for name, a, b in (("dX", dX1, dX0), ("dA", dA1, dA0), ("dB", dB1, dB0)):
        assert_close(name, host_f64(a), host_f64(b), SAME)
    Xo, Wo, Ao, Bo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    dXr, dAr, dBr, _ = O.lora_backward(dYo, Xo, Wo, Ao, Bo, alpha, p, seed)
    assert_close("dX", host_f64(dX1), dXr)
    assert_close("dA", host_f64(dA1), dAr)
    assert_close("dB", host_f64(dB1), dBr)


def test_multi_backward_with_saved_bits():
    """Rows without an adapter get no bits from the forward; the backward must not read them."""
    specs = [synth.AdapterSpec(16, 1.0, 0.0), synth.AdapterSpec(16, 2.0, 0.1), synth.AdapterSpec(32, 2.0, 0.2)]
    k, n, seed = 512, 384, 85
    segments = [(0, 256, 1), (384, 512, 0), (896, 256, 2), (1152, 128, 1)]   # rows 256..383 have no adapter
    pb = synth.PackedBatch(m=1408, segments=segments, valid=[s[1] for s in segments])
    raw = synth.multi_inputs(seed, k, n, specs, pb)
    X, W, dY = (to_dev(raw[x]) for x in ("X", "W", "dY"))
    m = X.shape[0]

    def adapters():
        return [api.Adapter(A=to_dev(A), B=to_dev(B), alpha=s.alpha, p=s.p) for (A, B), s in zip(raw["adapters"], specs)]

    ads0, ads1 = adapters(), adapters()
    bits = torch.full((m, k // 8), 0xA5, dtype=torch.uint8, device="cuda")   # stale bytes where no adapter writes
    _, S, _ = api.multi_lora_fwd(X, W, ads1, segments, seed, mask_bits=bits)
    dX0 = api.multi_lora_bwd(dY, X, W, ads0, segments, seed, S)
    dX1 = api.multi_lora_bwd(dY, X, W, ads1, segments, seed, S, mask_bits=bits)
    torch.cuda.synchronize()
    assert_close("dX", host_f64(dX1), host_f64(dX0), SAME)
    for i in range(len(specs)):
        assert_close(f"dA{i}", host_f64(ads1[i].dA), host_f64(ads0[i].dA), SAME)
        assert_close(f"dB{i}", host_f64(ads1[i].dB), host_f64(ads0[i].dB), SAME)
    Xo, Wo, dYo = (O.bf16_to_f64(raw[x]) for x in ("X", "W", "dY"))
    ads_o = [dict(A=O.bf16_to_f64(A), B=O.bf16_to_f64(B), alpha=s.alpha, p=s.p)
             for (A, B), s in zip(raw["adapters"], specs)]
    dXr, dA_list, dB_list, _, _ = O.multi_lora_backward(dYo, Xo, Wo, ads_o, segments, seed)
    assert_close("dX", host_f64(dX1), dXr)
    for i in range(len(specs)):
        assert_close(f"dA{i}", host_f64(ads1[i].dA), dA_list[i])
        assert_close(f"dB{i}", host_f64(ads1[i].dB), dB_list[i])


def test_dora_backward_with_saved_bits():
    m, k, n, r, alpha, p, seed = 256, 384, 512, 16, 2.0, 0.1, 86
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    wn2 = api.dora_weight_norm2(W)
    mag = torch.sqrt(wn2) * 1.1
    Y, S, g, bits = api.dora_fwd(X, W, A, B, mag, wn2, alpha, p, seed, want_mask=True)
    out0 = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, alpha, p, seed)
    out1 = api.dora_bwd(dY, X, W, A, B, S, Y, mag, g, alpha, p, seed, mask_bits=bits)
    torch.cuda.synchronize()
    for name, a, b in zip(("dX", "dA", "dB"), out1[:3], out0[:3]):
        assert_close(name, host_f64(a), host_f64(b), SAME)
    # dmag: fp32 column sums whose atomic order varies between calls
    assert_close("dmag", out1[3].double().cpu().numpy(), out0[3].double().cpu().numpy(), 1e-5)


def test_bits_of_the_wrong_shape_are_rejected():
    m, k, n, r = 128, 256, 256, 16
    raw = synth.layer_inputs(87, m, k, n, r)
    X, W, A, B, dY = (to_dev(raw[x]) for x in ("X", "W", "A", "B", "dY"))
    _, S, _ = api.lora_fwd(X, W, A, B, 1.0, 0.1, 1)
    with pytest.raises(ValueError):
        api.lora_bwd(dY, X, W, A, B, S, 1.0, 0.1, 1, mask_bits=torch.zeros((m, k), dtype=torch.uint8, device="cuda"))
