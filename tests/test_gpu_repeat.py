"""Repeated backward calls: every call right, not only the first.

A race between the warps of a pass (a flush reading an accumulator before its MMAs finish, two issuing
threads on one buffer) shows in some calls only, so a single call per shape can pass while the pass is
wrong.  These cases run many backward calls on one workspace at the square 4096 layer at m = 16384 (the
dS/dB pass in strip order at rank 64, in tile order at rank 16) and check each of them: dB against S'^T dY
formed in fp32 from the call's own inputs, dX against the first call's within rounding, and the workspace
back at zero after every call.  The first call itself is checked against the fp64 oracle in the parity tests.
"""
import pytest

from tests.gpu_helpers import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402


@pytest.mark.parametrize("r", [64, 16])
def test_backward_repeated_calls_each_right(r):
    m, k, n, calls = 16384, 4096, 4096, 60
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(1000 + r)
    X = torch.randn(m, k, device=dev, generator=g).bfloat16()
    W = (torch.randn(k, n, device=dev, generator=g) / k ** 0.5).bfloat16()
    A = ((torch.rand(k, r, device=dev, generator=g) * 2 - 1) / k ** 0.5).bfloat16()
    B = (torch.randn(r, n, device=dev, generator=g) * 0.02).bfloat16()
    dY = torch.randn(m, n, device=dev, generator=g).bfloat16()
    ws = torch.zeros(api.lora_workspace_size(m, k, n, r), dtype=torch.uint8, device=dev)
    Y, S, _ = api.lora_fwd(X, W, A, B, 2.0, 0.1, 5, ws=ws)
    ref_dB = S.float().t() @ dY.float()
    scale = ref_dB.abs().max()
    dX = torch.empty_like(X)
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    first_dX = None
    bad = []
    for i in range(calls):
        api.lora_bwd(dY, X, W, A, B, S, 2.0, 0.1, 5, dX=dX, dA=dA, dB=dB, ws=ws)
        torch.cuda.synchronize()
        err_dB = ((dB.float() - ref_dB).abs().max() / scale).item()
        if first_dX is None:
            first_dX = dX.float().clone()
        err_dX = ((dX.float() - first_dX).abs().max() / first_dX.abs().max()).item()
        nonzero = int(ws.count_nonzero())
        if err_dB > 1e-2 or err_dX > 1e-2 or nonzero:
            bad.append((i, err_dB, err_dX, nonzero))
            ws.zero_()
    assert api.lora_device_status(ws) == 0
    assert not bad, f"calls with wrong results or a dirty workspace: {bad[:5]}"
