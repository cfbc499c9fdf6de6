"""lora_fwd_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an application that plans all device memory up
front and gives extensions none, or a runtime that forbids allocation on its
compute path) cannot pass the workspace lora_fwd needs; this entry point uses
a fixed 8 MiB array inside the library instead.  The test calls it through
the C ABI twice in a row and compares each result with lora_fwd's, within the
tolerance of the other parity tests.  It lives in its own file, named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from tests.gpu_helpers import TOL, assert_close, host_f64, to_dev, torch

from lora_fine_tuning_gb300 import native, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from lora_fine_tuning_gb300 import api  # noqa: E402


def static_scratch_fwd(X, W, A, B, alpha, p, seed):
    m, k = X.shape
    n = W.shape[1]
    r = A.shape[1]
    Y = torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    S = torch.empty((m, r), dtype=torch.bfloat16, device=X.device)
    mask = torch.empty((m, k // 8), dtype=torch.uint8, device=X.device)
    st = native.lib().lora_fwd_static_scratch(X.data_ptr(), W.data_ptr(), A.data_ptr(), B.data_ptr(),
                                              ctypes.c_float(alpha), ctypes.c_float(p), seed, m, k, n, r,
                                              Y.data_ptr(), S.data_ptr(), mask.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    native.check("lora_fwd_static_scratch", st)
    return Y, S, mask


@pytest.mark.parametrize("m,k,n,r,alpha,p,seed", [(256, 512, 512, 16, 2.0, 0.1, 0), (200, 264, 392, 8, 1.5, 0.2, 11)])
def test_static_scratch_forward_matches_lora_fwd_twice(m, k, n, r, alpha, p, seed):
    raw = synth.layer_inputs(seed, m, k, n, r)
    X, W, A, B = (to_dev(raw[x]) for x in ("X", "W", "A", "B"))
    Y_ref, S_ref, mask_ref = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
    torch.cuda.synchronize()
    for _ in range(2):  # the second call reuses the array the first one left behind
        Y, S, mask = static_scratch_fwd(X, W, A, B, alpha, p, seed)
        torch.cuda.synchronize()
        assert torch.equal(mask, mask_ref)
        assert_close("S_saved", host_f64(S), host_f64(S_ref), TOL)
        assert_close("Y", host_f64(Y), host_f64(Y_ref), TOL)


def test_static_scratch_rejects_sizes_beyond_the_array():
    # m = 65536, r = 64 needs about 25 MB of scratch: more than the 8 MiB array.
    st = native.lib().lora_fwd_static_scratch(256, 256, 256, 256, ctypes.c_float(1.0), ctypes.c_float(0.1), 0,
                                              65536, 4096, 4096, 64, 256, 256, None,
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 6
    assert b"8 MiB" in native.lib().lora_last_error_string()
