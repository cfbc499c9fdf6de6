"""lora_fwd_static_scratch: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an application that plans all device memory up
front and gives extensions none, or a runtime that forbids allocation on its
compute path) cannot pass the workspace lora_fwd needs; this entry point uses
a fixed 8 MiB array inside the library instead.  The test calls it through
the C ABI twice in a row and compares each result with lora_fwd's, within the
tolerance of the other parity tests; it also calls it with a larger problem
and then a smaller one (the array is shared and must come back clean), checks
that warm calls leave the device's free memory unchanged, and that bad
arguments are refused with lora_fwd's status codes.  It lives in its own file,
named so that pytest collects it last.
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


def _inputs(m, k, n, r, seed):
    raw = synth.layer_inputs(seed, m, k, n, r)
    return [to_dev(raw[x]) for x in ("X", "W", "A", "B")]


def test_static_scratch_larger_then_smaller_problem():
    # a ragged multi-tile problem at rank 64, then a smaller one at rank 8: the second call must not see
    # anything the first left in the shared array
    for (m, k, n, r, alpha, p, seed) in [(1000, 520, 392, 64, 2.0, 0.15, 5), (300, 136, 200, 8, 1.0, 0.1, 6)]:
        X, W, A, B = _inputs(m, k, n, r, seed)
        Y_ref, S_ref, mask_ref = api.lora_fwd(X, W, A, B, alpha, p, seed, want_mask=True)
        Y, S, mask = static_scratch_fwd(X, W, A, B, alpha, p, seed)
        torch.cuda.synchronize()
        assert torch.equal(mask, mask_ref)
        assert_close("S_saved", host_f64(S), host_f64(S_ref), TOL)
        assert_close("Y", host_f64(Y), host_f64(Y_ref), TOL)


def test_static_scratch_warm_calls_allocate_no_device_memory():
    m, k, n, r, alpha, p, seed = 640, 512, 384, 16, 2.0, 0.1, 7
    X, W, A, B = _inputs(m, k, n, r, seed)
    Y = torch.empty((m, n), dtype=torch.bfloat16, device=X.device)
    S = torch.empty((m, r), dtype=torch.bfloat16, device=X.device)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        st = native.lib().lora_fwd_static_scratch(X.data_ptr(), W.data_ptr(), A.data_ptr(), B.data_ptr(),
                                                  ctypes.c_float(alpha), ctypes.c_float(p), seed, m, k, n, r,
                                                  Y.data_ptr(), S.data_ptr(), None, stream)
        native.check("lora_fwd_static_scratch", st)

    call()                      # loads the module and sets up the array on this device
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_scratch_refuses_bad_arguments_like_lora_fwd():
    lib = native.lib()
    stream = torch.cuda.current_stream().cuda_stream
    X, W, A, B = _inputs(256, 128, 128, 16, 8)
    Y = torch.empty((256, 128), dtype=torch.bfloat16, device=X.device)
    S = torch.empty((256, 16), dtype=torch.bfloat16, device=X.device)
    args = lambda **kw: dict(dict(X=X.data_ptr(), W=W.data_ptr(), A=A.data_ptr(), B=B.data_ptr(), alpha=1.0, p=0.1,
                                  m=256, k=128, n=128, r=16, Y=Y.data_ptr(), S=S.data_ptr()), **kw)  # noqa: E731

    def call(a):
        return lib.lora_fwd_static_scratch(a["X"], a["W"], a["A"], a["B"], ctypes.c_float(a["alpha"]),
                                           ctypes.c_float(a["p"]), 0, a["m"], a["k"], a["n"], a["r"], a["Y"],
                                           a["S"], None, stream)

    assert call(args(r=0)) == 1                     # LORA_EINVAL: rank below 8
    assert call(args(p=1.0)) == 1                   # LORA_EINVAL: drop rate outside [0, 1)
    assert call(args(X=X.data_ptr() + 2)) == 2      # LORA_EALIGN
    assert call(args(k=100)) == 3                   # LORA_ESHAPE: k not a multiple of 8
    assert call(args(Y=None)) == 1                  # LORA_EINVAL: no output
    assert call(args()) == 0
    torch.cuda.synchronize()
