"""The allocation-free forward call (fno_spectral_conv_forward_static).

It is meant for callers that may not call cudaMalloc -- code running under
another framework's allocator, or with a device memory budget fixed at
start-up -- and so can create neither a plan nor a workspace.  This file is
collected last so that a run stopping at its first failure has already run
every other test; it passes alone in a fresh process and after the rest.
"""
import numpy as np
import pytest
import torch

from fft_gemm_ifft_gb300 import SpectralConv, capi, workloads
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fno):
    yield


def static_forward(case, x, w):
    y = torch.empty(case.y_shape, dtype=x.dtype, device="cuda")
    code = capi.FNO_F32 if case.dtype == "f32" else capi.FNO_F16
    st = capi.fno_spectral_conv_forward_static(
        case.ndim, case.n, case.modes, x.shape[0], case.cin, case.cout, code, x.data_ptr(),
        w.data_ptr(), y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == capi.FNO_OK, capi.fno_status_string(st)
    return y


@pytest.mark.parametrize("name,n,modes,batch,cin,cout,dtype", [
    ("2d_f32", (128, 128), (16, 16), 8, 32, 32, "f32"),
    ("1d_f32", (256,), (16,), 4, 16, 16, "f32"),
    ("3d_small", (16, 16, 16), (4, 4, 4), 2, 3, 5, "f32"),
    ("2d_f16", (64, 64), (8, 8), 2, 4, 6, "f16"),
])
def test_static_matches_planned_forward_twice(name, n, modes, batch, cin, cout, dtype):
    case = workloads.small_case(n, modes, batch, cin, cout, dtype, index=5)
    conv = SpectralConv(case.n, case.modes, batch, cin, cout, dtype)
    w = to_dev(workloads.make_w(case, seed=31))
    # two calls in a row on different inputs: the second must not see the first
    for seed in (41, 42):
        x = to_dev(workloads.make_x(case, seed=seed))
        got = static_forward(case, x, w)
        ref = conv(x, w)
        torch.cuda.synchronize()
        assert_close(got.float().cpu().numpy(), ref.float().cpu().numpy().astype(np.float64),
                     dtype, f"{name} seed {seed}")
    conv.close()


def test_static_rejects_shapes_beyond_its_scratch():
    # the 3-D workload needs far more than the fixed scratch array holds
    case = workloads.CASES["3d_f32"]
    x = torch.empty(case.x_shape, device="cuda")
    w = torch.empty(case.weight_shape + (2,), device="cuda")
    y = torch.empty(case.y_shape, device="cuda")
    st = capi.fno_spectral_conv_forward_static(
        case.ndim, case.n, case.modes, case.batch, case.cin, case.cout, capi.FNO_F32,
        x.data_ptr(), w.data_ptr(), y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == capi.FNO_ERR_UNSUPPORTED
