"""GPU parity of the layer's gradients (fno_spectral_conv_backward) against
the float64 oracle's backward, which the CPU suite pins to the forward by
adjoint identities and exact finite differences."""
import numpy as np
import pytest
import torch

from fft_gemm_ifft_gb300 import FnoError, SpectralConv, capi, workloads
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # (n, modes, batch, cin, cout, dtype): every kernel family of the forward
    # runs the adjoint layer (1-D cluster kernel, 128^2 and 256^2 three-kernel
    # paths, 3-D, separate kernels for other shapes); Cin != Cout throughout
    ((256,), (16,), 3, 5, 7, "f32"),
    ((16,), (9,), 2, 3, 4, "f32"),
    ((128, 128), (16, 16), 2, 6, 4, "f32"),
    ((128, 128), (16, 16), 2, 6, 20, "f32"),
    ((128, 128), (16, 16), 2, 3, 5, "f16"),
    ((256, 256), (32, 32), 1, 4, 3, "f16"),
    ((64, 64, 64), (16, 16, 16), 1, 3, 2, "f32"),
    ((16, 32), (3, 7), 2, 3, 5, "f32"),
    ((8, 8, 16), (2, 3, 9), 2, 2, 3, "bf16"),
    ((32, 32), (4, 4), 3, 4, 2, "bf16"),
    ((6, 9), (2, 5), 2, 2, 3, "f32"),
    ((1000,), (40,), 2, 3, 2, "f32"),
]


@pytest.fixture(scope="module", autouse=True)
def _lib(fno, oracle_mod):
    yield


def _case_id(c):
    n, m, b, ci, co, dt = c
    return f"{'x'.join(map(str, n))}_m{'x'.join(map(str, m))}_b{b}_{ci}to{co}_{dt}"


def _inputs(case, seed):
    x = workloads.make_x(case, seed=seed)
    w = workloads.make_w(case, seed=seed + 1)
    w = workloads.to_storage((w.astype(np.float64) * case.cin * case.cout * 2 - 1) / case.cin,
                             case.dtype)
    dyc = workloads.small_case(case.n, case.modes, case.batch, case.cout, case.cout, case.dtype)
    dy = workloads.make_x(dyc, seed=seed + 2)
    return x, w, dy


@pytest.mark.parametrize("spec", CASES, ids=[_case_id(c) for c in CASES])
def test_backward_matches_oracle(spec, oracle_mod):
    n, modes, b, ci, co, dt = spec
    case = workloads.small_case(n, modes, b, ci, co, dt)
    x, w, dy = _inputs(case, 500 + sum(n))
    conv = SpectralConv(n, modes, b, ci, co, dt, capi.FNO_PLAN_BACKWARD)
    dx, dw = conv.backward(to_dev(x, dt), to_dev(w, dt), to_dev(dy, dt))
    torch.cuda.synchronize()
    assert conv.device_error() == 0
    rdx, rdw = oracle_mod.spectral_conv_backward(x.astype(np.float64), workloads.as_complex(w),
                                                 dy.astype(np.float64), modes)
    assert_close(dx.float().cpu().numpy(), rdx, dt, "dx")
    assert_close(dw.float().cpu().numpy(),
                 np.stack([rdw.real, rdw.imag], axis=-1), dt, "dw")
    conv.close()


def test_backward_partial_requests_and_forward_still_works(oracle_mod):
    case = workloads.small_case((128, 128), (16, 16), 2, 4, 4, "f32")
    x, w, dy = _inputs(case, 77)
    conv = SpectralConv(case.n, case.modes, 2, 4, 4, "f32", capi.FNO_PLAN_BACKWARD)
    X, W, DY = to_dev(x), to_dev(w), to_dev(dy)
    dx_only, none = conv.backward(None, W, DY, need_dw=False)
    assert none is None
    none, dw_only = conv.backward(X, None, DY, need_dx=False)
    assert none is None
    dx, dw = conv.backward(X, W, DY)
    torch.cuda.synchronize()
    assert torch.equal(dx_only, dx) and torch.equal(dw_only, dw)
    y = conv(X, W)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle_mod.spectral_conv(x, workloads.as_complex(w),
                                                           case.modes), "f32", "forward")
    conv.close()


def test_backward_errors():
    case = workloads.small_case((32, 32), (4, 4), 1, 2, 3, "f32")
    x, w, dy = _inputs(case, 5)
    X, W, DY = to_dev(x), to_dev(w), to_dev(dy)
    s = torch.cuda.current_stream().cuda_stream
    plain = SpectralConv(case.n, case.modes, 1, 2, 3)
    with pytest.raises(FnoError) as ei:
        plain.backward(X, W, DY)
    assert ei.value.status == capi.FNO_ERR_INVALID_ARG
    conv = SpectralConv(case.n, case.modes, 1, 2, 3, "f32", capi.FNO_PLAN_BACKWARD)
    ws = conv.workspace.data_ptr()
    dx = torch.empty_like(X)
    st = capi.fno_spectral_conv_backward(conv.handle, X.data_ptr(), W.data_ptr(), DY.data_ptr(),
                                         None, None, ws, s)
    assert st == capi.FNO_ERR_INVALID_ARG
    st = capi.fno_spectral_conv_backward(conv.handle, X.data_ptr(), W.data_ptr(), DY.data_ptr(),
                                         DY.data_ptr(), None, ws, s)
    assert st == capi.FNO_ERR_ALIASING
    st = capi.fno_spectral_conv_backward(conv.handle, X.data_ptr(), W.data_ptr(), DY.data_ptr(),
                                         dx.data_ptr() + 4, None, ws, s)
    assert st == capi.FNO_ERR_MISALIGNED
    st = capi.fno_spectral_conv_backward(conv.handle, X.data_ptr(), None, DY.data_ptr(),
                                         dx.data_ptr(), None, ws, s)
    assert st == capi.FNO_ERR_INVALID_ARG
    conv.close()
    plain.close()
