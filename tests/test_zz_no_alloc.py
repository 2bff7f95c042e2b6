"""The allocation-free forward call (fno_spectral_conv_forward_static).

It is meant for callers that may not call cudaMalloc -- code running under
another framework's allocator, or with a device memory budget fixed at
start-up -- and so can create neither a plan nor a workspace.  Its output is
compared with the float64 oracle on the same seeded inputs, over two calls in
a row (the scratch array keeps the first call's contents), and with the
planned forward.  This file is collected last so that a run stopping at its
first failure has already run every other test; it passes alone in a fresh
process and after the rest.
"""
import numpy as np
import pytest
import torch

from fft_gemm_ifft_gb300 import SpectralConv, capi, workloads
from parity_util import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20        # the library's fixed scratch array


@pytest.fixture(scope="module", autouse=True)
def _lib(fno, oracle_mod):
    yield


def static_call(case, batch, x, w, y):
    return capi.fno_spectral_conv_forward_static(
        case.ndim, case.n, case.modes, batch, case.cin, case.cout,
        capi.DTYPE_CODES[case.dtype], x.data_ptr(), w.data_ptr(), y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def static_forward(case, x, w):
    y = torch.empty((x.shape[0], case.cout) + case.n, dtype=x.dtype, device="cuda")
    st = static_call(case, x.shape[0], x, w, y)
    assert st == capi.FNO_OK, capi.fno_status_string(st)
    return y


@pytest.mark.parametrize("name,n,modes,batch,cin,cout,dtype", [
    ("2d_f32", (128, 128), (16, 16), 8, 32, 32, "f32"),
    ("1d_f32", (256,), (16,), 4, 16, 16, "f32"),
    ("3d_small", (16, 16, 16), (4, 4, 4), 2, 3, 5, "f32"),
    ("2d_f16", (64, 64), (8, 8), 2, 4, 6, "f16"),
    ("2d_bf16", (64, 64), (8, 8), 3, 5, 4, "bf16"),
    ("1d_bf16", (512,), (33,), 2, 3, 2, "bf16"),
])
def test_static_matches_oracle_twice(name, n, modes, batch, cin, cout, dtype):
    case = workloads.small_case(n, modes, batch, cin, cout, dtype, index=5)
    w_np = workloads.make_w(case, seed=31)
    w = to_dev(w_np, dtype)
    conv = SpectralConv(case.n, case.modes, batch, cin, cout, dtype)
    # two calls in a row on different inputs: the second must not see the first
    for seed in (41, 42):
        x_np = workloads.make_x(case, seed=seed)
        x = to_dev(x_np, dtype)
        got = static_forward(case, x, w)
        torch.cuda.synchronize()
        got_np = got.float().cpu().numpy()
        assert_close(got_np, run_oracle(case, x_np, w_np), dtype, f"{name} seed {seed}")
        # and it agrees with the planned forward on the same device inputs
        ref = conv(x, w)
        torch.cuda.synchronize()
        assert_close(got_np, ref.float().cpu().numpy().astype(np.float64), dtype,
                     f"{name} seed {seed} vs planned")
    assert conv.device_error() == 0
    conv.close()


def _unfused_workspace(case, batch):
    st, ws, _ = capi.fno_spectral_conv_query(case.ndim, case.n, case.modes, batch, case.cin,
                                             case.cout, capi.DTYPE_CODES[case.dtype],
                                             capi.FNO_PLAN_UNFUSED)
    assert st == capi.FNO_OK
    return ws


def test_static_limit_edges():
    # a shape whose intermediates fill the scratch array exactly is accepted and
    # correct; one batch row more is rejected before anything is enqueued
    case = workloads.small_case((256,), (16,), 1, 16, 16, "f32", index=6)
    lo, hi = 1, 1 << 20
    while lo < hi:                              # largest batch that fits
        mid = (lo + hi + 1) // 2
        if _unfused_workspace(case, mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    under, over = lo, lo + 1
    assert _unfused_workspace(case, under) <= SCRATCH_BYTES < _unfused_workspace(case, over)
    assert _unfused_workspace(case, under) > SCRATCH_BYTES - (64 << 10)   # within 64 KiB

    big = case.with_batch(under)
    x_np = workloads.make_x(big, seed=43)
    w_np = workloads.make_w(big, seed=44)
    x, w = to_dev(x_np), to_dev(w_np)
    y = torch.full((over, case.cout) + case.n, float("nan"), device="cuda")
    xo = torch.zeros((over, case.cin) + case.n, device="cuda")
    st = static_call(case, over, xo, w, y)
    assert st == capi.FNO_ERR_UNSUPPORTED
    st = static_call(case, under, x, w, y[:under])
    assert st == capi.FNO_OK, capi.fno_status_string(st)
    torch.cuda.synchronize()
    got = y[:under].cpu().numpy()
    assert np.isnan(got[-1:]).sum() == 0 and np.isnan(y[under:].cpu().numpy()).all()
    for b in (0, under // 2, under - 1):
        ref = run_oracle(case, x_np[b:b + 1], w_np)
        assert_close(got[b:b + 1], ref, "f32", f"limit batch {under}, sample {b}")


def test_static_rejects_shapes_beyond_its_scratch():
    # the 3-D workload needs far more than the fixed scratch array holds
    case = workloads.CASES["3d_f32"]
    x = torch.empty(case.x_shape, device="cuda")
    w = torch.empty(case.weight_shape + (2,), device="cuda")
    y = torch.empty(case.y_shape, device="cuda")
    st = static_call(case, case.batch, x, w, y)
    assert st == capi.FNO_ERR_UNSUPPORTED
