"""Failure detection on the device without a GPU fault: each bounded wait the
fused kernels use is made to run out (it waits for something nothing will
do), must give up within its limit, report FNO_ERR_DEVICE_TIMEOUT through the
plan's error word, and leave the context usable for the next forward call.
Also: one batch sharded over two plans on two streams gives the result of one
plan over the whole batch (the replica / weak-scaling split of the bench)."""
import time

import numpy as np
import pytest
import torch

from fft_gemm_ifft_gb300 import SpectralConv, capi, workloads
from parity_util import assert_close, run_oracle, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fno, oracle_mod):
    yield


@pytest.mark.parametrize("which", [0, 1], ids=["flag", "mbarrier"])
def test_bounded_wait_times_out_and_context_survives(which):
    case = workloads.small_case((64, 64), (8, 8), 2, 3, 4, "f32")
    x, w = workloads.make_x(case, seed=5), workloads.make_w(case, seed=6)
    conv = SpectralConv(case.n, case.modes, 2, 3, 4)
    assert conv.device_error() == capi.FNO_OK
    t0 = time.perf_counter()
    assert capi.fno_plan_check_bounded_wait(conv.handle, which,
                                            torch.cuda.current_stream().cuda_stream) == 0
    st = conv.device_error()
    dt = time.perf_counter() - t0
    assert st == capi.FNO_ERR_DEVICE_TIMEOUT, capi.fno_status_string(st)
    assert 0.4 < dt < 5.0, f"wait gave up after {dt:.3f} s (limit 0.5 s)"
    # reading the error cleared it; the context and the plan still work
    assert conv.device_error() == capi.FNO_OK
    y = conv(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    assert conv.device_error() == capi.FNO_OK
    assert_close(y.cpu().numpy(), run_oracle(case, x, w), "f32", "forward after a time-out")
    conv.close()


def test_bounded_wait_rejects_bad_arguments():
    conv = SpectralConv((32, 32), (4, 4), 1, 2, 2)
    s = torch.cuda.current_stream().cuda_stream
    assert capi.fno_plan_check_bounded_wait(None, 0, s) == capi.FNO_ERR_INVALID_ARG
    assert capi.fno_plan_check_bounded_wait(conv.handle, 2, s) == capi.FNO_ERR_INVALID_ARG
    assert conv.device_error() == capi.FNO_OK
    conv.close()


@pytest.mark.parametrize("name", ["2d_f32", "2d_f16"])
def test_batch_sharded_over_two_streams(name):
    full = workloads.CASES[name]
    half = full.batch // 2
    x, w = workloads.make_x(full), workloads.make_w(full)
    X, W = to_dev(x, full.dtype), to_dev(w, full.dtype)
    one = SpectralConv(full.n, full.modes, full.batch, full.cin, full.cout, full.dtype)
    shards = [SpectralConv(full.n, full.modes, half, full.cin, full.cout, full.dtype)
              for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    y_one = one(X, W)
    torch.cuda.synchronize()
    y = torch.empty_like(y_one)
    for k in range(2):
        # each shard reads and writes its own contiguous slice of the batch
        with torch.cuda.stream(streams[k]):
            shards[k](X[k * half:(k + 1) * half], W, y[k * half:(k + 1) * half],
                      stream=streams[k])
    torch.cuda.synchronize()
    for c in [one] + shards:
        assert c.device_error() == capi.FNO_OK
    a = y.float().cpu().numpy()
    b = y_one.float().cpu().numpy()
    assert_close(a, b.astype(np.float64), full.dtype, "two shards vs one plan")
    for bi in (0, half - 1, half, full.batch - 1):
        ref = run_oracle(full, x[bi:bi + 1], w)
        assert_close(a[bi:bi + 1], ref, full.dtype, f"shard sample b={bi}")
    for c in [one] + shards:
        c.close()
