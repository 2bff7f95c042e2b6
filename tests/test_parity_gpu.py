"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs (element by element), plus edge cases and the error
paths of the forward call."""
import numpy as np
import pytest
import torch

import oracle
from fft_gemm_ifft_gb300 import FNO_PLAN_UNFUSED, FnoError, SpectralConv, capi, workloads
from parity_util import assert_close, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

SMALL = [
    # (n, modes, batch, cin, cout, dtype)
    ((256,), (16,), 4, 16, 16, "f32"),
    ((256,), (16,), 3, 5, 11, "f16"),
    ((256,), (16,), 2, 5, 7, "bf16"),
    ((1024,), (64,), 3, 12, 20, "f32"),
    ((512,), (257,), 2, 4, 3, "f16"),
    ((256,), (129,), 1, 64, 2, "f32"),
    ((16,), (9,), 2, 3, 5, "f32"),
    ((8,), (5,), 1, 1, 1, "f32"),
    ((128, 128), (16, 16), 3, 32, 32, "f32"),
    ((128, 128), (16, 16), 1, 5, 7, "f32"),
    ((128, 128), (1, 1), 2, 4, 4, "f32"),
    ((128, 128), (16, 16), 2, 6, 5, "f16"),
    ((128, 128), (16, 16), 2, 6, 5, "bf16"),
    ((32, 32), (4, 4), 2, 3, 3, "bf16"),
    ((128, 128), (16, 16), 2, 64, 64, "f32"),
    ((128, 128), (16, 16), 1, 64, 37, "f32"),
    ((128, 128), (16, 16), 9, 3, 2, "f32"),
    ((128, 128), (16, 16), 10, 3, 40, "f32"),    # > 2 output images per SM: one-pass kernel C
    # fp32 tensor-core mixing: 64 outputs (one mode on M; 16 / 32 batch rows on
    # N) and 32 outputs (two modes on M; 8 / 16 rows each), 32 or 64 inputs
    ((128, 128), (16, 16), 16, 64, 64, "f32"),
    ((128, 128), (16, 16), 20, 32, 64, "f32"),
    ((128, 128), (16, 16), 5, 64, 32, "f32"),
    ((128, 128), (16, 16), 12, 32, 32, "f32"),
    ((16, 32), (3, 7), 3, 5, 3, "f32"),
    ((32, 16), (16, 9), 2, 2, 3, "f32"),
    ((64, 64), (16, 16), 2, 8, 8, "f32"),
    ((256, 256), (32, 32), 1, 8, 8, "f16"),
    ((256, 256), (32, 32), 2, 3, 5, "f16"),
    ((256, 256), (32, 32), 1, 4, 4, "bf16"),
    ((256, 256), (32, 32), 3, 4, 2, "f32"),
    ((64, 64), (8, 8), 2, 4, 6, "f16"),
    ((64, 64, 64), (16, 16, 16), 1, 4, 4, "f32"),
    # extents that are not powers of two, and large extents (separate kernels)
    ((12,), (7,), 2, 3, 4, "f32"),
    ((2048,), (64,), 2, 4, 4, "f32"),
    ((3000,), (100,), 1, 2, 3, "f32"),
    ((4096,), (17,), 1, 2, 2, "bf16"),
    ((6, 10), (2, 4), 2, 3, 2, "f32"),
    ((24, 40), (5, 9), 2, 4, 3, "f16"),
    ((6, 10, 14), (2, 3, 4), 1, 2, 3, "f32"),
    ((64, 64, 64), (16, 16, 16), 2, 5, 3, "f32"),
    ((64, 64, 64), (16, 16, 16), 3, 3, 5, "f16"),
    ((64, 64, 64), (16, 16, 16), 1, 3, 2, "bf16"),
    # weights by TMA with a partial last box of input channels (3-D: 16 per box;
    # 128^2: 16 per box, Cin x Cout >= 2048)
    ((64, 64, 64), (16, 16, 16), 3, 20, 24, "f32"),
    ((128, 128), (16, 16), 3, 40, 60, "f32"),
    ((8, 8, 8), (2, 3, 4), 2, 3, 2, "f32"),
    ((4, 8, 16), (2, 4, 9), 2, 2, 2, "f32"),
    ((32, 32, 32), (8, 8, 8), 2, 3, 4, "f16"),
]


def case_id(c):
    n, m, b, ci, co, dt = c
    return f"{'x'.join(map(str, n))}_m{'x'.join(map(str, m))}_b{b}_{ci}to{co}_{dt}"


@pytest.fixture(scope="module", autouse=True)
def _lib(fno, oracle_mod):
    yield


@pytest.mark.parametrize("flags", [0, FNO_PLAN_UNFUSED, capi.FNO_PLAN_PERSISTENT,
                                   capi.FNO_PLAN_SIMT_MIX, capi.FNO_PLAN_SIMT_TRANSFORM,
                                   capi.FNO_PLAN_TENSOR_EXTRA],
                         ids=["default", "unfused", "persistent", "simt_mix",
                              "simt_transform", "tensor_extra"])
@pytest.mark.parametrize("spec", SMALL, ids=[case_id(c) for c in SMALL])
def test_small_cases_match_oracle(spec, flags):
    n, modes, b, ci, co, dt = spec
    case = workloads.small_case(n, modes, b, ci, co, dt, index=7)
    x = workloads.make_x(case, seed=100 + sum(n))
    w = workloads.make_w(case, seed=200 + sum(modes))
    # a random weight with negative parts too, so sign errors cannot cancel
    w = workloads.to_storage((w.astype(np.float64) * case.cin * case.cout * 2 - 1) / case.cin,
                             case.dtype)
    got, _ = run_gpu(case, x, w, flags)
    ref = run_oracle(case, x, w)
    assert_close(got, ref, dt, case_id(spec))


@pytest.mark.parametrize("n", [(8,), (16,), (8, 8), (16, 32), (4, 4, 8), (8, 4, 16)])
def test_all_modes_identity_reproduces_input(n):
    modes = tuple(v // 2 for v in n[:-1]) + (n[-1] // 2 + 1,)
    cin = 3
    case = workloads.small_case(n, modes, 2, cin, cin, "f32")
    x = workloads.make_x(case, seed=5)
    w = np.zeros(case.weight_shape + (2,), dtype=np.float32)
    for i in range(cin):
        w[:, i, i, ..., 0] = 1.0
    got, _ = run_gpu(case, x, w)
    assert np.max(np.abs(got - x)) < 1e-5 * np.max(np.abs(x))


def test_single_hot_mode_each_block_3d():
    # one block's weight at a time: every other block must contribute nothing
    case = workloads.small_case((16, 16, 16), (4, 4, 4), 1, 2, 2, "f32")
    x = workloads.make_x(case, seed=11)
    for blk in range(4):
        w = np.zeros(case.weight_shape + (2,), dtype=np.float32)
        w[blk, :, :, 1, 2, 3, 0] = 0.5
        w[blk, :, :, 1, 2, 3, 1] = -0.25
        got, _ = run_gpu(case, x, w)
        ref = run_oracle(case, x, w)
        assert_close(got, ref, "f32", f"block {blk}")


@pytest.mark.parametrize("name", ["1d_f32", "2d_f32"])
def test_full_size_workload_full_compare(name):
    case = workloads.CASES[name]
    x, w = workloads.make_x(case), workloads.make_w(case)
    got, _ = run_gpu(case, x, w)
    ref = run_oracle(case, x, w)
    assert_close(got, ref, case.dtype, name)


@pytest.mark.parametrize("name,samples", [("2d_f16", (0, 31)), ("2d_bf16", (0, 31)),
                                          ("3d_f32", (0, 3))])
def test_full_size_workload_sampled(name, samples):
    # the GPU runs the whole batch; the oracle checks whole samples of it
    # (each sample's output depends only on that sample's input)
    case = workloads.CASES[name]
    x, w = workloads.make_x(case), workloads.make_w(case)
    got, _ = run_gpu(case, x, w)
    for b in samples:
        ref = run_oracle(case, x[b:b + 1], w)
        assert_close(got[b:b + 1], ref, case.dtype, f"{name}[b={b}]")


def test_fused_and_unfused_agree_and_are_deterministic():
    case = workloads.CASES["2d_f32"]
    x, w = workloads.make_x(case), workloads.make_w(case)
    a, _ = run_gpu(case, x, w)
    b, _ = run_gpu(case, x, w)
    c, _ = run_gpu(case, x, w, FNO_PLAN_UNFUSED)
    d, _ = run_gpu(case, x, w, capi.FNO_PLAN_SIMT_TRANSFORM)
    e, _ = run_gpu(case, x, w, capi.FNO_PLAN_SIMT_TRANSFORM)
    f, _ = run_gpu(case, x, w, capi.FNO_PLAN_PERSISTENT)
    assert_close(f, c.astype(np.float64), "f32", "persistent vs unfused")
    assert np.array_equal(a, b), "two runs of the same plan differ"
    assert np.array_equal(d, e), "two runs of the register-FFT plan differ"
    assert_close(a, c.astype(np.float64), "f32", "fused vs unfused")
    assert_close(d, c.astype(np.float64), "f32", "register-FFT kernels vs unfused")


@pytest.mark.parametrize("name,kernels", [("1d_f32", 1), ("2d_f32", 3), ("2d_f16", 3),
                                          ("2d_bf16", 3), ("3d_f32", 3)])
def test_every_workload_runs_fused(name, kernels):
    case = workloads.CASES[name]
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype)
    assert conv.kernel_count == kernels
    conv.close()
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype,
                        FNO_PLAN_UNFUSED)
    assert conv.kernel_count == 2 * len(case.n) + 1
    conv.close()


@pytest.mark.parametrize("name", ["2d_f16", "2d_bf16"])
def test_tensor_core_and_simt_kernels_agree(name):
    # both within the half-storage bar of the oracle (sampled) and of each other
    case = workloads.CASES[name]
    x, w = workloads.make_x(case), workloads.make_w(case)
    a, _ = run_gpu(case, x, w)
    b, _ = run_gpu(case, x, w, capi.FNO_PLAN_SIMT_MIX)
    c, _ = run_gpu(case, x, w)
    d, _ = run_gpu(case, x, w, capi.FNO_PLAN_SIMT_MIX | capi.FNO_PLAN_SIMT_TRANSFORM)
    assert np.array_equal(a, c), "two runs of the tensor-core kernels differ"
    assert_close(a, b.astype(np.float64), case.dtype, "tensor-core vs SIMT mixing")
    assert_close(a, d.astype(np.float64), case.dtype, "tensor-core vs SIMT kernels")
    for s in (0, case.batch - 1):
        ref = run_oracle(case, x[s:s + 1], w)
        assert_close(a[s:s + 1], ref, case.dtype, f"{name}[b={s}] tensor-core mixing")


def test_fused_3d_and_unfused_agree():
    case = workloads.CASES["3d_f32"]
    x, w = workloads.make_x(case), workloads.make_w(case)
    a, ka = run_gpu(case, x, w)
    b, _ = run_gpu(case, x, w)
    c, kc = run_gpu(case, x, w, FNO_PLAN_UNFUSED)
    assert ka == 3 and kc == 7
    assert np.array_equal(a, b), "two runs of the same plan differ"
    assert_close(a, c.astype(np.float64), "f32", "3-D fused vs unfused")


@pytest.mark.parametrize("name,chunks_a,chunks_c", [("2d_f32", 1, 1), ("3d_f32", 8, 8)])
def test_trace_three_kernel_variant(name, chunks_a, chunks_c):
    # one record per CTA of each kernel; kernel B's CTAs start before A's last
    # one ends at the earliest (programmatic dependent launch), never wait past it
    case = workloads.CASES[name]
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype,
                        capi.FNO_PLAN_TRACE)
    x, w = workloads.make_x(case), workloads.make_w(case)
    y = conv(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    st, recs = capi.fno_plan_get_trace(conv.handle)
    assert st == capi.FNO_OK
    phases = [r[0] for r in recs]
    assert phases.count(0) == case.batch * case.cin * chunks_a
    assert phases.count(2) == case.batch * case.cout * chunks_c
    assert phases.count(1) > 0 and len(recs) == len(phases)
    for r in recs:
        assert 0 < r[4] <= r[5] <= r[7], r
    end_a = max(r[7] for r in recs if r[0] == 0)
    end_b = max(r[7] for r in recs if r[0] == 1)
    assert min(r[5] for r in recs if r[0] == 1) >= end_a - 1000   # globaltimer granularity
    assert min(r[5] for r in recs if r[0] == 2) >= end_b - 1000
    if name == "2d_f32":
        ref = run_oracle(case, x, w)
    else:
        ref = None
    got = y.cpu().numpy()
    if ref is not None:
        assert_close(got, ref, "f32", "traced three-kernel forward")
    conv.close()


PACKED_CASES = [
    ((256,), (16,), 3, 5, 7, "f32"),               # 1-D cluster kernel
    ((128, 128), (16, 16), 2, 6, 5, "f32"),        # three-kernel 128^2
    ((128, 128), (16, 16), 2, 6, 5, "f32", capi.FNO_PLAN_PERSISTENT),
    ((256, 256), (32, 32), 2, 3, 5, "f16"),        # tensor-core mixing
    ((256, 256), (32, 32), 3, 64, 64, "f16"),      # ... weights as operand images
    ((256, 256), (32, 32), 2, 64, 64, "bf16"),
    ((256, 256), (32, 32), 1, 4, 4, "bf16", capi.FNO_PLAN_SIMT_MIX),
    ((64, 64, 64), (16, 16, 16), 1, 3, 2, "f32"),  # 3-D
    ((16, 32), (3, 8), 2, 3, 5, "f32"),            # separate kernels
]


@pytest.mark.parametrize("spec", PACKED_CASES, ids=[case_id(c[:6]) + ("_f" if len(c) > 6 else "")
                                                   for c in PACKED_CASES])
def test_packed_weights_match_oracle(spec):
    n, modes, b, ci, co, dt = spec[:6]
    flags = capi.FNO_PLAN_PACKED_WEIGHTS | (spec[6] if len(spec) > 6 else 0)
    case = workloads.small_case(n, modes, b, ci, co, dt)
    x = workloads.make_x(case, seed=61)
    w = workloads.to_storage((workloads.make_w(case, seed=62).astype(np.float64) * ci * co * 2 - 1)
                             / ci, dt)
    conv = SpectralConv(n, modes, b, ci, co, dt, flags)
    W = to_dev(w, dt)
    wp = conv.pack_weights(W)
    torch.cuda.synchronize()
    assert not torch.equal(wp, W) or w.size <= 8
    y = conv(to_dev(x, dt), wp)
    torch.cuda.synchronize()
    assert conv.device_error() == 0
    assert_close(y.float().cpu().numpy(), run_oracle(case, x, w), dt, "packed weights")
    conv.close()


def test_output_red_zones_untouched():
    case = workloads.small_case((64, 64), (8, 8), 2, 3, 4, "f32")
    x, w = workloads.make_x(case, seed=3), workloads.make_w(case, seed=4)
    conv = SpectralConv(case.n, case.modes, 2, 3, 4)
    guard = 1024
    ny = int(np.prod(case.y_shape))
    buf = torch.full((ny + 2 * guard,), 12345.0, device="cuda")
    y = buf[guard:guard + ny].view(case.y_shape)
    conv(to_dev(x), to_dev(w), y)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 12345.0) and torch.all(buf[guard + ny:] == 12345.0)
    assert_close(y.cpu().numpy(), run_oracle(case, x, w), "f32", "red zone case")
    conv.close()


def test_forward_error_paths():
    case = workloads.small_case((32, 32), (4, 4), 1, 2, 2, "f32")
    conv = SpectralConv(case.n, case.modes, 1, 2, 2)
    x = to_dev(workloads.make_x(case, seed=1))
    w = to_dev(workloads.make_w(case, seed=2))
    y = torch.empty(case.y_shape, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ws = conv.workspace.data_ptr() if conv.workspace is not None else None
    st = capi.fno_spectral_conv_forward(conv.handle, x.data_ptr() + 4, w.data_ptr(),
                                        y.data_ptr(), ws, s)
    assert st == capi.FNO_ERR_MISALIGNED
    st = capi.fno_spectral_conv_forward(conv.handle, x.data_ptr(), w.data_ptr(),
                                        x.data_ptr(), ws, s)
    assert st == capi.FNO_ERR_ALIASING
    st = capi.fno_spectral_conv_forward(conv.handle, 0, w.data_ptr(), y.data_ptr(), ws, s)
    assert st == capi.FNO_ERR_INVALID_ARG
    with pytest.raises(TypeError):
        conv(x.double(), w)
    conv.close()


def test_injected_launch_failure_reports_and_recovers(monkeypatch):
    case = workloads.small_case((32, 32), (4, 4), 1, 2, 2, "f32")
    x, w = workloads.make_x(case, seed=1), workloads.make_w(case, seed=2)
    conv = SpectralConv(case.n, case.modes, 1, 2, 2)
    monkeypatch.setenv("FNO_FAULT_INJECT", "launch")
    with pytest.raises(FnoError) as ei:
        conv(to_dev(x), to_dev(w))
    assert ei.value.status == capi.FNO_ERR_CUDA
    monkeypatch.delenv("FNO_FAULT_INJECT")
    y = conv(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    assert conv.device_error() == capi.FNO_OK
    assert_close(y.cpu().numpy(), run_oracle(case, x, w), "f32", "after recovery")
    conv.close()


def test_plan_create_destroy_many_times_no_leak():
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(50):
        st, h = capi.fno_spectral_conv_plan(2, [128, 128], [16, 16], 8, 32, 32, capi.FNO_F32)
        assert st == capi.FNO_OK
        assert capi.fno_plan_destroy(h) == capi.FNO_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free0 - free1 < 8 << 20


def test_trace_records_every_item():
    case = workloads.CASES["2d_f32"]
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype,
                        capi.FNO_PLAN_TRACE | capi.FNO_PLAN_PERSISTENT)
    x, w = workloads.make_x(case), workloads.make_w(case)
    y = conv(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    st, recs = capi.fno_plan_get_trace(conv.handle)
    assert st == capi.FNO_OK
    phases = [r[0] for r in recs]
    nin, nout = case.batch * case.cin, case.batch * case.cout
    assert phases.count(0) % nin == 0 and phases.count(0) > 0
    assert phases.count(2) // nout == phases.count(0) // nin and phases.count(2) % nout == 0
    assert phases.count(1) > 0
    for r in recs:
        assert r[4] <= r[5] <= r[6] <= r[7], r
    # tracing does not change the result
    assert_close(y.cpu().numpy(), run_oracle(case, x, w), "f32", "traced forward")
    st, _ = capi.fno_plan_get_trace(SpectralConv((16,), (4,), 1, 1, 1).handle)
    assert st == capi.FNO_ERR_INVALID_ARG
    conv.close()


PADDED = [
    # (n, pad, modes, batch, cin, cout, dtype): the layer on a zero-padded,
    # cropped domain against the oracle's plain pad -> layer -> crop
    ((12,), (4,), (4,), 2, 3, 5, "f32"),
    ((250,), (6,), (16,), 3, 4, 4, "f32"),            # padded to a power of two
    ((10,), (5,), (5,), 2, 2, 3, "f32"),              # odd transform length, no Nyquist
    ((6,), (2,), (5,), 1, 3, 2, "f32"),               # Nyquist bin kept
    ((100, 120), (28, 8), (16, 16), 2, 8, 6, "f32"),  # 2-D, L = 128 x 128
    ((6, 10), (2, 6), (2, 6), 2, 3, 2, "f16"),
    ((5, 7), (3, 1), (3, 2), 2, 2, 3, "bf16"),
    ((30, 20, 12), (2, 12, 4), (8, 8, 5), 1, 3, 4, "f32"),   # 3-D, L = 32^3 x 16
]


@pytest.mark.parametrize("spec", PADDED, ids=[f"{'x'.join(map(str, c[0]))}_p"
                                               f"{'x'.join(map(str, c[1]))}_{c[6]}"
                                              for c in PADDED])
def test_padded_layer_matches_oracle(spec):
    n, pad, modes, b, ci, co, dt = spec
    L = tuple(a + p for a, p in zip(n, pad))
    case = workloads.small_case(n, modes, b, ci, co, dt, index=9)
    wcase = workloads.small_case(L, modes, b, ci, co, dt, index=9)
    x = workloads.make_x(case, seed=300 + sum(n))
    w = workloads.make_w(wcase, seed=400 + sum(pad))
    conv = SpectralConv(n, modes, b, ci, co, dt, pad=pad)
    assert conv.kernel_count == 2 * len(n) + 1              # the separate kernels
    y = torch.full((b, co) + n, float("nan"), device="cuda").to(conv.torch_dtype)
    conv(to_dev(x, dt), to_dev(w, dt), y)
    torch.cuda.synchronize()
    assert conv.device_error() == 0
    conv.close()
    ref = oracle.spectral_conv_padded(x.astype(np.float64), workloads.as_complex(w), modes, pad)
    assert_close(y.float().cpu().numpy(), ref, dt, f"padded {spec}")


def test_padded_zero_pad_equals_periodic_plan():
    case = workloads.small_case((64, 64), (8, 8), 2, 4, 4, "f32", index=9)
    x, w = workloads.make_x(case, seed=5), workloads.make_w(case, seed=6)
    a, _ = run_gpu(case, x, w, FNO_PLAN_UNFUSED)
    conv = SpectralConv(case.n, case.modes, 2, 4, 4, "f32", pad=(0, 0))
    b = conv(to_dev(x), to_dev(w)).cpu().numpy()
    conv.close()
    assert np.array_equal(a, b)
