"""GPU parity of the FNO forward stack (fno_forward) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from fft_gemm_ifft_gb300 import FnoModel, capi, workloads
from parity_util import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(fno, oracle_mod):
    yield


def run_model(case, x, params, batch, flags=0):
    m = FnoModel(batch, case.h, case.w, case.modes, case.cin_lift, case.width, case.nlayers,
                 case.hidden, case.cout, flags=flags)
    dev = {k: to_dev(v) for k, v in params.items()}
    y = m(to_dev(x), dev)
    torch.cuda.synchronize()
    assert m.device_error() == 0
    kernels = m.kernel_count
    m.close()
    return y.cpu().numpy(), kernels


def test_small_stack_matches_oracle():
    case = workloads.FnoCase("small", batch=2, width=8, nlayers=2, h=32, w=32, modes=(4, 4),
                             hidden=16, cout=2)
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    got, _ = run_model(case, x, p, case.batch)
    ref = oracle.fno_forward(x, workloads.fno_params_for_oracle(p), case.modes)
    assert_close(got, ref, "f32", "small FNO stack")


@pytest.mark.parametrize("shape", [
    # batch, width, nlayers, h, w, modes, hidden, cout: channel counts that are
    # not multiples of the 64-wide tiles and span two input-channel chunks,
    # several output groups, and pixel counts below one 128-pixel tile
    (3, 70, 1, 16, 16, (4, 4), 70, 3),
    (2, 5, 2, 2, 2, (1, 1), 9, 1),
    (1, 12, 2, 8, 16, (2, 3), 130, 8),
    (2, 6, 1, 12, 20, (3, 4), 10, 1),
    # tensor-core linears (32 / 64 input channels, multiples of 16 outputs),
    # including a last tile with fewer than 128 pixels
    (2, 32, 2, 8, 16, (2, 3), 48, 3),
    (1, 64, 1, 8, 8, (2, 2), 16, 2),
    (3, 64, 2, 16, 32, (4, 4), 128, 1),
], ids=["ragged_channels", "tiny_grid", "wide_hidden", "grid_not_power_of_two",
        "tc_32_channels", "tc_partial_tile", "tc_64_channels"])
def test_stack_ragged_tiles(shape):
    b, width, nl, h, w, modes, hidden, cout = shape
    case = workloads.FnoCase("ragged", batch=b, width=width, nlayers=nl, h=h, w=w,
                             modes=modes, hidden=hidden, cout=cout)
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    got, _ = run_model(case, x, p, case.batch)
    ref = oracle.fno_forward(x, workloads.fno_params_for_oracle(p), case.modes)
    assert_close(got, ref, "f32", f"FNO stack {shape}")


@pytest.mark.parametrize("shape", [
    # batch, width, nlayers, hidden, cout on the 128 x 128 grid, 16 x 16 modes:
    # the layers' output half as one GEMM per image row (default) or as the
    # inverse kernel plus the 1x1-linear kernel (FNO_PLAN_SPLIT_LAYER); batch 3
    # leaves the persistent CTAs unequal tile counts, the last layer has no GELU
    (2, 64, 2, 128, 1),
    (3, 32, 2, 48, 2),
    (1, 64, 1, 16, 3),
], ids=["w64", "w32_uneven_tiles", "single_layer"])
@pytest.mark.parametrize("flags", [0, capi.FNO_PLAN_SPLIT_LAYER, capi.FNO_PLAN_TENSOR_EXTRA],
                         ids=["fused_layer", "split_layer", "fused_layer_tc_mix"])
def test_layer_output_paths_match_oracle(shape, flags):
    b, width, nl, hidden, cout = shape
    case = workloads.FnoCase("layer", batch=b, width=width, nlayers=nl, h=128, w=128,
                             modes=(16, 16), hidden=hidden, cout=cout)
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    got, kernels = run_model(case, x, p, case.batch, flags)
    # lift, four kernels a layer, head
    assert kernels == 2 + 4 * nl
    ref = oracle.fno_forward(x, workloads.fno_params_for_oracle(p), case.modes)
    assert_close(got, ref, "f32", f"FNO stack {shape} flags={flags}")


@pytest.mark.parametrize("shape", [
    # batch, width, nlayers, h, w, hidden, cout: the persistent head kernel's
    # variants (32 / 64 inputs, 64 / 128 hidden units, one or several outputs),
    # pixel counts that are whole 128-pixel tiles, tile counts that leave the
    # CTAs unequal shares
    (3, 64, 1, 16, 32, 128, 1),
    (2, 32, 1, 32, 16, 64, 3),
    (1, 64, 1, 8, 48, 64, 8),
    (5, 32, 1, 16, 16, 128, 2),
], ids=["c64_h128_o1", "c32_h64_o3", "c64_h64_o8", "c32_h128_o2"])
def test_head_kernel_shapes(shape):
    b, width, nl, h, w, hidden, cout = shape
    case = workloads.FnoCase("head", batch=b, width=width, nlayers=nl, h=h, w=w, modes=(2, 2),
                             hidden=hidden, cout=cout)
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    got, _ = run_model(case, x, p, case.batch)
    ref = oracle.fno_forward(x, workloads.fno_params_for_oracle(p), case.modes)
    assert_close(got, ref, "f32", f"FNO head {shape}")


def test_fused_layer_output_is_a_different_path():
    # the fused output half sums the inverse row DFT and the 1x1 linear in one
    # accumulator: equal to the split path within rounding, not bit for bit
    case = workloads.FnoCase("layer", batch=1, width=64, nlayers=1, h=128, w=128,
                             modes=(16, 16), hidden=16, cout=1)
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    fused, _ = run_model(case, x, p, case.batch, 0)
    split, _ = run_model(case, x, p, case.batch, capi.FNO_PLAN_SPLIT_LAYER)
    assert not np.array_equal(fused, split)
    assert_close(fused, split, "f32", "fused vs split layer output")


def test_full_stack_sampled():
    case = workloads.FNO_CASE
    x = workloads.make_fno_inputs(case)
    p = workloads.make_fno_params(case)
    got, _ = run_model(case, x, p, case.batch)
    q = workloads.fno_params_for_oracle(p)
    for b in (0, case.batch - 1):
        ref = oracle.fno_forward(x[b:b + 1], q, case.modes)
        assert_close(got[b:b + 1], ref, "f32", f"FNO b={b}")


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [
    # batch, width, nlayers, h, w, modes, hidden, cout, flags
    (2, 8, 2, 32, 32, (4, 4), 16, 2, 0),
    (3, 70, 1, 16, 16, (4, 4), 70, 3, 0),           # ragged channel tiles
    # the 128^2 layers: the one-GEMM output half (16-bit activations, no
    # remainder operand) and the split form
    (2, 64, 2, 128, 128, (16, 16), 128, 1, 0),
    (3, 32, 2, 128, 128, (16, 16), 48, 2, 0),
    (2, 64, 2, 128, 128, (16, 16), 128, 1, 512),
    # the persistent head kernel with 16-bit activations and output, 8-output
    # variant (32 -> 64 -> 3) on whole 128-pixel tiles
    (2, 32, 1, 16, 32, (2, 2), 64, 3, 0),
], ids=["small", "ragged_channels", "layer_128", "layer_128_w32", "layer_128_split",
        "head_c32_h64_o3"])
def test_stack_16bit_storage(dt, shape):
    # x, the activations, spec_w and out stored in fp16 / bf16, arithmetic in
    # float32; the oracle runs in float64 on the same rounded x and spec_w, so
    # the difference is the rounding of the stored activations (the 16-bit
    # tolerance class)
    b, width, nl, h, w, modes, hidden, cout, flags = shape
    case = workloads.FnoCase("half", batch=b, width=width, nlayers=nl, h=h, w=w, modes=modes,
                             hidden=hidden, cout=cout)
    x = workloads.to_storage(workloads.make_fno_inputs(case), dt)
    p = workloads.make_fno_params(case)
    p["spec_w"] = workloads.to_storage(p["spec_w"], dt)
    m = FnoModel(b, h, w, modes, case.cin_lift, width, nl, hidden, cout, flags=flags, dtype=dt)
    dev = {k: to_dev(v, dt) if k == "spec_w" else to_dev(v) for k, v in p.items()}
    y = m(to_dev(x, dt), dev)
    torch.cuda.synchronize()
    assert y.dtype == m.torch_dtype
    assert m.device_error() == 0
    m.close()
    ref = oracle.fno_forward(x.astype(np.float64), workloads.fno_params_for_oracle(p), modes)
    assert_close(y.float().cpu().numpy(), ref, dt, f"16-bit FNO stack {shape}")


@pytest.mark.parametrize("shape", [
    # batch, width, nlayers, h, w, modes, hidden, cout
    (2, 8, 2, 32, 32, (4, 4), 16, 2),             # register-tiled linears
    (2, 64, 2, 128, 128, (16, 16), 128, 1),       # three-kernel 128^2 layers, tensor-core linears
], ids=["small", "layer_128"])
def test_fno_forward_graph_capture_replays(shape):
    # One fno_forward captured in a CUDA graph, replayed twice on new inputs
    # (and new parameters) copied into the captured buffers; each replay is
    # compared with the oracle.  The call allocates nothing and syncs nothing,
    # so the graph holds the whole stack.
    b, width, nl, h, w, modes, hidden, cout = shape
    case = workloads.FnoCase("graph", batch=b, width=width, nlayers=nl, h=h, w=w, modes=modes,
                             hidden=hidden, cout=cout)
    m = FnoModel(b, h, w, modes, case.cin_lift, width, nl, hidden, cout)
    x0 = workloads.make_fno_inputs(case)
    p0 = workloads.make_fno_params(case)
    xd = to_dev(x0)
    pd = {k: to_dev(v) for k, v in p0.items()}
    yd = torch.empty(m.y_shape, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        m(xd, pd, yd, stream=s)                    # warm-up outside the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            m(xd, pd, yd, stream=s)
    r = np.random.default_rng(77)
    for rep in range(2):
        x = x0.copy()
        x[:, 0] = r.standard_normal(x[:, 0].shape).astype(np.float32)
        p = {k: (v * np.float32(1.0 + 0.25 * (rep + 1))).astype(np.float32)
             if k in ("spec_w", "pw_w") else v for k, v in p0.items()}
        xd.copy_(torch.from_numpy(x))
        for k in ("spec_w", "pw_w"):
            pd[k].copy_(torch.from_numpy(p[k]))
        yd.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert m.device_error() == 0
        ref = oracle.fno_forward(x, workloads.fno_params_for_oracle(p), modes)
        assert_close(yd.cpu().numpy(), ref, "f32", f"graph replay {rep} {shape}")
    m.close()
