"""Run a workload's forward a fixed number of times, for profiler captures.

    python -m fft_gemm_ifft_gb300.profile_run --workload 2d_f32 --iters 20 [--flags 0]
    python -m fft_gemm_ifft_gb300.profile_run --workload fno2d_f32 --iters 20 --time

Inputs are seeded (``workloads``) and rotate through enough (x, w, y) sets to
exceed twice the L2 size, as in the benchmark; every forward is an eager call
through the C ABI on one stream.  ``--workload fno2d_f32`` runs the FNO stack
(``fno_forward``) instead of one layer.  With ``--time`` the forwards are timed
with CUDA events on the launching stream (after the same number of warm-up
forwards) and the median and 10th/90th percentiles are printed.  Exits non-zero
if the device error word is set.  The profiler picks kernels with -k/-s/-c.
"""
from __future__ import annotations

import argparse
import math
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="2d_f32")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the batch size")
    ap.add_argument("--channels", type=int, default=0,
                    help="override the input and output channel counts")
    ap.add_argument("--trace", default="", help="write the last call's work-item trace "
                    "(CSV) here and print a per-phase summary")
    ap.add_argument("--time", action="store_true", help="time each forward with CUDA events")
    ap.add_argument("--dtype", default="f32", choices=["f32", "f16", "bf16"],
                    help="storage type of the FNO stack (fno2d_f32 workload shape)")
    ap.add_argument("--sets", type=int, default=0,
                    help="input sets rotated over (default: enough to cover twice the L2; "
                         "1 keeps the inputs L2-resident)")
    ap.add_argument("--backward", action="store_true",
                    help="run (and time) fno_spectral_conv_backward (dx and dw) instead")
    args = ap.parse_args(argv)

    import torch

    from . import SpectralConv, build, workloads
    build.build()
    if args.workload == workloads.FNO_CASE.name:
        return run_fno(args)
    case = workloads.CASES[args.workload]
    if args.batch:
        case = case.with_batch(args.batch)
    if args.channels:
        import dataclasses
        case = dataclasses.replace(case, cin=args.channels, cout=args.channels)
    from . import capi
    flags = args.flags | (capi.FNO_PLAN_TRACE if args.trace else 0)
    if args.backward:
        flags |= capi.FNO_PLAN_BACKWARD
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype, flags)
    x_np, w_np = workloads.make_x(case), workloads.make_w(case)
    set_bytes = x_np.nbytes + w_np.nbytes + math.prod(case.y_shape) * case.elem_bytes
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or (126 << 20)
    nsets = args.sets or max(2, math.ceil(2 * l2 / set_bytes))
    xs = [workloads.to_torch_storage(x_np, case.dtype).cuda() for _ in range(nsets)]
    ws = [workloads.to_torch_storage(w_np, case.dtype).cuda() for _ in range(nsets)]
    if flags & capi.FNO_PLAN_PACKED_WEIGHTS:
        ws = [conv.pack_weights(w) for w in ws]
    ys = [torch.empty(case.y_shape, dtype=conv.torch_dtype, device="cuda") for _ in range(nsets)]
    step = lambda i: conv(xs[i % nsets], ws[i % nsets], ys[i % nsets])
    if args.backward:
        dxs = [torch.empty_like(x) for x in xs]
        dws = [torch.empty_like(w) for w in ws]
        step = lambda i: conv.backward(xs[i % nsets], ws[i % nsets], ys[(i + 1) % nsets],
                                       dx=dxs[i % nsets], dw=dws[i % nsets])
        for y in ys:
            y.copy_(torch.randn(y.shape, dtype=torch.float32).to(y.dtype))
    if args.time:
        report_times(case.name, case.batch, time_steps(step, args.iters))
    else:
        for i in range(args.iters):
            step(i)
    torch.cuda.synchronize()
    if args.trace:
        tst, recs = capi.fno_plan_get_trace(conv.handle)
        if tst != capi.FNO_OK:
            print("trace unavailable:", capi.fno_status_string(tst))
        else:
            summarize_trace(recs, args.trace)
    st = conv.device_error()
    conv.close()
    print(f"{args.iters} forwards of {case.name}, kernels/forward {conv.kernel_count}, "
          f"device status {st}")
    return 0 if st == 0 else 1


def time_steps(step, iters):
    """Per-call device times (microseconds) of `iters` calls after as many warm-up
    calls, CUDA events on the current stream."""
    import torch
    for i in range(iters):
        step(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    torch.cuda.synchronize()
    ev[0].record()
    for i in range(iters):
        step(i)
        ev[i + 1].record()
    torch.cuda.synchronize()
    return sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(iters))


def report_times(name, batch, ts):
    med = ts[len(ts) // 2]
    print(f"{name}: median {med:.2f} us (p10 {ts[len(ts) // 10]:.2f}, p90 "
          f"{ts[(9 * len(ts)) // 10]:.2f}) over {len(ts)} calls, {batch / med * 1e6:.1f} samples/s")


def run_fno(args) -> int:
    import torch

    from . import FnoModel, workloads
    case = workloads.FNO_CASE
    batch = args.batch or case.batch
    dt = args.dtype
    m = FnoModel(batch, case.h, case.w, case.modes, case.cin_lift, case.width, case.nlayers,
                 case.hidden, case.cout, flags=args.flags, dtype=dt)
    x = workloads.to_torch_storage(
        workloads.to_storage(workloads.make_fno_inputs(case, batch), dt), dt).cuda()
    p = {k: (workloads.to_torch_storage(workloads.to_storage(v, dt), dt) if k == "spec_w"
             else torch.from_numpy(v)).cuda()
         for k, v in workloads.make_fno_params(case).items()}
    y = torch.empty(m.y_shape, dtype=m.torch_dtype, device="cuda")
    step = lambda i: m(x, p, y)
    if args.time:
        report_times(case.name, batch, time_steps(step, args.iters))
    else:
        for i in range(args.iters):
            step(i)
    torch.cuda.synchronize()
    st = m.device_error()
    m.close()
    print(f"{args.iters} forwards of {case.name}, kernels/forward {m.kernel_count}, "
          f"device status {st}")
    return 0 if st == 0 else 1


def summarize_trace(recs, path):
    """Per-phase timeline of one fused launch: when each phase ran and where
    its items spent their time (microseconds)."""
    if not recs:
        print("empty trace")
        return
    t0 = min(r[4] for r in recs)
    with open(path, "w") as f:
        f.write("phase,group,index,worker,start_us,ready_us,compute_us,end_us\n")
        for r in recs:
            f.write(",".join(str(v) for v in r[:4]) + "," +
                    ",".join(f"{(t - t0) / 1e3:.3f}" for t in r[4:]) + "\n")
    names = {0: "A transform", 1: "B mixing", 2: "C inverse"}
    print(f"{'phase':12s} {'items':>5s} {'first':>7s} {'last':>7s} {'wait':>6s} "
          f"{'compute':>7s} {'tail':>6s}   (us; wait/compute/tail = mean per item)")
    for ph in sorted({r[0] for r in recs}):
        rs = [r for r in recs if r[0] == ph]
        n = len(rs)
        first = min(r[4] for r in rs) - t0
        last = max(r[7] for r in rs) - t0
        wait = sum(r[5] - r[4] for r in rs) / n
        comp = sum(r[6] - r[5] for r in rs) / n
        tail = sum(r[7] - r[6] for r in rs) / n
        print(f"{names.get(ph, ph):12s} {n:5d} {first / 1e3:7.2f} {last / 1e3:7.2f} "
              f"{wait / 1e3:6.2f} {comp / 1e3:7.2f} {tail / 1e3:6.2f}")
    print(f"kernel span {(max(r[7] for r in recs) - t0) / 1e3:.2f} us (first item start to "
          f"last item end)")


if __name__ == "__main__":
    sys.exit(main())
