"""Run a workload's forward a fixed number of times, for profiler captures.

    python -m fft_gemm_ifft_gb300.profile_run --workload 2d_f32 --iters 20 [--flags 0]

Inputs are seeded (``workloads``) and rotate through enough (x, w, y) sets to
exceed twice the L2 size, as in the benchmark; every forward is an eager call
through the C ABI on one stream.  Exits non-zero if the device error word is
set.  The profiler picks kernels with -k/-s/-c.
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
    ap.add_argument("--trace", default="", help="write the last call's work-item trace "
                    "(CSV) here and print a per-phase summary")
    args = ap.parse_args(argv)

    import torch

    from . import SpectralConv, build, workloads
    build.build()
    case = workloads.CASES[args.workload]
    if args.batch:
        case = case.with_batch(args.batch)
    from . import capi
    flags = args.flags | (capi.FNO_PLAN_TRACE if args.trace else 0)
    if args.trace and not flags & capi.FNO_PLAN_TENSOR_CORES:
        flags |= capi.FNO_PLAN_PERSISTENT       # the trace covers the persistent kernels
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype, flags)
    x_np, w_np = workloads.make_x(case), workloads.make_w(case)
    set_bytes = x_np.nbytes + w_np.nbytes + math.prod(case.y_shape) * case.elem_bytes
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or (126 << 20)
    nsets = max(2, math.ceil(2 * l2 / set_bytes))
    xs = [torch.from_numpy(x_np).cuda() for _ in range(nsets)]
    ws = [torch.from_numpy(w_np).cuda() for _ in range(nsets)]
    ys = [torch.empty(case.y_shape, dtype=conv.torch_dtype, device="cuda") for _ in range(nsets)]
    for i in range(args.iters):
        conv(xs[i % nsets], ws[i % nsets], ys[i % nsets])
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
