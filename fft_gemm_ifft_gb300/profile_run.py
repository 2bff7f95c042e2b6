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
    args = ap.parse_args(argv)

    import torch

    from . import SpectralConv, build, workloads
    build.build()
    case = workloads.CASES[args.workload]
    if args.batch:
        case = case.with_batch(args.batch)
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype,
                        args.flags)
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
    st = conv.device_error()
    conv.close()
    print(f"{args.iters} forwards of {case.name}, kernels/forward {conv.kernel_count}, "
          f"device status {st}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
