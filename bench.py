"""Benchmark of the FNO spectral-convolution layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload 2d_f32]

One step is one forward pass of the layer (truncated forward FFT, per-mode
mixing, inverse FFT) over one batch of the workload, through the C ABI.
Inputs are resident in device memory before the timed region; successive
steps rotate through enough distinct (x, w, y) sets to exceed twice the L2
size, so every step reads and writes HBM.  Steps are replayed from a CUDA
graph (the forward call is capturable) so host launch overhead does not
pace the GPU.  Under torchrun each rank runs its own batch (weak scaling,
replicas: the layer has no exchange step), the timed region is bracketed by
barriers and the slowest rank's time is reported.

``--impl reference`` times the float64 CPU oracle on the same workload (one
sample of the batch per step, on all host cores); it is a deliberately slow
baseline, printed in the same JSON format.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "spectral-conv samples/s & achieved HBM GB/s / roofline fraction on 1 GB300"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="2d_f32")
    ap.add_argument("--flags", type=int, default=0, help="FNO_PLAN_* bits (ablations)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=200)
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    """Digest of the CUDA sources: a traffic figure taken from an ncu capture
    is reported only while the kernels are unchanged since that capture."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fft_gemm_ifft_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (profiles/traffic.json), or None if the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("source_digest") != kernel_source_digest():
            return None
        return int(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the GPU is loaded."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.out.name) as f:
            for ln in f:
                p = [v.strip() for v in ln.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.out.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of one float per rank (the slowest rank's time); a no-op
    for a single process.  Works on any process-group backend: the tensor
    lives on `device` (a CUDA device under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(batch_per_rank: int, world: int, steps: int, ms_max: float) -> float:
    """Samples per second of the whole job: every rank runs `steps` forwards
    of its own batch (weak scaling), timed by the slowest rank."""
    return world * batch_per_rank * steps / (ms_max / 1e3)


def e2e_pipelined(torch, conv, case, x_np, ws, stream, steps, world, dev, dist):
    """Milliseconds for `steps` host-to-host forwards through the public API,
    pipelined over three slots (H2D, layer, D2H on their own streams)."""
    from fft_gemm_ifft_gb300 import workloads
    nslot = 3
    x_host = workloads.to_torch_storage(x_np, case.dtype).pin_memory()
    y_host = [torch.empty(case.y_shape, dtype=conv.torch_dtype).pin_memory() for _ in range(nslot)]
    xd = [torch.empty(case.x_shape, dtype=conv.torch_dtype, device=dev) for _ in range(nslot)]
    yd = [torch.empty(case.y_shape, dtype=conv.torch_dtype, device=dev) for _ in range(nslot)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()

    def run(n):
        done_out = [None] * nslot          # D2H of the slot's previous step
        for i in range(n):
            k = i % nslot
            with torch.cuda.stream(s_in):
                if done_out[k] is not None:
                    s_in.wait_event(done_out[k])       # slot free: its output has left
                xd[k].copy_(x_host, non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
            stream.wait_event(e_in)
            conv(xd[k], ws[k % len(ws)], yd[k], stream=stream)
            e_cp = ev()
            e_cp.record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_cp)
                y_host[k].copy_(yd[k], non_blocking=True)
                done_out[k] = ev()
                done_out[k].record(s_out)

    run(nslot)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    stream.wait_event(e0)
    s_out.wait_event(e0)
    run(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return max_over_ranks(e0.elapsed_time(e1), world, dev)


def bench_gpu(args, rank, world, local):
    import numpy as np
    import torch
    import torch.distributed as dist

    from fft_gemm_ifft_gb300 import SpectralConv, workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = workloads.CASES[args.workload]
    conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout, case.dtype,
                        args.flags)
    x_np, w_np = workloads.make_x(case), workloads.make_w(case)
    set_bytes = (x_np.nbytes + w_np.nbytes + math.prod(case.y_shape) * case.elem_bytes)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0)) or (126 << 20)
    nsets = max(2, math.ceil(2 * l2 / set_bytes))
    xs = [workloads.to_torch_storage(x_np, case.dtype).to(dev) for _ in range(nsets)]
    ws = [workloads.to_torch_storage(w_np, case.dtype).to(dev) for _ in range(nsets)]
    from fft_gemm_ifft_gb300 import capi as _capi
    if args.flags & _capi.FNO_PLAN_PACKED_WEIGHTS:
        # weights are parameters: packed once per set, outside the timed region
        ws = [conv.pack_weights(w) for w in ws]
    ys = [torch.empty(case.y_shape, dtype=conv.torch_dtype, device=dev) for _ in range(nsets)]

    stream = torch.cuda.Stream(device=dev)
    steps = max(1, args.steps)
    per_graph = min(steps, nsets * max(1, 64 // nsets))
    reps, tail = divmod(steps, per_graph)

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                conv(xs[i % nsets], ws[i % nsets], ys[i % nsets], stream=stream)
        return g

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):            # eager warm-up steps
            conv(xs[i % nsets], ws[i % nsets], ys[i % nsets], stream=stream)
        stream.synchronize()
        assert conv.device_error(stream) == 0
        graph = capture(per_graph)
        graph_tail = capture(tail) if tail else None
        for _ in range(3):
            graph.replay()
        stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # pre-heat of the same workload so the clock samples see a loaded GPU
    with torch.cuda.stream(stream):
        t_end = time.time() + 1.5
        while time.time() < t_end:
            graph.replay()
            stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        if graph_tail is not None:
            graph_tail.replay()
        end.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_max = max_over_ranks(start.elapsed_time(end), world, dev)
    stream.synchronize()
    assert conv.device_error(stream) == 0

    # L2-resident ("hot") figure for workloads whose set fits in L2: the same
    # number of forwards on one (x, w, y) set, reported beside the rotated value
    hot_ms = None
    if set_bytes < l2:
        with torch.cuda.stream(stream):
            g_hot = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_hot, stream=stream):
                for _ in range(per_graph):
                    conv(xs[0], ws[0], ys[0], stream=stream)
            for _ in range(3):
                g_hot.replay()
            h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            h0.record(stream)
            for _ in range(reps):
                g_hot.replay()
            h1.record(stream)
        torch.cuda.synchronize(dev)
        hot_ms = max_over_ranks(h0.elapsed_time(h1), world, dev) / (reps * per_graph)
        assert conv.device_error(stream) == 0

    # end to end through the public API: every step copies its input from pinned
    # host memory, runs the layer and copies its output back to pinned host
    # memory.  The steps are pipelined over three device buffer slots and three
    # streams (copy in, layer, copy out), as a serving loop would run them: the
    # input of step i+1 and the output of step i-1 move while step i computes.
    e2e_steps = max(3, args.e2e_steps)
    e2e_ms = e2e_pipelined(torch, conv, case, x_np, ws, stream, e2e_steps, world, dev, dist)

    value = whole_job_rate(case.batch, world, steps, ms_max)
    kernel_ms = ms_max / steps          # back-to-back graph replay: per-forward duration
    peak, peak_kind = measured_peaks()
    alg_bytes = case.algorithmic_bytes()
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "samples/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms_max / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if case.dtype == "f32" else f"{case.dtype}-storage/f32-accumulate",
        "data": "synthetic (seeded N(0,1) fields, U[0,1)/(Cin*Cout) complex weights)",
        "config": {
            "workload": f"{case.name}: {case.ndim}-D spectral conv, B={case.batch}, "
                        f"Cin={case.cin}, Cout={case.cout}, N={'x'.join(map(str, case.n))}, "
                        f"modes={'x'.join(map(str, case.modes))} per block, "
                        f"{case.nblk} block(s)",
            "global_batch": world * case.batch,
            "parallelism": f"replicas x{world}",
            "l2": f"rotating {nsets} distinct (x, w, y) sets = {nsets * set_bytes >> 20} MiB "
                  f"> 2 x L2 ({l2 >> 20} MiB)",
            "timing": f"CUDA-graph replay of {per_graph} forwards x {reps} (+{tail}), "
                      "CUDA events on the launching stream",
            "plan_flags": args.flags,
            "weights": ("packed mode-major once per set, outside the timed region"
                        if args.flags & 128 else "as given (nblk, Cin, Cout, modes)"),
            "hot_l2_ms_per_step": hot_ms,
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "fno_spectral_conv_forward" if conv.kernel_count > 1
                      else "fused spectral-conv kernel",
            "kernels_per_forward": conv.kernel_count,
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": alg_bytes,
            # the committed capture covers the default kernels only
            "traffic": recorded_traffic(case.name) if args.flags == 0 else None,
        },
        "e2e": {
            "value": round(whole_job_rate(case.batch, world, e2e_steps, e2e_ms), 1),
            "unit": "samples/s",
            "h2d_bytes_per_step": int(math.prod(case.x_shape) * case.elem_bytes),
            "pipelining": "3 buffer slots; input copy, layer and output copy on separate streams",
            "d2h_bytes_per_step": int(math.prod(case.y_shape) * case.elem_bytes),
        },
        "gpu_launches": steps * conv.kernel_count,
        "clocks": clocks,
    }
    return result, case, x_np, w_np


def cpu_baseline(case, x_np, w_np, seconds: float):
    """The oracle as it stands, on the host cores, over whole samples of the
    same workload until `seconds` of work have run."""
    import numpy as np

    import oracle
    from fft_gemm_ifft_gb300 import workloads

    oracle.build()
    nthreads = len(os.sched_getaffinity(0))
    oracle.set_threads(nthreads)
    wc = workloads.as_complex(w_np)
    done, t0 = 0, time.perf_counter()
    while True:
        b = done % case.batch
        oracle.spectral_conv(x_np[b:b + 1].astype(np.float64), wc, case.modes)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = oracle.get_threads()
    # the same oracle on one thread, over a third of the time
    oracle.set_threads(1)
    done1, t1 = 0, time.perf_counter()
    while True:
        b = done1 % case.batch
        oracle.spectral_conv(x_np[b:b + 1].astype(np.float64), wc, case.modes)
        done1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= seconds / 3:
            break
    oracle.set_threads(nthreads)
    return {"value": round(done / el, 3), "unit": "samples/s", "cores": cores,
            "kind": "oracle",
            "value_1_thread": round(done1 / el1, 3),
            "sample": f"{done} single samples of {case.name} (one batch element each, "
                      f"{el:.1f} s, float64 radix-2 FFT + explicit loops, OpenMP); "
                      f"one thread: {done1} samples in {el1:.1f} s"}


def bench_reference(args, rank, world):
    """Reference arm: the float64 oracle on the host cores."""
    if rank != 0:
        return None
    import numpy as np

    import oracle
    from fft_gemm_ifft_gb300 import workloads

    oracle.build()
    case = workloads.CASES[args.workload]
    x_np, w_np = workloads.make_x(case), workloads.make_w(case)
    wc = workloads.as_complex(w_np)
    nthreads = len(os.sched_getaffinity(0))
    oracle.set_threads(nthreads)
    for i in range(min(max(args.warmup, 3), 10)):
        oracle.spectral_conv(x_np[i % case.batch:i % case.batch + 1].astype(np.float64), wc,
                             case.modes)
    budget = 150.0                       # seconds of timed oracle work at most
    t0 = time.perf_counter()
    timed = 0
    for i in range(args.steps):
        b = i % case.batch
        oracle.spectral_conv(x_np[b:b + 1].astype(np.float64), wc, case.modes)
        timed += 1
        el = time.perf_counter() - t0
        if el * (timed + 1) / timed > budget:
            break
    el = time.perf_counter() - t0
    value = timed / el
    sample = (f"each step = one sample (batch element) of {case.name} through the float64 "
              f"oracle; {timed} of {args.steps} steps timed in {el:.1f} s "
              f"(capped at {budget:.0f} s)")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "samples/s",
        "n_gpus": world,
        "steps": timed,
        "warmup": args.warmup,
        "ms_per_step": el * 1e3 / timed,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, same workload as the gb300 arm)",
        "config": {"workload": case.name, "global_batch": case.batch,
                   "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "samples/s",
                         "cores": oracle.get_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "samples/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        # the reference arm is the CPU oracle: rank 0 alone runs and prints
        res = bench_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0:
        from fft_gemm_ifft_gb300 import build
        build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    result, case, x_np, w_np = bench_gpu(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(case, x_np, w_np, args.cpu_seconds)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
