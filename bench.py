"""Benchmark of the FNO spectral-convolution layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload 2d_f16] [--no-per-config]

One step is one forward pass of the layer (truncated forward FFT, per-mode
mixing, inverse FFT) over one batch of the workload, through the C ABI.  The
headline workload is the largest single-GPU one: B=32, C=64, 256x256, 32x32
modes per block, fp16 storage with float32 accumulation (570 MB of
algorithmic traffic per forward).  Inputs are resident in device memory before
the timed region; successive steps rotate through enough distinct (x, w, y)
sets to exceed twice the L2 size, so every step reads and writes HBM.  Steps
are replayed from a CUDA graph (the forward call is capturable) so host launch
overhead does not pace the GPU.  Under torchrun each rank runs its own batch
(weak scaling, replicas: the layer has no exchange step), the timed region is
bracketed by barriers and the slowest rank's time is reported.

The same JSON line carries ``per_config``: every workload (the 1-D, 2-D fp32,
2-D fp16 and 3-D layers and the 2-D FNO stack, the last as one captured
``fno_forward``) timed the same way for about ``--per-config-seconds`` of
device time each, with its own roofline, clocks and the relative L2 error of
one sample against the float64 oracle (checked after the timing, outside it).

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
HEADLINE = "2d_f16"
# every workload, in the order of the per-config record
PER_CONFIG = ("1d_f32", "2d_f32", "2d_f16", "3d_f32", "fno2d_f32")
# plan flags each workload runs with by default (FNO_PLAN_* bits): the 16-bit
# 256x256 layers take their weights packed once into the tensor-core mixing's
# operand images (FNO_PLAN_PACKED_WEIGHTS; weights are parameters)
DEFAULT_FLAGS = {"2d_f16": 128, "2d_bf16": 128}
# relative L2 bars against the float64 oracle
REL_TOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--flags", type=int, default=-1,
                    help="FNO_PLAN_* bits (ablations); default: the workload's own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--per-config-seconds", type=float, default=0.5)
    ap.add_argument("--no-check", action="store_true",
                    help="skip the oracle check of one sample per workload")
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


def kernel_source_digest(sources=None) -> str:
    """Digest of the CUDA sources behind a workload's kernels (the listed
    translation units and every header; all units when none are listed): a
    traffic figure taken from an ncu capture is reported only while those
    kernels are unchanged since that capture."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fft_gemm_ifft_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith(".cuh") or (fn.endswith(".cu") and (sources is None or fn in sources)):
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
        if e.get("source_digest") != kernel_source_digest(e.get("sources")):
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


def e2e_pipelined(torch, conv, case, x_np, ws, stream, steps, world, dev):
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
        import torch.distributed as dist
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


def _rel_l2(got, ref):
    import numpy as np
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(float(np.linalg.norm(ref)), 1e-300))


def _l2_bytes(torch, dev):
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0)) or (126 << 20)


def graph_timing(torch, stream, step, steps, nsets, warmup, world, dev, sample_clocks=True):
    """Time exactly `steps` calls of step(i) replayed from CUDA graphs on
    `stream` (CUDA events on that stream, barriers and a synchronize on both
    sides), after `warmup` eager calls and a 1.5 s pre-heat of the same graph
    during which, and during the timed region, nvidia-smi samples the clocks.
    Returns (ms for the whole timed region, max over ranks; clocks; layout)."""
    steps = max(1, steps)
    per_graph = min(steps, nsets * max(1, 64 // nsets))
    reps, tail = divmod(steps, per_graph)

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                step(i)
        return g

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
        stream.synchronize()
        graph = capture(per_graph)
        graph_tail = capture(tail) if tail else None
        for _ in range(3):
            graph.replay()
        stream.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if sample_clocks:
        sampler.start()
    with torch.cuda.stream(stream):
        t_end = time.time() + 1.5
        while time.time() < t_end:
            graph.replay()
            stream.synchronize()
    if world > 1:
        import torch.distributed as dist
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
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.stop() if sample_clocks else None
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    layout = f"CUDA-graph replay of {per_graph} forwards x {reps} (+{tail})"
    return ms, clocks, layout


def calibrated_steps(torch, stream, step, nsets, seconds):
    """Forwards that fill about `seconds` of device time (one eager pass of
    a few forwards measures the per-forward time first)."""
    n = max(4, nsets)
    with torch.cuda.stream(stream):
        for i in range(n):
            step(i)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    per = max(e0.elapsed_time(e1) / n, 1e-3)          # ms
    return int(min(200000, max(64, seconds * 1e3 / per)))


class LayerSets:
    """One plan, its rotating (x, w, y) sets on the device and the step."""

    def __init__(self, torch, case, flags, dev):
        from fft_gemm_ifft_gb300 import SpectralConv, capi, workloads
        self.case, self.flags = case, flags
        self.conv = SpectralConv(case.n, case.modes, case.batch, case.cin, case.cout,
                                 case.dtype, flags)
        self.x_np, self.w_np = workloads.make_x(case), workloads.make_w(case)
        self.set_bytes = (self.x_np.nbytes + self.w_np.nbytes
                          + math.prod(case.y_shape) * case.elem_bytes)
        self.l2 = _l2_bytes(torch, dev)
        self.nsets = max(2, math.ceil(2 * self.l2 / self.set_bytes))
        self.xs = [workloads.to_torch_storage(self.x_np, case.dtype).to(dev)
                   for _ in range(self.nsets)]
        ws = [workloads.to_torch_storage(self.w_np, case.dtype).to(dev)
              for _ in range(self.nsets)]
        if flags & capi.FNO_PLAN_PACKED_WEIGHTS:
            # weights are parameters: packed once per set, outside the timed region
            ws = [self.conv.pack_weights(w) for w in ws]
        self.ws = ws
        self.ys = [torch.empty(case.y_shape, dtype=self.conv.torch_dtype, device=dev)
                   for _ in range(self.nsets)]
        self.stream = torch.cuda.Stream(device=dev)

    def step(self, i):
        k = i % self.nsets
        self.conv(self.xs[k], self.ws[k], self.ys[k], stream=self.stream)

    def l2_note(self):
        return (f"rotating {self.nsets} distinct (x, w, y) sets = "
                f"{self.nsets * self.set_bytes >> 20} MiB > 2 x L2 ({self.l2 >> 20} MiB)")

    def sample_rel_l2(self, b=0):
        """Parity check of one sample of set 0 (written by the timed replays)
        against the float64 oracle; runs after the timing, outside it."""
        import numpy as np

        import oracle
        from fft_gemm_ifft_gb300 import workloads
        self.stream.synchronize()
        got = self.ys[0][b:b + 1].float().cpu().numpy()
        ref = oracle.spectral_conv(self.x_np[b:b + 1].astype(np.float64),
                                   workloads.as_complex(self.w_np), self.case.modes)
        return _rel_l2(got, ref)

    def close(self):
        self.conv.close()


def roofline_obj(alg_bytes, ms_per_forward, kernel, kernels, traffic):
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (ms_per_forward / 1e3) / 1e9
    return {
        "bound": "hbm",
        "kernel": kernel,
        "kernels_per_forward": kernels,
        "achieved": round(achieved, 1),
        "peak": peak,
        "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
        "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "algorithmic_bytes_per_launch": alg_bytes,
        "traffic": traffic,
    }


def workload_text(case):
    return (f"{case.name}: {case.ndim}-D spectral conv, B={case.batch}, Cin={case.cin}, "
            f"Cout={case.cout}, N={'x'.join(map(str, case.n))}, "
            f"modes={'x'.join(map(str, case.modes))} per block, {case.nblk} block(s), "
            f"{case.dtype} storage")


def layer_record(torch, case, flags, steps, warmup, world, dev, seconds=None):
    """Time one spectral-conv workload; returns (record, LayerSets)."""
    ls = LayerSets(torch, case, flags, dev)
    if seconds is not None:
        steps = calibrated_steps(torch, ls.stream, ls.step, ls.nsets, seconds)
    ms, clocks, layout = graph_timing(torch, ls.stream, ls.step, steps, ls.nsets, warmup,
                                      world, dev)
    assert ls.conv.device_error(ls.stream) == 0
    per = ms / steps
    rec = {
        "value": round(whole_job_rate(case.batch, world, steps, ms), 1),
        "unit": "samples/s",
        "ms_per_step": per,
        "steps": steps,
        "dtype": "f32" if case.dtype == "f32" else f"{case.dtype}-storage/f32-accumulate",
        "workload": workload_text(case),
        "plan_flags": flags,
        "timing": layout + ", CUDA events on the launching stream",
        "l2": ls.l2_note(),
        "roofline": roofline_obj(case.algorithmic_bytes(), per, "fno_spectral_conv_forward",
                                 ls.conv.kernel_count,
                                 recorded_traffic(case.name) if flags == DEFAULT_FLAGS.get(
                                     case.name, 0) else None),
        "clocks": clocks,
    }
    return rec, ls


def fno_record(torch, steps, warmup, world, dev, seconds=None, check=True):
    """The FNO stack (fno_forward), replayed from a CUDA graph."""
    import numpy as np

    from fft_gemm_ifft_gb300 import FnoModel, workloads
    case = workloads.FNO_CASE
    m = FnoModel(case.batch, case.h, case.w, case.modes, case.cin_lift, case.width,
                 case.nlayers, case.hidden, case.cout)
    fx = workloads.make_fno_inputs(case)
    fp = workloads.make_fno_params(case)
    nsets = 2
    xs = [torch.from_numpy(fx).to(dev) for _ in range(nsets)]
    p = {k: torch.from_numpy(v).to(dev) for k, v in fp.items()}
    ys = [torch.empty(m.y_shape, dtype=torch.float32, device=dev) for _ in range(nsets)]
    stream = torch.cuda.Stream(device=dev)
    step = lambda i: m(xs[i % nsets], p, ys[i % nsets], stream=stream)
    if seconds is not None:
        steps = calibrated_steps(torch, stream, step, nsets, seconds)
    ms, clocks, layout = graph_timing(torch, stream, step, steps, nsets, warmup, world, dev)
    assert m.device_error(stream) == 0
    per = ms / steps
    rec = {
        "value": round(whole_job_rate(case.batch, world, steps, ms), 1),
        "unit": "samples/s",
        "ms_per_step": per,
        "steps": steps,
        "dtype": "f32",
        "workload": (f"{case.name}: 2-D FNO forward, B={case.batch}, lift {case.cin_lift}->"
                     f"{case.width}, {case.nlayers} layers (spectral conv modes "
                     f"{case.modes[0]}x{case.modes[1]} x 2 blocks + 1x1 linear, GELU), head "
                     f"{case.width}->{case.hidden}->{case.cout}, {case.h}x{case.w}"),
        "timing": layout + " (fno_forward captured whole), CUDA events on the launching stream",
        "l2": "each forward streams its 64-channel activations (64 MiB each) through HBM",
        "roofline": roofline_obj(case.algorithmic_bytes(), per, "fno_forward", m.kernel_count,
                                 None),
        "clocks": clocks,
    }
    if check:
        import oracle
        stream.synchronize()
        got = ys[0][0:1].cpu().numpy()
        ref = oracle.fno_forward(fx[0:1], workloads.fno_params_for_oracle(fp), case.modes)
        rec["rel_l2_sample"] = _rel_l2(got, ref)
        rec["rel_l2_tol"] = 1e-5
    m.close()
    return rec


def bench_gpu(args, rank, world, local):
    import torch

    from fft_gemm_ifft_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = workloads.CASES[args.workload]
    flags = DEFAULT_FLAGS.get(case.name, 0) if args.flags < 0 else args.flags
    rec, ls = layer_record(torch, case, flags, args.steps, args.warmup, world, dev)
    conv, stream = ls.conv, ls.stream
    steps = max(1, args.steps)

    # L2-resident ("hot") figure for workloads whose set fits in L2: the same
    # forwards on one (x, w, y) set, reported beside the rotated value
    hot_ms = None
    if ls.set_bytes < ls.l2:
        hot = lambda i: conv(ls.xs[0], ls.ws[0], ls.ys[0], stream=stream)
        ms_hot, _, _ = graph_timing(torch, stream, hot, steps, ls.nsets, 3, world, dev,
                                    sample_clocks=False)
        hot_ms = ms_hot / steps

    # end to end through the public API: every step copies its input from pinned
    # host memory, runs the layer and copies its output back to pinned host
    # memory.  The steps are pipelined over three device buffer slots and three
    # streams (copy in, layer, copy out), as a serving loop would run them: the
    # input of step i+1 and the output of step i-1 move while step i computes.
    e2e_steps = max(3, args.e2e_steps)
    e2e_ms = e2e_pipelined(torch, conv, case, ls.x_np, ls.ws, stream, e2e_steps, world, dev)
    parity = None
    if rank == 0 and not args.no_check:
        parity = {"rel_l2_sample": ls.sample_rel_l2(0), "rel_l2_tol": REL_TOL[case.dtype],
                  "sample": "batch element 0 of set 0 against the float64 oracle"}
    result = {
        "metric": METRIC,
        "value": rec["value"],
        "unit": "samples/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": rec["dtype"],
        "data": "synthetic (seeded N(0,1) fields, U[0,1)/(Cin*Cout) complex weights)",
        "config": {
            "workload": rec["workload"],
            "global_batch": world * case.batch,
            "parallelism": f"replicas x{world}",
            "l2": rec["l2"],
            "timing": rec["timing"],
            "plan_flags": flags,
            "weights": ("packed once per set into the mixing kernel's operand layout, "
                        "outside the timed region (weights are parameters)"
                        if flags & 128 else "as given (nblk, Cin, Cout, modes)"),
            "hot_l2_ms_per_step": hot_ms,
        },
        "roofline": rec["roofline"],
        "e2e": {
            "value": round(whole_job_rate(case.batch, world, e2e_steps, e2e_ms), 1),
            "unit": "samples/s",
            "h2d_bytes_per_step": int(math.prod(case.x_shape) * case.elem_bytes),
            "pipelining": "3 buffer slots; input copy, layer and output copy on separate streams",
            "d2h_bytes_per_step": int(math.prod(case.y_shape) * case.elem_bytes),
        },
        "gpu_launches": steps * conv.kernel_count,
        "clocks": rec["clocks"],
    }
    if parity is not None:
        result["parity"] = parity
    x_np, w_np = ls.x_np, ls.w_np
    ls.close()
    del ls
    torch.cuda.empty_cache()

    if not args.no_per_config:
        per = {}
        for name in PER_CONFIG:
            if name == case.name:
                r = dict(rec)
                if parity is not None:
                    r.update(parity)
                per[name] = r
                continue
            if name == workloads.FNO_CASE.name:
                per[name] = fno_record(torch, 0, 3, world, dev, args.per_config_seconds,
                                       check=rank == 0 and not args.no_check)
            else:
                c = workloads.CASES[name]
                r, lsc = layer_record(torch, c, DEFAULT_FLAGS.get(name, 0), 0, 3, world, dev,
                                      args.per_config_seconds)
                if rank == 0 and not args.no_check:
                    r["rel_l2_sample"] = lsc.sample_rel_l2(0)
                    r["rel_l2_tol"] = REL_TOL[c.dtype]
                lsc.close()
                del lsc
                torch.cuda.empty_cache()
                per[name] = r
        result["per_config"] = per
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
