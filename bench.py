#!/usr/bin/env python3
"""Benchmark of the forward 2-D convolution on one or more GB300 GPUs.

One step = one conv2d_fwd call over a full batch of the workload: argument
checks, filter repack, input transform (window tensor or channels-last copy,
per the chosen algorithm), the contraction kernel and its epilogue.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--dtype DT]
                  [--algo A] [--impl reference]

Prints ONE JSON line (rank 0).  Default workload: the VGG-style layer
(N=64, Cin=512, 28x28, Cout=512, 3x3, stride 1, pad 1; the largest of the
workloads and a compute-bound 3x3 layer) in fp16 with fp32 accumulation.  Timing: CUDA events on the launching stream around the whole
run of K back-to-back steps (per-step event pairs are snapped to a ~2 us
completion tick on this platform and would bias short steps), each step on
the next of several rotating input/filter/output/workspace sets whose total
exceeds the 129 MB L2 (a step never finds its operands in L2 from an earlier
step); W untimed warm-up steps; barrier + synchronize around the timed
region; max over ranks.  Multi-GPU runs are independent batches per rank
(weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "conv fwd TFLOP/s (2*N*Cout*Ho*Wo*Cin*Kh*Kw/t), % of roofline, workspace MB"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20
# DRAM bytes (read + write) per launch of the contraction kernel, from ncu
# captures (launch lists where there is one, else the full capture; writes
# that stay in L2 during a replay read as 0); null for workloads without such
# a capture.  All from the current kernels, one full-size launch each.
NCU_TRAFFIC_BYTES = {
    ("resnet_stage1", "f16", "padded_tc"): 14.39e6,
    ("vgg", "f16", "implicit_tc"): 64.85e6,
    ("sweep_k1", "f16", "implicit_tc"): 16.85e6,
    ("sweep_k3", "f16", "padded_tc"): 18.75e6,
    ("stem", "f16", "im2win_tc"): 40.57e6,
}
ROTATION_BYTES = 3 * L2_BYTES         # rotating sets: together at least three L2s


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


def fp32_alu_peak_tflops(sm_count: int, mhz: float) -> float:
    """FFMA peak: SMs x 128 fp32 lanes x 2 FLOP x clock."""
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def cpu_oracle_baseline(wl, dtype, budget_s=12.0, threads=None, inputs=None):
    """Time the fp64 oracle (as it stands) on host threads over a bounded
    sample of the workload: whole (n, co) output planes taken in order,
    enough of them for about ``budget_s`` seconds (the whole batch at most).
    Returns a cpu_baseline dict in TFLOP/s."""
    import concurrent.futures as cf
    from oracle import ref
    threads = threads or (os.cpu_count() or 1)
    d = inputs if inputs is not None else synth.make_inputs(wl, dtype)
    X64, W64 = d["X64"], d["W64"]
    N = X64.shape[0]
    Ho, Wo = wl.out_hw()
    Y = np.empty((N, wl.Co, Ho, Wo))
    S = np.empty_like(Y)
    plane_flops = 2 * Ho * Wo * wl.Ci * wl.Kh * wl.Kw
    t0 = time.perf_counter()
    ref.conv2d_slice(X64, W64, Y, S, wl.stride, wl.pad, 0, 1, 0, 1)
    t_plane = max(time.perf_counter() - t0, 1e-6)
    planes = int(min(N * wl.Co, max(1, budget_s * threads / t_plane)))
    jobs = [(i // wl.Co, i % wl.Co) for i in range(planes)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda j: ref.conv2d_slice(X64, W64, Y, S, wl.stride, wl.pad, j[0], j[0] + 1, j[1], j[1] + 1),
                    jobs))
    dt = time.perf_counter() - t0
    flops = planes * plane_flops
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{planes} of {N * wl.Co} output planes (n, co in order) of {wl.name}, "
                      f"{flops / 1e9:.2f} GFLOP in {dt:.2f} s, fp64 7-loop on {threads} threads"}


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest of every rank's x (one all-reduce; identity on one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's independent batch over the slowest rank's time."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def _workload(args):
    wl = synth.WORKLOADS[args.workload]
    if args.batch:
        # Profiling aid: the same layer at a smaller batch (never the default).
        wl = wl.scaled(N=args.batch, name=f"{wl.name}_n{args.batch}")
    # fp16 where the workload has it (the dtype of the tensor-peak target), else its first dtype.
    dtype = args.dtype or ("f16" if "f16" in wl.dtypes else wl.dtypes[0])
    return wl, dtype


def run_reference(args, rank, world):
    """Reference arm: the oracle on the host cores, a bounded sample per step."""
    wl, dtype = _workload(args)
    if rank != 0:
        return
    # Each step times a bounded sample; the whole run stays within ~2 minutes.
    per_step = min(3.0, 120.0 / (args.steps + args.warmup))
    inputs = synth.make_inputs(wl, dtype)
    for _ in range(args.warmup):
        cpu_oracle_baseline(wl, dtype, budget_s=per_step / 4, inputs=inputs)
    samples = [cpu_oracle_baseline(wl, dtype, budget_s=per_step, inputs=inputs) for _ in range(args.steps)]
    vals = [s["value"] for s in samples]
    v = statistics.median(vals)
    step_ms = wl.flops() / (v * 1e12) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "N": wl.N, "Cin": wl.Ci, "H": wl.H, "W": wl.W, "Cout": wl.Co,
                       "Kh": wl.Kh, "Kw": wl.Kw, "stride": wl.stride, "pad": wl.pad, "input_dtype": dtype},
            "cpu_baseline": {**samples[0], "value": v},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist
    from dense_convolution_gb300 import build, capi
    from dense_convolution_gb300.conv import Conv2d

    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    wl, dtype = _workload(args)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]

    d = synth.make_inputs(wl, dtype)
    xh = (torch.from_numpy(d["X"]) if dtype != "bf16" else d["X"]).contiguous().pin_memory()
    wh = (torch.from_numpy(d["W"]) if dtype != "bf16" else d["W"]).contiguous().pin_memory()
    tuning = {}
    for kv in filter(None, args.tune.split(",")):
        k, v = kv.split("=")
        tuning[k.strip()] = int(v)
    op = Conv2d(wl.N, wl.Ci, wl.H, wl.W, wl.Co, wl.Kh, wl.Kw, wl.stride, wl.pad, dtype, args.algo, tuning=tuning)
    # Rotating operand sets (X, W, Y, workspace), together >= 3 x L2.
    x0 = xh.to(dev)
    w0 = wh.to(dev)
    set_bytes = (x0.numel() * x0.element_size() + w0.numel() * w0.element_size() +
                 int(np.prod(op.out_shape)) * x0.element_size() + op.workspace_bytes)
    # A multiple of three, so that the streamed end-to-end pass below can give
    # each of its three streams sets of its own.
    n_sets = int(min(18, max(3, -(-ROTATION_BYTES // set_bytes))))
    n_sets = -(-n_sets // 3) * 3
    sets = []
    for i in range(n_sets):
        xi = x0 if i == 0 else x0.clone()
        wi = w0 if i == 0 else w0.clone()
        sets.append((xi, wi, op.alloc_output(dev), op.alloc_workspace(dev)))
    x, w, y, ws = sets[0]
    yh = torch.empty(y.shape, dtype=tdt, pin_memory=True)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    launches = capi.conv2d_launches_per_call(op.desc)

    def step(i=0, ev0=None, ev1=None):
        xi, wi, yi, wsi = sets[i % n_sets]
        if ev0 is None:
            capi.conv2d_fwd(op.desc, xi.data_ptr(), wi.data_ptr(), yi.data_ptr(), wsi.data_ptr(), wsi.numel(), sp)
        else:
            capi.conv2d_fwd_profiled(op.desc, xi.data_ptr(), wi.data_ptr(), yi.data_ptr(), wsi.data_ptr(),
                                     wsi.numel(), sp, ev0.cuda_event, ev1.cuda_event)

    for i in range(max(3, args.warmup, n_sets)):
        step(i)
    torch.cuda.synchronize()
    assert capi.conv2d_device_status(sp) == 0

    K = args.steps
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in kev:          # materialise the raw events before handing them to the library
        a.record(stream)
        b.record(stream)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # Headline: K plain calls back to back on rotating sets, one event
        # pair around all of them (the library's kernels overlap each other
        # within and across calls through programmatic dependent launch;
        # nothing is inserted between them).
        ev[0].record(stream)
        for i in range(K):
            step(i)
        ev[1].record(stream)
        torch.cuda.synchronize()
        # Roofline: the same K calls again, with the contraction kernel
        # bracketed by events recorded on the launch stream by the library.
        for i in range(K):
            step(i, *kev[i])
        torch.cuda.synchronize()
        # Keep the GPU busy long enough for the clock sampler to see the load.
        t_end = time.perf_counter() + (0.0 if args.quick else 0.4)
        while time.perf_counter() < t_end:
            for i in range(20):
                step(i)
            torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    assert capi.conv2d_device_status(sp) == 0
    ms = ev[0].elapsed_time(ev[1]) / K
    kms = sum(kern_ms) / K
    if launches == 1:
        # The call is the contraction kernel alone: the headline loop is K of
        # its launches back to back on this stream, so its event pair gives the
        # kernel's average duration without the per-launch events' own cost.
        kms = ms
    # A kernel cannot take longer than the whole call it is part of: a higher
    # per-launch reading is the events' own cost or a clock drop between the
    # two passes (seen under the power cap on the longest layers).
    kms = min(kms, ms)
    ms = max_over_ranks(ms, world, dev)

    # End to end through the C ABI on host buffers (conv2d_fwd_host): pinned
    # host X and W copied in, the call, Y copied out, every step, on one stream.
    def fwd_host(i, st, y_host=None):
        xi, wi, yi, wsi = sets[i]
        capi.conv2d_fwd_host(op.desc, xh.data_ptr(), wh.data_ptr(), (yh if y_host is None else y_host).data_ptr(),
                             xi.data_ptr(), wi.data_ptr(), yi.data_ptr(), wsi.data_ptr(), wsi.numel(), st)

    e2e_ms = []
    for i in range(3 if args.quick else max(3, min(K, 50))):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.fill_(1)
        e0.record(stream)
        fwd_host(0, sp)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_serial = sum(e2e_ms[1:]) / max(1, len(e2e_ms) - 1)
    e2e_serial = max_over_ranks(e2e_serial, world, dev)

    # The same calls streamed as a caller feeding batches would: round-robin
    # over three streams, each with operand sets of its own, so that one call's
    # copies overlap other calls' compute.  Every call still copies its X and W
    # in and its Y out.
    def e2e_pipelined(nsteps):
        streams = [torch.cuda.Stream(dev) for _ in range(3)]
        y_hosts = [yh] + [torch.empty(y.shape, dtype=tdt, pin_memory=True) for _ in range(2)]   # one per stream
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for s_ in streams:
            s_.wait_event(t0)
        for i in range(nsteps):
            k = i % 3
            fwd_host(k + 3 * ((i // 3) % (n_sets // 3)), streams[k].cuda_stream, y_hosts[k])
        for s_ in streams:
            ev = torch.cuda.Event()
            ev.record(s_)
            stream.wait_event(ev)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / nsteps

    n_pipe = 6 if args.quick else max(6, min(K, 100))
    e2e_pipelined(min(n_pipe, 6))                        # warm-up
    e2e = max_over_ranks(e2e_pipelined(n_pipe), world, dev)

    # The bound of that mode: the same pinned-host copies (X and W in, Y out)
    # on the same three streams, with no convolution in between.
    def copies_only(nsteps):
        streams = [torch.cuda.Stream(dev) for _ in range(3)]
        y_hosts = [torch.empty(y.shape, dtype=tdt, pin_memory=True) for _ in range(3)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for s_ in streams:
            s_.wait_event(t0)
        for i in range(nsteps):
            k = i % 3
            xi, wi, yi, _ = sets[k + 3 * ((i // 3) % (n_sets // 3))]
            with torch.cuda.stream(streams[k]):
                xi.copy_(xh, non_blocking=True)
                wi.copy_(wh, non_blocking=True)
                y_hosts[k].copy_(yi, non_blocking=True)
        for s_ in streams:
            ev = torch.cuda.Event()
            ev.record(s_)
            stream.wait_event(ev)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / nsteps

    copies_only(min(n_pipe, 6))
    copy_ms = max_over_ranks(copies_only(n_pipe), world, dev)
    assert capi.conv2d_device_status(sp) == 0

    flops = wl.flops()
    value = job_tflops(flops, world, ms)
    peaks, src = _peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    elem = 4 if dtype == "f32" else 2
    Ho, Wo = wl.out_hw()
    # Algorithmic bytes: X, W and Y once each at their dtypes.
    alg_bytes = (wl.N * wl.Ci * wl.H * wl.W + wl.Co * wl.Ci * wl.Kh * wl.Kw + wl.N * wl.Co * Ho * Wo) * elem
    if dtype == "f32":
        cpeak = fp32_alu_peak_tflops(sm_count, peaks.get("sm_max_mhz", 2070.0))
        cbound, csrc = "alu", "derived: SMs x 128 FFMA lanes x 2 x max SM clock"
    else:
        cpeak = peaks["bf16_tflops"]
        cbound, csrc = "tensor", f"{src} bf16 dense burst (fp16 rate equal)"
    # Roofline: a layer whose arithmetic intensity (FLOP per algorithmic byte)
    # is below the ridge (compute peak / measured HBM copy bandwidth) is
    # reported against HBM with its algorithmic bytes, else against compute.
    hbm = peaks["hbm_gbs"]
    intensity = flops / alg_bytes
    if intensity < cpeak * 1e12 / (hbm * 1e9):
        bound, peak, unit, psrc = "hbm", hbm, "GB/s", f"{src} HBM copy bandwidth"
        achieved = alg_bytes / (kms * 1e-3) / 1e9
        step_frac = alg_bytes / (ms * 1e-3) / 1e9 / peak
    else:
        bound, peak, unit, psrc = cbound, cpeak, "TFLOP/s", csrc
        achieved = flops / (kms * 1e-3) / 1e12
        step_frac = (flops / (ms * 1e-3) / 1e12) / peak
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {"workload": wl.name, "N": wl.N, "Cin": wl.Ci, "H": wl.H, "W": wl.W, "Cout": wl.Co,
                   "Kh": wl.Kh, "Kw": wl.Kw, "stride": wl.stride, "pad": wl.pad, "algo": op.algo,
                   "accumulate": "f32",
                   "l2": f"{n_sets} rotating X/W/Y/workspace sets, {n_sets * set_bytes / 2 ** 20:.0f} MB > 129 MB L2; "
                         "no flush inside the timed region",
                   "workspace_mb": op.workspace_bytes / 2 ** 20,
                   "tuning": tuning or "automatic",
                   "im2win_tensor_mb": wl.N * wl.Ci * Ho * (wl.W + 2 * wl.pad) * wl.Kh * elem / 2 ** 20,
                   "parallelism": f"independent batch per GPU x{world}"},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": NCU_TRAFFIC_BYTES.get((wl.name, dtype, op.algo)),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)", "kernel": "contraction kernel",
                     "kernel_ms": kms, "peak_source": psrc,
                     "step_frac": step_frac, "intensity_flop_per_byte": intensity,
                     "algorithmic_bytes": alg_bytes},
        "gpu_launches": launches * K,
        "e2e": {"value": job_tflops(flops, world, e2e), "unit": "TFLOP/s",
                "h2d_bytes_per_step": xh.numel() * xh.element_size() + wh.numel() * wh.element_size(),
                "d2h_bytes_per_step": yh.numel() * yh.element_size(), "ms_per_step": e2e,
                "mode": "conv2d_fwd_host calls round-robin on three streams (copies of one call overlap others' compute)",
                "serial_ms_per_step": e2e_serial,
                "copy_bound_ms_per_step": copy_ms,
                "copy_bound": "the same pinned host<->device copies on the same three streams, no convolution",
                "link_gbs": (xh.numel() * xh.element_size() + wh.numel() * wh.element_size()
                             + yh.numel() * yh.element_size()) / (copy_ms * 1e-3) / 1e9},
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.quick):
        line["cpu_baseline"] = cpu_oracle_baseline(wl, dtype, inputs=d)
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="vgg", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--dtype", default=None, choices=list(synth.DTYPES))
    ap.add_argument("--algo", default="auto")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=0, help="profiling runs: override the workload's batch size")
    ap.add_argument("--tune", default="",
                    help="pipeline knobs for ablations, e.g. stages=1,sync_copies=1,raster=2,no_resident=1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no CPU baseline, 3 end-to-end steps, no clock-sustain loop")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        # One process per GPU: N GPUs need N ranks from the launcher.
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N ranks with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.impl != "reference":
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
