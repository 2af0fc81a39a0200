#!/usr/bin/env python3
"""Benchmark of the sm_103a dense HGEMM: HGEMM TFLOP/s at M=N=K=4096,
fp16 inputs, fp32 accumulate and output (row-major A, B, D; alpha=1,
beta=0), reported against the measured tensor-core peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the CPU oracle on a bounded sample

One step = one gemm_run over the workload (one launch of the persistent
kernel), inputs resident in HBM.  L2 is flushed before every step by writing
a 256 MiB buffer (outside the timed interval of the step); every step's GEMM
is timed with CUDA events on the launching stream, and the timed loop as a
whole is bracketed by a barrier and torch.cuda.synchronize().  With N > 1
(torchrun, one process per GPU) every rank runs an independent replica of
the same workload (a single GEMM of this size does not need to be sharded);
value = the flops of all ranks / the slowest rank's time.

The roofline object is that of the step's one kernel: the longer of the
tensor-pipe bound (2*M*N*K at the measured dense peak) and the HBM bound
(|A| + |B| (+ |C|) + |D| at the measured copy bandwidth) is `bound` (the
skinny and ragged shapes are reported in GB/s, the square ones in
TFLOP/s), the other one follows as `other_bound`.

Prints one JSON line (rank 0).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HGEMM TFLOP/s at M=N=K=4096 fp16→fp32 acc; % of GB300 dense FP16 tensor peak"
NOMINAL_DENSE_FP16_TFLOPS = 2250.0       # GB300 dense fp16/bf16 tensor peak (datasheet)
# datasheet dense rates of the other operand kinds relative to fp16/bf16
# (fp8 4.5 PFLOP/s, tf32 1.1 PFLOP/s): the measured bf16 peak times this
# ratio is the roofline peak of a kind with no measurement of its own
NOMINAL_RATIO = {"f16": 1.0, "bf16": 1.0, "e4m3": 2.0, "e5m2": 2.0, "tf32": 1100.0 / 2250.0}
FALLBACK_BF16_TFLOPS = 1900.0            # used only when no measured peak file is present
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sq4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--flush", choices=["write", "write_read", "none"], default="write_read",
                    help="L2 hygiene between steps: write a 256 MiB buffer (leaves it dirty in L2), "
                         "write then read it back (L2 left clean, holding none of the inputs), or none")
    # overrides of the workload (exploration; the JSON config records the result)
    ap.add_argument("--M", type=int)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    ap.add_argument("--layoutA", choices=["row", "col"])
    ap.add_argument("--layoutB", choices=["row", "col"])
    ap.add_argument("--accum", choices=["f32", "f16"])
    ap.add_argument("--out", choices=["f32", "f16", "bf16"])
    ap.add_argument("--epilogue", choices=["none", "bias", "bias_relu", "bias_gelu", "scale_bias_gelu"],
                    default="none", help="fused epilogue timed with the GEMM (random fp32 vectors)")
    ap.add_argument("--prior-art", choices=["wmma_naive", "wmma_shared", "mma_sync"],
                    help="time one of the pages' own warp-level kernels instead (fp16 row-major A and B; "
                         "comparison only)")
    ap.add_argument("--division", choices=["auto", "whole", "split", "early_split", "halves", "stream_k",
                                           "pair_split"],
                    default="auto", help="pin how the last wave's tiles are divided (gemm_plan_force_division)")
    ap.add_argument("--config", choices=["auto", "single_128x16", "single_128x64", "single_128x256", "pair_256x256",
                                         "pair_256x224"],
                    default="auto", help="pin the kernel configuration (gemm_plan_force_config)")
    ap.add_argument("--autotune", action="store_true",
                    help="time every candidate configuration first (gemm_plan_autotune) and run the fastest")
    return ap.parse_args()


def select_workload(args):
    import dataclasses
    import workloads as wl
    w = wl.WORKLOADS[args.workload]
    over = {k: v for k, v in (("M", args.M), ("N", args.N), ("K", args.K), ("layoutA", args.layoutA),
                              ("layoutB", args.layoutB), ("accum_dtype", args.accum),
                              ("out_dtype", args.out)) if v is not None}
    if over:
        w = dataclasses.replace(w, name=w.name + "+" + ",".join(f"{k}={v}" for k, v in over.items()), **over)
    return w


def job_throughput(local_total_ms: float, flops_per_step: float, steps: int, world: int, dist=None,
                   device=None) -> tuple[float, float]:
    """(slowest rank's total ms, whole-job TFLOP/s): every rank runs `steps`
    steps of its own replica; the job's time is the maximum over ranks and
    its work the steps of all ranks."""
    total_ms = float(local_total_ms)
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([total_ms], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, flops_per_step * steps * world / (total_ms * 1e-3) / 1e12


def metric_for(w) -> str:
    """The headline metric for its own workload; a plain description for the others."""
    if w.name == "sq4096":
        return METRIC
    return (f"GEMM TFLOP/s at M={w.M} N={w.N} K={w.K} {w.in_dtype}->{w.accum_dtype} acc->{w.out_dtype} "
            f"(2*M*N*K per step)")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def workload_desc(w) -> str:
    return (f"{w.name}: M={w.M} N={w.N} K={w.K}; A {w.in_dtype} {w.layoutA}-major, B {w.in_dtype} "
            f"{w.layoutB}-major, {w.dist}; {w.accum_dtype} accumulate, {w.out_dtype} row-major out; "
            f"alpha={w.alpha} beta={w.beta}")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None,
            "samples": len(sm),
            "reasons": sorted(reasons),
        }


def cpu_baseline(w, h, target_s: float = 12.0):
    """The oracle, as it stands, on the host cores: a bounded sample of the
    workload (whole rows of D), in the metric's unit."""
    import oracle
    import workloads as wl
    cores = os.cpu_count() or 1
    A, B = wl.bits(h.A), wl.bits(h.B)
    C = None if h.C is None else wl.bits(h.C)
    rows = max(cores, 8)
    # calibrate on a small slice, then size the sample to ~target_s
    t0 = time.perf_counter()
    oracle.gemm(w.in_dtype, A, B, C, min(rows, w.M), w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                w.out_dtype, w.alpha, w.beta, nthreads=cores)
    dt = time.perf_counter() - t0
    rows = int(min(w.M, max(rows, rows * target_s / max(dt, 1e-3))))
    rows = max(cores, rows // cores * cores)
    t0 = time.perf_counter()
    oracle.gemm(w.in_dtype, A, B, C, rows, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                w.out_dtype, w.alpha, w.beta, nthreads=cores)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    # the same triple loop on one thread, on a slice that takes about a fifth of the time
    r1 = max(1, min(w.M, int(rows / cores * 0.2)))
    t1 = time.perf_counter()
    oracle.gemm(w.in_dtype, A, B, C, r1, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                w.out_dtype, w.alpha, w.beta, nthreads=1)
    d1 = time.perf_counter() - t1
    f1 = 2.0 * r1 * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} rows of D ({rows}x{w.N}x{w.K}, {flops:.3g} flop) in {dt:.2f} s "
                      f"on {cores} threads",
            "single_thread": {"value": f1 / d1 / 1e12, "unit": "TFLOP/s",
                              "sample": f"first {r1} rows of D ({f1:.3g} flop) in {d1:.2f} s on 1 thread"}}


def kernel_sources_hash() -> str:
    """Hash of the sources the GEMM kernels are compiled from (the kernel, its
    PTX wrappers, the launch code and the per-configuration units)."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "tensor_core_dense_tma_gb300", "csrc")
    files = [os.path.join(csrc, n) for n in ("gemm_kernel.cuh", "ptx_sm103.cuh", "gemm_internal.cuh")]
    files += sorted(glob.glob(os.path.join(csrc, "gemm_cfg_*.cu")))
    hsh = hashlib.sha256()
    for fn in files:
        with open(fn, "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()[:16]


def traffic_from_profiles(workload: str, kernel_tag: str):
    """Per-launch DRAM bytes of this workload's kernel from the committed ncu
    summaries, if they were taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            kv = dict(line.strip().split("=", 1) for line in f if "=" in line and not line.startswith("#"))
    except OSError:
        return None
    if kv.get("sources_sha256") != kernel_sources_hash():
        return None
    val = kv.get(f"{workload}.{kernel_tag}.bytes_per_launch")
    return float(val) if val else None


def rooflines(w, avg_s: float, tensor_peak: float, hbm_peak: float, traffic, peak_src: str,
              ratio: float) -> dict:
    """The roofline of the step's one kernel.  Two bounds apply to a GEMM:
    the tensor pipe (2*M*N*K flop at the measured dense peak) and HBM (the
    algorithmic bytes |A| + |B| (+ |C|) + |D|, each moved once, at the
    measured copy bandwidth).  The one that takes longer is the roofline
    reported (`bound`); the other follows under `other_bound`, so shapes
    below the ridge (skinny, ragged) are reported in GB/s and the square
    ones in TFLOP/s."""
    flops = float(w.flops)
    nbytes = float(w.algorithmic_bytes())
    t_flop = flops / (tensor_peak * 1e12)
    t_byte = nbytes / (hbm_peak * 1e9)
    src = "measured" if peak_src == "measured" else "fallback"
    tensor = {"bound": "tensor", "achieved": flops / avg_s / 1e12, "peak": tensor_peak, "unit": "TFLOP/s",
              "frac": t_flop / avg_s, "traffic": traffic,
              "peak_source": (f"{src} bf16 dense GEMM burst (MEASURED_PEAKS.json)" if src == "measured"
                              else "fallback 1.9 PFLOP/s bf16 burst")
                             + (", fp16:bf16 = 1:1" if ratio == 1.0 else
                                f", x {ratio:.3g} = the datasheet ratio of {w.in_dtype} to bf16 dense rates"),
              "algorithmic": f"2*M*N*K = {flops:.4g} flop per launch"}
    hbm = {"bound": "hbm", "achieved": nbytes / avg_s / 1e9, "peak": hbm_peak, "unit": "GB/s",
           "frac": t_byte / avg_s, "traffic": traffic,
           "peak_source": (f"{src} HBM copy bandwidth (MEASURED_PEAKS.json, read + write bytes)"
                           if src == "measured" else "fallback 6.8 TB/s copy"),
           "pct_of_nominal_7900_gbs": 100.0 * nbytes / avg_s / 7.9e12,
           "algorithmic": f"|A|+|B|{'+|C|' if w.beta != 0.0 else ''}+|D| = {nbytes:.6g} bytes per launch"}
    primary, other = (hbm, tensor) if t_byte > t_flop else (tensor, hbm)
    primary["other_bound"] = other
    primary["arithmetic_intensity_flop_per_byte"] = flops / nbytes
    primary["ridge_flop_per_byte"] = tensor_peak * 1e12 / (hbm_peak * 1e9)
    primary["bound_us"] = max(t_flop, t_byte) * 1e6
    return primary


def run_reference(args):
    """The CPU oracle on the host cores, each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import workloads as wl
    w = select_workload(args)
    h = wl.make_inputs(w)
    cores = os.cpu_count() or 1
    A, B = wl.bits(h.A), wl.bits(h.B)
    C = None if h.C is None else wl.bits(h.C)
    rows = cores   # one row per core per step: a few seconds per step
    for _ in range(args.warmup):
        oracle.gemm(w.in_dtype, A, B, C, rows, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                    w.out_dtype, w.alpha, w.beta, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm(w.in_dtype, A, B, C, rows, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                    w.out_dtype, w.alpha, w.beta, nthreads=cores)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    val = flops / dt / 1e12
    out = {
        "impl": "reference", "metric": metric_for(w), "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(w), "sample": f"{rows} rows of D per step"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows}x{w.N}x{w.K} per step (rows of D), {args.steps} steps"},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


def main():
    args = parse()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("bad --steps/--warmup")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import tensor_core_dense_tma_gb300 as tc
    import workloads as wl
    from tensor_core_dense_tma_gb300 import build as tcbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if not tcbuild.up_to_date():
        if rank == 0:
            tcbuild.build()
        if dist:
            dist.barrier()

    w = select_workload(args)
    h = wl.make_inputs(w)
    A = h.A.to(dev)
    B = h.B.to(dev)
    C = None if h.C is None else h.C.to(dev)
    D = torch.empty((w.M, h.ldc), dtype=wl.DTYPES[w.out_dtype], device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(i):
        if args.flush == "none":
            return
        flush.fill_(float(i))                 # evicts everything else from L2 ...
        if args.flush == "write_read":
            torch.sum(flush, dim=0, out=flush_sink)  # ... and leaves it clean (written back, re-read)
    plan = tc.Plan(w.in_dtype, local)
    A_l = wl.logical(A, w.M, w.K, w.layoutA)
    B_l = wl.logical(B, w.K, w.N, w.layoutB)
    C_l = None if C is None else C[:, :w.N]
    D_l = D[:, :w.N]
    stream = torch.cuda.current_stream(dev)
    ep = {}
    if args.epilogue != "none":
        g = torch.Generator(device="cpu").manual_seed(4242)
        if "bias" in args.epilogue:
            ep["bias"] = torch.randn(w.N, generator=g).to(dev)
        if "scale" in args.epilogue:
            ep["row_scale"] = (0.5 + torch.rand(w.M, generator=g)).to(dev)
            ep["col_scale"] = (0.5 + torch.rand(w.N, generator=g)).to(dev)
        for a in ("relu", "gelu"):
            if a in args.epilogue:
                ep["act"] = a

    def step():
        if args.prior_art:
            tc.run_prior_art(args.prior_art, A_l, B_l, D_l, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype,
                             stream=stream.cuda_stream)
            return
        plan.gemm(A_l, B_l, C_l, D_l, alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype,
                  out_dtype=w.out_dtype, stream=stream.cuda_stream, **ep)

    if args.config != "auto":
        plan.force_config(args.config)
    if args.division != "auto":
        plan.force_division(args.division)
    tuning = None
    if args.autotune:
        _, rows = plan.autotune(A_l, B_l, C_l, D_l, alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype,
                                out_dtype=w.out_dtype, reps=5, stream=stream.cuda_stream)
        tuning = {"candidates": len(rows), "chosen": next(r["config"] for r in rows if r["chosen"]),
                  "model": next(r["config"] for r in rows if r["model"]),
                  "chosen_us": min(r["us"] for r in rows),
                  "model_us": next(r["us"] for r in rows if r["model"])}

    for i in range(args.warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if os.environ.get("CUDA_VISIBLE_DEVICES") is None else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = plan.launches
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(i)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    launches = args.steps if args.prior_art else plan.launches - launches0
    clocks = sampler.stop() if rank == 0 else None
    assert plan.device_status() == 0, "device status word reports an error"

    per_step = [s.elapsed_time(e) for s, e in zip(starts, ends)]   # ms
    total_ms, value = job_throughput(sum(per_step), w.flops, args.steps, world, dist, dev)
    ms_per_step = total_ms / args.steps

    # end to end through the public API with host buffers (pinned), copies timed
    e2e = None
    if not args.no_e2e and not args.prior_art:
        hA = h.A.pin_memory()
        hB = h.B.pin_memory()
        hC = None if h.C is None else h.C.pin_memory()
        hD = torch.empty((w.M, w.N), dtype=wl.DTYPES[w.out_dtype], pin_memory=True)
        hA_l = wl.logical(hA, w.M, w.K, w.layoutA)
        hB_l = wl.logical(hB, w.K, w.N, w.layoutB)
        hC_l = None if hC is None else hC[:, :w.N]
        for _ in range(3):
            plan.gemm_host(hA_l, hB_l, hC_l, hD, alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype,
                           out_dtype=w.out_dtype, stream=stream, **ep)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            # every step copies its inputs in and its result out (ordered on `stream`)
            plan.gemm_host(hA_l, hB_l, hC_l, hD, alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype,
                           out_dtype=w.out_dtype, stream=stream, sync=False, **ep)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size() + (
            0 if hC is None else hC.numel() * hC.element_size())
        d2h = hD.numel() * hD.element_size()
        e2e = {"value": w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "gemm_run_host (C ABI) on pinned host A, B (C) and D: copies in, row blocks of D "
                       "computed and copied back, overlapped on internal streams"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_src = measured_peaks()
    avg_s = ms_per_step * 1e-3
    achieved = w.flops / avg_s / 1e12
    ratio = NOMINAL_RATIO[w.in_dtype]
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) * ratio   # fp16 dense rate = bf16 dense rate
    kernel_tag = ("prior_art_" + args.prior_art if args.prior_art else
                  plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype).split()[0])
    traffic = traffic_from_profiles(w.name, kernel_tag)
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    roofline = rooflines(w, avg_s, peak, hbm_peak, traffic, peak_src, ratio)
    roofline["kernel"] = kernel_tag
    try:
        # tensor-core rate probe (no memory traffic): cycles per 256x256x16 MMA and the peak
        # it implies at the clock measured meanwhile; outside the timed region
        probe = tc.gemm_measure_mma_rate(dev.index if dev.index is not None else 0, w.in_dtype,
                                         w.accum_dtype, 256)
        roofline["mma_probe"] = {k: probe[k] for k in ("cycles_per_mma", "flop_per_clk_per_sm", "sm_mhz",
                                                       "peak_tflops_at_clock")}
        roofline["mma_probe"]["peak_tflops_at_2070_mhz"] = probe["sms"] * probe["flop_per_clk_per_sm"] * 2070e6 / 1e12
    except Exception as e:   # the probe is context; never fail the bench on it
        roofline["mma_probe"] = {"error": str(e)[:120]}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(w, h)
    out = {
        "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.in_dtype, "data": "synthetic",
        "config": {
            "workload": workload_desc(w),
            "accumulate": w.accum_dtype, "out": w.out_dtype,
            "l2": {"write": f"flushed before every step by a {L2_FLUSH_BYTES >> 20} MiB write (outside the "
                            "step's events; the dirty lines are written back during the step)",
                   "write_read": f"flushed before every step by a {L2_FLUSH_BYTES >> 20} MiB write followed by "
                                 "a read of the same buffer (outside the step's events): L2 holds no input "
                                 "and no dirty line when the step starts",
                   "none": "not flushed (inputs may be L2-resident)"}[args.flush],
            "parallelism": "replicas" if world > 1 else "single",
            "pct_of_nominal_dense_fp16": 100.0 * value / world / NOMINAL_DENSE_FP16_TFLOPS,
            "nominal_dense_fp16_tflops": NOMINAL_DENSE_FP16_TFLOPS,
            "pct_of_nominal_dense_same_kind": 100.0 * value / world / (NOMINAL_DENSE_FP16_TFLOPS * ratio),
            "kernel_config": (kernel_tag if args.prior_art else
                              plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)),
            "epilogue": args.epilogue,
            "autotune": tuning,
            "wall_s_timed_loop": wall,
            "step_ms_min": min(per_step), "step_ms_median": statistics.median(per_step),
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    print(json.dumps(out), flush=True)
    plan.close()
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
