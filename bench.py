#!/usr/bin/env python
"""Benchmark: FP8 block-scaled GEMM (and MXFP8 GEMM) throughput on GB300.

One "step" = one GEMM over one batch of synthetic inputs resident in HBM
(for the grouped MoE workloads: the leader descriptor plus the grouped GEMM).
Prints ONE JSON line (rank 0). Default workload: the blockscale GEMM
M=4096 N=2048 K=7168 (narrow-N, deep-K) at seed 0. Blockscale lines also time
the promote-free twin and the E4M3-output variant on the same operands; MoE
lines time the unpaired arm beside the paired one.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
  python bench.py --ksweep [--workload bs_...]    # fixed + slope per K block, kernel vs twin

Timing: W untimed steps, then K timed steps between a barrier +
cuda.synchronize() on both sides. Before every step a 256 MiB buffer is
written to flush the 126 MiB L2 (outside the per-step CUDA-event pair on the
launching stream); ms_per_step is the mean of the per-step event durations.
Multi-GPU (torchrun): every rank runs the same GEMM on its own GPU (weak
scaling, no collective on the data path); the per-rank times are max-reduced.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "TFLOP/s and % of FP8 dense roofline per (M,N,K), 1×GB300, vs CPU oracle"
DEFAULT_WORKLOAD = "bs_narrowN_4096x2048x7168"
FLUSH_BYTES = 256 << 20
# Pages' own absolute numbers for an identical workload and metric (MI355X, context only):
# PR "1x32 ue8m0 (MXFP8) 8-wave FlyDSL GEMM for gfx950", section "Measured" (new kernel, µs).
PAGE_US = {"mx_16384x5120x2048": 157.0, "mx_16384x8192x1280": 175.8, "mx_1024x5120x2048": 35.5,
           "mx_2048x5120x2048": 42.7, "mx_4096x5120x2048": 65.2, "mx_1024x8192x1280": 30.6,
           "mx_2048x8192x1280": 37.9, "mx_4096x8192x1280": 56.4}
KERNEL_NAMES = {"bs": "fp8bs_blockscale_kernel", "mx": "fp8bs_mxfp8_kernel"}


def kernel_name(decoded):
    """The kernel a configuration runs (decoded configuration id)."""
    kind, sched = decoded["kind"], decoded["schedule"]
    if kind == "mxfp8_pair":
        return "fp8bs_mxfp8_pair_kernel"
    if kind == "mxfp8":
        return "fp8bs_mxfp8_sk_kernel" if sched == "stream_k" else "fp8bs_mxfp8_kernel"
    if kind == "blockscale_pair":
        return "fp8bs_blockscale_pair_kernel"
    return "fp8bs_blockscale_kernel"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-twin", action="store_true", help="skip the promote-free twin timing (blockscale)")
    p.add_argument("--no-mx-gates", action="store_true",
                   help="default line: skip timing the two gated MXFP8 workloads (M = 16384) beside it")
    p.add_argument("--ref-seconds", type=float, default=240.0,
                   help="reference arm: CPU time budget of the whole run (warm-up + timed steps)")
    p.add_argument("--raster", type=int, choices=[0, 1], default=None,
                   help="force the tile order of the workload's configuration (0: N panels in groups, M inside; "
                        "1: the converse); default: the shape rule's")
    p.add_argument("--raster-group", type=int, default=0, help="panels per raster group (0 = default 1)")
    p.add_argument("--raster-sweep", action="store_true",
                   help="time the workload's GEMM for both raster directions and several group sizes "
                        "(skill card 'Mechanism B'); one JSON line")
    p.add_argument("--cpu-all", action="store_true",
                   help="time the oracle on every workload (full C, all host cores) and on one core for the "
                        "smallest blockscale and MXFP8 workloads; one JSON line, no GPU")
    p.add_argument("--ksweep", action="store_true",
                   help="blockscale: time the kernel and its twin over K at the workload's M, N; print the "
                        "fixed + slope fit (skill card 'Bottleneck diagnosis' step 6) instead of the bench line")
    p.add_argument("--warmup-seconds", type=float, default=1.0,
                   help="minimum warm-up duration (clock sampling); 0 for profiler runs")
    return p.parse_args()


def workload_shape(name):
    w = workloads.WORKLOADS[name]
    return w["kind"], w["M"], w["N"], w["K"]


def algorithmic_bytes(kind, M, N, K):
    """Each operand read once, C written once."""
    if kind == "bs":
        return M * K + N * K + 4 * M * (K // 128) + 4 * ((N + 127) // 128) * (K // 128) + 2 * M * N
    return M * K + N * K + M * (K // 32) + N * (K // 32) + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        # fp8 dense = 2 x the measured bf16 dense rate (nominal ratio 4.5 / 2.25 PFLOP/s)
        return {"fp8_tflops": 2.0 * float(pk["bf16_tflops"]), "hbm_gbs": float(pk["hbm_gbs"]),
                "source": "measured"}
    except Exception:
        return {"fp8_tflops": 2.0 * 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


def source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "fp8_block_scaled_e4m3_gb300", "csrc")
    for fn in sorted(os.listdir(d)):
        with open(os.path.join(d, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_values(kernel, workload):
    """Key/value lines of the committed ncu summary of this kernel on this workload,
    or None when there is none or it was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_hash") != source_hash():
        return None
    return vals


def _profiled_float(kernel, workload, key):
    vals = profiled_values(kernel, workload)
    try:
        return float(vals[key]) if vals else None
    except (KeyError, ValueError):
        return None


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this exact kernel source."""
    return _profiled_float(kernel, workload, "dram_bytes_per_launch")


def profiled_tensor_active(kernel, workload):
    """ncu sm__pipe_tensor_cycles_active (% of peak sustained, elapsed) from the same summary."""
    return _profiled_float(kernel, workload, "sm__pipe_tensor_cycles_active.pct_of_peak_sustained_elapsed")


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, pg, torch, device):
    """The slowest rank's time (every rank gets it); `pg` is torch.distributed or None."""
    if pg is None:
        return ms
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world, flops_per_rank, ms):
    """Whole-job throughput: every rank runs one GEMM of `flops_per_rank` per step
    (weak scaling, no exchange), the job's step time is the slowest rank's."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def make_device_inputs(kind, M, N, K, seed, torch):
    x = workloads.make_inputs(kind, M, N, K, seed)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if kind == "bs":
        host = [x.A, workloads.a_scale_to_kmajor(x.a_scale), x.B, np.ascontiguousarray(x.b_scale, np.float32)]
    else:
        host = [x.A, x.a_e8m0, x.B, x.b_e8m0]
    return x, host, [dev(h) for h in host]


def cpu_oracle_sample(kind, x, target_s):
    """Time the oracle (as it stands) on a bounded row sample of this workload."""
    import oracle
    M, N, K = x.M, x.N, x.K
    f = (lambda r0, r1: oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, rows=(r0, r1))) if kind == "bs" else \
        (lambda r0, r1: oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0, rows=(r0, r1)))
    threads = oracle.max_threads()
    rows = min(M, max(threads, 8))
    t0 = time.perf_counter()
    f(0, rows)
    dt = time.perf_counter() - t0
    if dt < target_s / 4 and rows < M:
        rows = int(min(M, max(rows + 1, rows * (target_s / max(dt, 1e-3)) * 0.9)))
        t0 = time.perf_counter()
        f(0, rows)
        dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of C ({rows}x{N} outputs, full K={K}) in {dt:.2f} s, "
                      f"fp64 dequantise + naive triple loop, OpenMP over rows"}


def _oracle_fn(kind, x):
    import oracle
    if kind == "bs":
        return lambda r0, r1: oracle.blockscale(x.A, x.a_scale, x.B, x.b_scale, rows=(r0, r1))
    return lambda r0, r1: oracle.mxfp8(x.A, x.a_e8m0, x.B, x.b_e8m0, rows=(r0, r1))


def run_reference(args):
    """The oracle as it stands, timed on the host cores. Every step computes the
    same rows of C: all of C when the whole run (warm-up + timed steps) fits the
    --ref-seconds budget at the measured rate, else the first rows that do (the
    line says how many). ms_per_step is the measured wall time of one step; the
    value is the measured rate over those steps (nothing is extrapolated)."""
    import oracle
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    kind, M, N, K = workload_shape(args.workload)
    x = workloads.make_inputs(kind, M, N, K, args.seed)
    fn = _oracle_fn(kind, x)
    threads = oracle.max_threads()
    probe = min(M, max(threads, 8))
    t0 = time.perf_counter()
    fn(0, probe)
    per_row = (time.perf_counter() - t0) / probe
    n_steps = args.warmup + args.steps
    rows = M if per_row * M * n_steps <= args.ref_seconds else \
        int(min(M, max(threads, args.ref_seconds / (n_steps * per_row))))
    walls = []
    for i in range(n_steps):
        t0 = time.perf_counter()
        fn(0, rows)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            walls.append(dt)
    ms = statistics.mean(walls) * 1e3
    flops = 2.0 * rows * N * K
    val = flops / (ms * 1e-3) / 1e12
    what = "all of C" if rows == M else f"rows 0..{rows - 1} of C (bounded by --ref-seconds {args.ref_seconds:g})"
    cb = {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
          "sample": f"every step: {what}, {rows}x{N} outputs, full K={K}; fp64 dequantise + naive triple loop, "
                    f"OpenMP over rows; mean step {ms / 1e3:.2f} s"}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K, "seed": args.seed},
            "rows_per_step": rows, "extrapolated": False,
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_cpu_all(args):
    """Oracle time on every blockscale and MXFP8 workload (seed 0, all of C, all
    host cores), plus one core for the smallest blockscale workload and the
    M = 1024 MXFP8 workloads (a child process with OMP_NUM_THREADS=1)."""
    import oracle
    import platform
    out = {"cpu_all": True, "cores": oracle.max_threads(), "cpu": platform.processor() or platform.machine(),
           "kind": "oracle", "what": "all of C per workload, seed 0, fp64 dequantise + naive triple loop, "
                                     "OpenMP over rows", "workloads": {}}
    for name, w in workloads.WORKLOADS.items():
        if w["kind"] not in ("bs", "mx"):
            continue
        kind, M, N, K = workload_shape(name)
        x = workloads.make_inputs(kind, M, N, K, 0)
        fn = _oracle_fn(kind, x)
        t0 = time.perf_counter()
        fn(0, M)
        dt = time.perf_counter() - t0
        out["workloads"][name] = {"seconds": dt, "tflops": 2.0 * M * N * K / dt / 1e12}
    single = {}
    for name in ("bs_tiny_256x512x512", "mx_1024x5120x2048", "mx_1024x8192x1280"):
        code = (f"import sys, time, json; sys.path.insert(0, {ROOT!r}); import bench, workloads, oracle; "
                f"k, M, N, K = bench.workload_shape({name!r}); x = workloads.make_inputs(k, M, N, K, 0); "
                f"fn = bench._oracle_fn(k, x); t0 = time.perf_counter(); fn(0, M); dt = time.perf_counter() - t0; "
                f"print(json.dumps({{'threads': oracle.max_threads(), 'seconds': dt, "
                f"'tflops': 2.0 * M * N * K / dt / 1e12}}))")
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
        single[name] = json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else {"error": r.stderr[-300:]}
    out["single_core"] = single
    print(json.dumps(out), flush=True)
    return 0


def apply_raster_knobs(args, f, kind, M, N, K):
    """--raster / --raster-group: force the tile order of the shape rule's configuration."""
    f.set_raster_group(args.raster_group)
    if args.raster is not None:
        cid = f.select_config(kind, M, N, K, f.device_info()["num_sms"])
        f.set_config_override(cid - ((cid // 10) % 10) * 10 + 10 * args.raster)


def run_raster_sweep(args):
    """Time the workload's GEMM (its own configuration) under each tile order:
    raster 0 / 1 and panel groups of 1, 2, 4, 8, 16 (L2 flushed, CUDA events)."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    kind, M, N, K = workload_shape(args.workload)
    _, _, d = make_device_inputs(kind, M, N, K, args.seed, torch)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gemm = f.gemm_blockscale if kind == "bs" else f.gemm_mxfp8
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    base = f.select_config(kind, M, N, K, f.device_info()["num_sms"])
    n = max(10, min(args.steps, 50))
    rows = []
    try:
        for raster in (0, 1):
            for group in (1, 2, 4, 8, 16):
                f.set_config_override(base - ((base // 10) % 10) * 10 + 10 * raster)
                f.set_raster_group(group)
                for _ in range(3):
                    gemm(d[0], d[1], d[2], d[3], C=C)
                ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
                for a, b in ev:
                    flush.fill_(1)
                    a.record(stream)
                    gemm(d[0], d[1], d[2], d[3], C=C)
                    b.record(stream)
                torch.cuda.synchronize()
                assert f.get_status() == 0
                us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
                rows.append({"raster": raster, "group": group, "config_id": f.last_config_id(), "us": us,
                             "tflops": 2.0 * M * N * K / (us * 1e-6) / 1e12})
    finally:
        f.set_config_override(0)
        f.set_raster_group(0)
    print(json.dumps({"raster_sweep": args.workload, "M": M, "N": N, "K": K, "shape_rule_config": base,
                      "l2": "flushed", "steps": n, "points": rows}), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    import fp8_block_scaled_e4m3_gb300 as f

    kind, M, N, K = workload_shape(args.workload)
    x, host, d = make_device_inputs(kind, M, N, K, args.seed, torch)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    gemm = f.gemm_blockscale if kind == "bs" else f.gemm_mxfp8
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        gemm(d[0], d[1], d[2], d[3], C=C)

    apply_raster_knobs(args, f, kind, M, N, K)
    # correctness gate and runtime signature before timing
    step()
    assert f.get_status() == 0
    cfg_id = f.last_config_id()
    assert f.decode_config(cfg_id)["kind"].startswith("blockscale" if kind == "bs" else "mxfp8")

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    # Warm-up: at least W steps and at least one second of load, so the clock
    # sampler (started above, stopped after the timed loop) sees steady-state clocks.
    t_w = time.perf_counter()
    n_w = 0
    while n_w < max(args.warmup, 3) or time.perf_counter() - t_w < args.warmup_seconds:
        flush.fill_(1)
        step()
        n_w += 1
        if n_w % 50 == 0:
            torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(1)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    per_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(statistics.mean(per_ms), pg, torch, "cuda")
    kernel_ms = ms
    if kind == "mx":
        # The dominant kernel alone (the GEMM on packed scales, without the
        # scale-pack launch), same protocol: L2 flush, CUDA events on the stream.
        a_sf = f.pack_mx_scales(d[1], K)
        b_sf = f.pack_mx_scales(d[3], K)
        for _ in range(3):
            f.gemm_mxfp8_packed(d[0], a_sf, d[2], b_sf, C=C)
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(1)
            kev[i][0].record(stream)
            f.gemm_mxfp8_packed(d[0], a_sf, d[2], b_sf, C=C)
            kev[i][1].record(stream)
        torch.cuda.synchronize()
        kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
        assert f.get_status() == 0
    assert f.get_status() == 0
    # hot-L2 figure beside the cold one: the same step back to back, no flush
    for _ in range(3):
        step()
    hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for a, b in hev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    assert f.get_status() == 0
    hot_ms = statistics.mean(a.elapsed_time(b) for a, b in hev)
    if args.raster is not None or args.raster_group:
        f.set_config_override(0)   # the twin and the MXFP8 lines below run their own shape rules
        f.set_raster_group(0)

    flops = 2.0 * M * N * K
    value = aggregate_tflops(world, flops, ms)
    peaks = load_peaks()
    kernel_tflops = flops / (kernel_ms * 1e-3) / 1e12
    kname = kernel_name(f.decode_config(cfg_id))
    traffic = profiled_traffic(kname, args.workload)
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peaks["fp8_tflops"], "unit": "TFLOP/s",
                "frac": kernel_tflops / peaks["fp8_tflops"], "traffic": traffic,
                "tensor_active_pct_ncu": profiled_tensor_active(kname, args.workload),
                "peak_source": f"{peaks['source']}: 2 x MEASURED_PEAKS bf16_tflops (fp8/bf16 nominal ratio 2)"
                if peaks["source"] == "measured" else "fallback 2 x 1900 TFLOP/s bf16",
                "algorithmic_bytes": algorithmic_bytes(kind, M, N, K),
                "hbm_time_frac": (algorithmic_bytes(kind, M, N, K) / (peaks["hbm_gbs"] * 1e9)) / (kernel_ms * 1e-3),
                "kernel": kname, "kernel_ms": kernel_ms}

    twin = None
    if kind == "bs" and not args.no_twin:
        twin = measure_twin(args, torch, f, d, C, flush, stream, flops, kernel_ms, peaks)

    e4m3 = None
    if kind == "bs" and not args.no_twin and N % 16 == 0:
        e4m3 = measure_e4m3out(args, torch, f, d, flush, stream, flops, kernel_ms, peaks, M, N)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, torch, f, kind, M, N, K, host, gemm)

    mx_gates = None
    if kind == "bs" and args.workload == DEFAULT_WORKLOAD and not args.no_mx_gates:
        mx_gates = {w: measure_mx_gate(args, torch, f, w, flush, stream, peaks) for w in MX_GATES}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(kind, x, args.cpu_seconds)

    page_us = PAGE_US.get(args.workload)
    vs = value / (flops / (page_us * 1e-6) / 1e12) if page_us else None
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": vs, "dtype": "e4m3 x e4m3 -> f32 accumulate -> bf16", "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K, "seed": args.seed,
                       "l2": "flushed before every step by a 256 MiB write (outside the timed events)",
                       "kernel_config": f.decode_config(cfg_id), "config_id": cfg_id,
                       "parallelism": f"{world} independent replicas (weak scaling)",
                       "wall_s_timed_loop": wall, "warmup_steps_run": n_w, "ms_min": min(per_ms),
                       "ms_median": statistics.median(per_ms), "hot_l2_ms_per_step": hot_ms},
            "roofline": roofline, "ceiling_twin": twin, "e4m3_out": e4m3, "mxfp8_gates": mx_gates,
            "gpu_launches": args.steps * (f.lib().fp8bs_launches_per_call() if kind == "bs"
                                          else f.lib().fp8mx_launches_per_call()),
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


MX_GATES = ("mx_16384x5120x2048", "mx_16384x8192x1280")


def measure_mx_gate(args, torch, f, workload, flush, stream, peaks):
    """One of the two gated MXFP8 workloads (M = 16384), timed beside the default
    blockscale line with the same protocol (L2 flushed before every step, CUDA
    events on the launching stream, warm-up first): the public call (scale pack
    + GEMM, what a user of fp8mx_gemm gets) and the GEMM alone on packed scales
    (the roofline kernel). The configuration that ran is asserted to be the
    CTA-pair kernel the shape rule picks for M >= 4096."""
    kind, M, N, K = workload_shape(workload)
    _, _, d = make_device_inputs(kind, M, N, K, 0, torch)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    n = max(5, min(args.steps, 50))

    def timed(fn):
        for _ in range(3):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        assert f.get_status() == 0
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    call_ms = timed(lambda: f.gemm_mxfp8(d[0], d[1], d[2], d[3], C=C))
    cfg_id = f.last_config_id()
    dec = f.decode_config(cfg_id)
    assert dec["kind"] == "mxfp8_pair", dec
    a_sf = f.pack_mx_scales(d[1], K)
    b_sf = f.pack_mx_scales(d[3], K)
    gemm_ms = timed(lambda: f.gemm_mxfp8_packed(d[0], a_sf, d[2], b_sf, C=C))
    assert f.last_config_id() == cfg_id
    flops = 2.0 * M * N * K
    kname = kernel_name(dec)
    tf = flops / (gemm_ms * 1e-3) / 1e12
    return {"M": M, "N": N, "K": K, "seed": 0, "config_id": cfg_id, "steps": n,
            "public_call": {"ms": call_ms, "achieved": flops / (call_ms * 1e-3) / 1e12,
                            "frac": flops / (call_ms * 1e-3) / 1e12 / peaks["fp8_tflops"], "unit": "TFLOP/s",
                            "launches": f.lib().fp8mx_launches_per_call()},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["fp8_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["fp8_tflops"], "kernel": kname, "kernel_ms": gemm_ms,
                         "traffic": profiled_traffic(kname, workload),
                         "tensor_active_pct_ncu": profiled_tensor_active(kname, workload),
                         "algorithmic_bytes": algorithmic_bytes(kind, M, N, K)},
            "gate": {"frac_at_least": 0.60, "met": tf / peaks["fp8_tflops"] >= 0.60}}


def measure_twin(args, torch, f, d, C, flush, stream, flops, kernel_ms, peaks):
    """The same A and B through the promote-free twin (one fp32 scale for the whole
    tensor, applied once in the epilogue), timed with the same protocol. The gap
    between the two kernels is what the per-block scales cost on this shape."""
    alpha = 0.03125
    for _ in range(3):
        f.gemm_tensorscale(d[0], d[2], alpha, C=C)
    assert f.get_status() == 0
    twin_cfg = f.last_config_id()
    n = max(3, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush.fill_(1)
        ev[i][0].record(stream)
        f.gemm_tensorscale(d[0], d[2], alpha, C=C)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert f.get_status() == 0
    twin_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    tf = flops / (twin_ms * 1e-3) / 1e12
    return {"kernel": "fp8bs_tensorscale_kernel", "config_id": twin_cfg, "steps": n, "kernel_ms": twin_ms,
            "achieved": tf, "frac": tf / peaks["fp8_tflops"], "unit": "TFLOP/s",
            "scale_tax": kernel_ms / twin_ms - 1.0}


def measure_e4m3out(args, torch, f, d, flush, stream, flops, kernel_ms, peaks, M, N):
    """The same GEMM with the E4M3 output epilogue (C8 = e4m3(c_scale * C), one
    byte per element instead of two), timed with the same protocol."""
    C8 = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    c_scale = 32.0
    for _ in range(3):
        f.gemm_blockscale_e4m3out(d[0], d[1], d[2], d[3], c_scale, C8=C8)
    assert f.get_status() == 0
    n = max(3, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush.fill_(1)
        ev[i][0].record(stream)
        f.gemm_blockscale_e4m3out(d[0], d[1], d[2], d[3], c_scale, C8=C8)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    assert f.get_status() == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    tf = flops / (ms * 1e-3) / 1e12
    return {"kernel": "fp8bs_blockscale_kernel (E4M3 C)", "config_id": f.last_config_id(), "steps": n,
            "kernel_ms": ms, "achieved": tf, "frac": tf / peaks["fp8_tflops"], "unit": "TFLOP/s",
            "c_bytes": M * N, "speedup_vs_bf16_c": kernel_ms / ms}


def measure_e2e(args, torch, f, kind, M, N, K, host, gemm):
    """Same metric through the public API with host buffers: every step uploads all of
    its inputs from pinned host memory, runs the GEMM and downloads C into pinned host
    memory, all inside the timed region. Consecutive steps are pipelined the way a
    serving loop would run them: uploads on one stream, GEMMs on a second, downloads on
    a third, with two sets of device and host buffers, so step k+1's upload overlaps
    step k's GEMM and step k-1's download. Time = first upload start to last download
    end; value = steps x 2MNK / time. (Splitting each direction over two copy streams
    measured slower: the host link, ~190 GB/s per direction here, is the bound.)"""
    pinned = [[torch.from_numpy(np.ascontiguousarray(h)).pin_memory() for h in host] for _ in range(2)]
    dev = [[torch.empty_like(p, device="cuda") for p in pinned[0]] for _ in range(2)]
    C = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    C_host = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_gemm, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(p.numel() * p.element_size() for p in pinned[0])
    d2h = C_host[0].numel() * C_host[0].element_size()
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "gemm", "out")}

    def run(n, t0=None, t1=None):
        torch.cuda.synchronize()
        if t0 is not None:
            t0.record(s_in)
        for k in range(n):
            b = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev["gemm"][b])      # GEMM k-2 has read these inputs
                for p, dv in zip(pinned[b], dev[b]):
                    dv.copy_(p, non_blocking=True)
                ev["in"][b].record(s_in)
            with torch.cuda.stream(s_gemm):
                s_gemm.wait_event(ev["in"][b])
                if k >= 2:
                    s_gemm.wait_event(ev["out"][b])     # C of step k-2 has been downloaded
                gemm(dev[b][0], dev[b][1], dev[b][2], dev[b][3], C=C[b])
                ev["gemm"][b].record(s_gemm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["gemm"][b])
                C_host[b].copy_(C[b], non_blocking=True)
                ev["out"][b].record(s_out)
        if t1 is not None:
            t1.record(s_out)
        torch.cuda.synchronize()

    run(4)
    n = max(5, min(args.steps, 50))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    run(n, t0, t1)
    ms = t0.elapsed_time(t1) / n
    assert f.get_status() == 0
    return {"value": 2.0 * M * N * K / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "pipeline": "uploads, GEMMs and downloads of consecutive steps on three streams"}


# ------------------------------------------------------------ grouped MoE stage-1
def moe_stats(block_expert, num_experts):
    be = np.asarray(block_expert)
    runs = np.diff(np.flatnonzero(np.r_[True, be[1:] != be[:-1], True])) if len(be) else np.zeros(0, int)
    pairs = int(np.sum(runs // 2))
    return {"n_blocks": int(len(be)), "experts_used": int(len(runs)), "pair_count": pairs,
            "pair_count_fraction": pairs / max(1, len(be)), "paired_block_fraction": 2 * pairs / max(1, len(be))}


def moe_work(w, x):
    """Useful FLOPs (routed rows only), and algorithmic bytes: the sorted rows and
    their scales read once, each used expert's weights and scales read once, C written once."""
    rows = x.A.shape[0]
    N, K = w["N"], w["K"]
    used = len(np.unique(x.block_expert))
    flops = 2.0 * w["tokens"] * w["top_k"] * N * K
    nbytes = (rows * K + 4 * rows * (K // 128) + used * (N * K + 4 * (N // 128) * (K // 128)) + 2 * rows * N)
    return flops, nbytes


def moe_cpu_sample(x, target_s):
    import oracle
    t0 = time.perf_counter()
    done = 0
    b = 0
    while b < x.n_blocks and (done == 0 or time.perf_counter() - t0 < target_s):
        e = int(x.block_expert[b])
        rows = slice(64 * b, 64 * b + 64)
        oracle.blockscale(x.A[rows], x.a_scale[rows], x.B[e], x.b_scale[e])
        done += 1
        b += 1
    dt = time.perf_counter() - t0
    flops = 2.0 * 64 * done * x.N * x.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{done} of {x.n_blocks} sort blocks (64 rows each, padded rows included) in {dt:.2f} s, "
                      f"fp64 dequantise + naive triple loop"}


def run_moe(args):
    import torch
    world, rank, local = dist_setup(args)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        pg = dist
    import fp8_block_scaled_e4m3_gb300 as f

    w = workloads.WORKLOADS[args.workload]
    E, N, K = w["experts"], w["N"], w["K"]
    x = workloads.make_moe_inputs(w["tokens"], w["top_k"], E, N, K, seed=args.seed, skew=w["skew"])
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    host = [x.A, workloads.a_scale_to_kmajor(x.a_scale), x.block_expert]
    A, sa, be = [dev(h) for h in host]
    B, sb = dev(x.B), dev(x.b_scale)
    lead = torch.empty(x.n_blocks, dtype=torch.int32, device="cuda")
    nl = torch.empty(1, dtype=torch.int32, device="cuda")
    C = torch.empty((x.A.shape[0], N), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def segment(pair=True, a=A, s_a=sa, table=be, out=C):
        f.moe_leaders(table, E, pair=pair, leaders=lead, n_leaders=nl)
        f.gemm_moe(a, s_a, B, sb, table, lead, nl, C=out)

    def timed(fn, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush.fill_(1)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        assert f.get_status() == 0
        return [a.elapsed_time(b) for a, b in ev]

    segment()
    assert f.get_status() == 0
    cfg_id = f.last_config_id()
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    t_w = time.perf_counter()
    n_w = 0
    while n_w < max(args.warmup, 3) or time.perf_counter() - t_w < args.warmup_seconds:
        flush.fill_(1)
        segment()
        n_w += 1
        if n_w % 50 == 0:
            torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    per_ms = timed(segment, args.steps)
    if pg:
        pg.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(statistics.mean(per_ms), pg, torch, "cuda")
    n_ab = max(3, min(args.steps, 100))
    gemm_ms = statistics.mean(timed(lambda: f.gemm_moe(A, sa, B, sb, be, lead, nl, C=C), n_ab))
    n_leaders_paired = int(nl.item())
    unpaired_ms = statistics.mean(timed(lambda: segment(pair=False), n_ab))
    n_leaders_unpaired = int(nl.item())
    paired_ms = statistics.mean(timed(segment, n_ab))
    desc_ms = statistics.mean(timed(lambda: f.moe_leaders(be, E, leaders=lead, n_leaders=nl), n_ab))

    flops, nbytes = moe_work(w, x)
    value = aggregate_tflops(world, flops, ms)
    peaks = load_peaks()
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tensor = 2.0 * x.A.shape[0] * N * K / (peaks["fp8_tflops"] * 1e12)   # padded rows go through the MMAs
    if t_hbm >= t_tensor:
        achieved = nbytes / (gemm_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "traffic": None}
    else:
        achieved = 2.0 * x.A.shape[0] * N * K / (gemm_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["fp8_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["fp8_tflops"], "traffic": None}
    roofline["traffic"] = profiled_traffic("fp8bs_blockscale_kernel", args.workload)
    roofline.update({"kernel": "fp8bs_blockscale_kernel (grouped)", "kernel_ms": gemm_ms,
                     "algorithmic_bytes": nbytes, "hbm_time_us": t_hbm * 1e6, "tensor_time_us": t_tensor * 1e6,
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS hbm_gbs / 2 x bf16_tflops)"})

    e2e = None
    if not args.no_e2e:
        # per step: the routed rows, their scales and the routing table up, C down (weights resident)
        pin = [torch.from_numpy(np.ascontiguousarray(h)).pin_memory() for h in host]
        outp = torch.empty(C.shape, dtype=C.dtype).pin_memory()
        dA, dsa, dbe = [torch.empty_like(p, device="cuda") for p in pin]

        def e2e_step():
            for dst, src in zip((dA, dsa, dbe), pin):
                dst.copy_(src, non_blocking=True)
            segment(a=dA, s_a=dsa, table=dbe)
            outp.copy_(C, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        n_e = max(3, min(args.steps, 50))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / n_e
        e2e = {"value": aggregate_tflops(world, flops, e_ms), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(p.numel() * p.element_size() for p in pin)),
               "d2h_bytes_per_step": int(outp.numel() * outp.element_size()), "ms_per_step": e_ms,
               "pipeline": "serial: upload, segment, download per step on one stream"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = moe_cpu_sample(x, args.cpu_seconds)

    st = moe_stats(x.block_expert, E)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 accumulate -> bf16", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": w["tokens"], "top_k": w["top_k"], "experts": E,
                       "N": N, "K": K, "skew": w["skew"], "seed": args.seed, "rows": int(x.A.shape[0]),
                       "step": "leader descriptor + grouped GEMM (paired)",
                       "flops": "2 * tokens * top_k * N * K (routed rows only)",
                       "l2": "flushed before every step by a 256 MiB write (outside the timed events)",
                       "kernel_config": f.decode_config(cfg_id), "config_id": cfg_id,
                       "parallelism": f"{world} independent replicas (weak scaling)",
                       "wall_s_timed_loop": wall, "warmup_steps_run": n_w, "ms_min": min(per_ms)},
            "roofline": roofline,
            "pairing": dict(st, n_leaders_paired=n_leaders_paired, n_leaders_unpaired=n_leaders_unpaired,
                            paired_segment_ms=paired_ms, unpaired_segment_ms=unpaired_ms,
                            descriptor_ms=desc_ms, speedup=unpaired_ms / paired_ms),
            "gpu_launches": args.steps * 2, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def run_moe_reference(args):
    """The oracle on the grouped workload: every step computes the same sort
    blocks (all of them when the run fits --ref-seconds, else the first ones
    that do); ms_per_step is the measured wall time of one step."""
    import oracle
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_moe_inputs(w["tokens"], w["top_k"], w["experts"], w["N"], w["K"], seed=args.seed,
                                  skew=w["skew"])

    def blocks(nb):
        for b in range(nb):
            e = int(x.block_expert[b])
            rows = slice(64 * b, 64 * b + 64)
            oracle.blockscale(x.A[rows], x.a_scale[rows], x.B[e], x.b_scale[e])

    t0 = time.perf_counter()
    blocks(1)
    per_block = time.perf_counter() - t0
    n_steps = args.warmup + args.steps
    nb = x.n_blocks if per_block * x.n_blocks * n_steps <= args.ref_seconds else \
        int(min(x.n_blocks, max(1, args.ref_seconds / (n_steps * per_block))))
    walls = []
    for i in range(n_steps):
        t0 = time.perf_counter()
        blocks(nb)
        if i >= args.warmup:
            walls.append(time.perf_counter() - t0)
    ms = statistics.mean(walls) * 1e3
    val = 2.0 * 64 * nb * x.N * x.K / (ms * 1e-3) / 1e12
    cb = {"value": val, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
          "sample": f"every step: {nb} of {x.n_blocks} sort blocks (64 rows each, padded rows included), "
                    f"fp64 dequantise + naive triple loop; mean step {ms / 1e3:.2f} s"}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "seed": args.seed}, "blocks_per_step": nb, "extrapolated": False,
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ksweep(args):
    """t(K) = fixed + slope * K/128 for the blockscale kernel and its promote-free
    twin at the workload's M and N (L2 flushed, CUDA events, least squares)."""
    import torch
    import fp8_block_scaled_e4m3_gb300 as f
    kind, M, N, K0 = workload_shape(args.workload)
    assert kind == "bs", "--ksweep is for blockscale workloads"
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    n = max(10, min(args.steps, 100))
    ks = [k for k in (1024, 2048, 3072, 4096, 5120, 6144, 7168) if k <= max(K0, 1024)]
    rows = []
    for K in ks:
        x, _, d = make_device_inputs("bs", M, N, K, args.seed, torch)
        out = {"K": K, "KB": K // 128}
        for name, fn in (("blockscale", lambda: f.gemm_blockscale(*d)),
                         ("twin", lambda: f.gemm_tensorscale(d[0], d[2], 1e-6))):
            for _ in range(3):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for a, b in ev:
                flush.fill_(1)
                a.record(stream)
                fn()
                b.record(stream)
            torch.cuda.synchronize()
            assert f.get_status() == 0
            out[name + "_us"] = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
            out[name + "_config"] = f.last_config_id()
        rows.append(out)
    fit = {}
    kb = np.array([r["KB"] for r in rows], dtype=np.float64)
    for name in ("blockscale", "twin"):
        t = np.array([r[name + "_us"] for r in rows])
        slope, fixed = np.polyfit(kb, t, 1)
        fit[name] = {"fixed_us": fixed, "slope_us_per_kblock": slope}
    print(json.dumps({"ksweep": args.workload, "M": M, "N": N, "l2": "flushed", "points": rows, "fit": fit,
                      "note": "slope per K block of the whole GEMM; per CTA divide by the tiles each CTA holds"}),
          flush=True)
    return 0


def main():
    args = parse()
    if args.cpu_all:
        return run_cpu_all(args)
    if args.ksweep:
        return run_ksweep(args)
    if args.raster_sweep:
        return run_raster_sweep(args)
    moe = workloads.WORKLOADS[args.workload]["kind"] == "moe"
    if args.impl == "reference":
        return run_moe_reference(args) if moe else run_reference(args)
    return run_moe(args) if moe else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
