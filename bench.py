#!/usr/bin/env python3
"""Benchmark: fp32 GEMM TFLOP/s on the 4096^3 and 8192^3 workloads.

One step = one C = A*B at M=N=K=4096 (A, B uniform[-1,1), seed 2) followed by
one at M=N=K=8192 (uniform[-1,1), seed 4), both through the library's C ABI
with inputs already in HBM.  `value` is the step's flops divided by the step's
device time (CUDA events on the launching stream), i.e. aggregate TFLOP/s
over the two shapes; per-shape figures are under `per_shape`.  Every GEMM's
operands (192 MB and 768 MB) exceed the 129 MB L2, and each 4096^3 GEMM
follows an 8192^3 one, so no launch starts with its inputs in L2.

`e2e` repeats the step through mt_sgemm_host with pinned host buffers: the
host->device copies of A and B, the GEMM and the device->host copy of C are
all inside its timed region.

`--impl reference` times the reference arm instead: the CPU oracle (fp64
accumulation, all host cores) on a bounded sample of rows of the same two
GEMMs, reported in the same metric.

Multi-GPU (torchrun): every rank runs the same step on its own GPU (replicas;
the GEMM has no exchange step), timing is the max over ranks and `value`
counts the work of all ranks.
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
sys.path.insert(0, ROOT)

import gemm_inputs  # noqa: E402

STEP_WORKLOADS = ("square_4096", "square_8192")
METRIC = "fp32 GEMM TFLOP/s (4096^3, 8192^3) and % of GB300 fp32 FFMA peak"
GB300_SMS = 152
FP32_LANES_PER_SM = 128
SM_MAX_MHZ_FALLBACK = 2070.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def ffma_peak_tflops(sms: int, mhz: float) -> float:
    """FP32 FFMA peak: SMs x 128 lanes x 2 flop x clock."""
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        setattr(self, name, time.time())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        """Median SM clock and active throttle reasons of the samples taken
        inside the timed window (between mark('t0') and mark('t1'))."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", 0.0), getattr(self, "t1", float("inf"))
        inside = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.1]
        for line in inside:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(steps: int, budget_s: float):
    """Times the CPU oracle on row samples of the step's GEMMs.

    Returns (tflops, seconds, cores, description).  The sample is sized from
    a short calibration so the timed part takes about `budget_s` seconds in
    total over `steps` repetitions.
    """
    import numpy as np
    import oracle
    mats = {}
    for name in STEP_WORKLOADS:
        A, B = gemm_inputs.make_workload(name)
        mats[name] = (A.numpy(), B.numpy())
    cores = oracle.max_threads()
    # Calibrate: a few rows of each shape.
    rate = {}
    for name, (A, B) in mats.items():
        rows = np.arange(2 * cores, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.sgemm_rows(A, B, rows)
        dt = time.perf_counter() - t0
        rate[name] = len(rows) / max(dt, 1e-6)  # rows per second
    # Split the budget evenly between the shapes: a row sample of at most M
    # rows (a whole multiple of the thread count, spread evenly over the
    # matrix), repeated if the budget allows more.
    per_shape = budget_s / max(steps, 1) / len(mats)
    plan = {}
    for name in mats:
        M = gemm_inputs.WORKLOADS[name].M
        want = max(cores, int(rate[name] * per_shape) // cores * cores)
        nrows = min(want, M)
        plan[name] = (nrows, max(1, want // nrows))
    total_flops, total_t = 0.0, 0.0
    for _ in range(max(steps, 1)):
        for name, (A, B) in mats.items():
            w = gemm_inputs.WORKLOADS[name]
            nrows, reps = plan[name]
            rows = np.linspace(0, w.M - 1, nrows).astype(np.int64)
            for _r in range(reps):
                t0 = time.perf_counter()
                oracle.sgemm_rows(A, B, rows)
                total_t += time.perf_counter() - t0
                total_flops += 2.0 * len(rows) * w.N * w.K
    desc = ", ".join(f"{plan[n][0]} of {gemm_inputs.WORKLOADS[n].M} rows of {n} x{plan[n][1]}"
                     for n in mats) + f" per step x {max(steps, 1)} steps"
    return total_flops / total_t / 1e12, total_t, cores, desc


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    budget = float(os.environ.get("MT_ORACLE_BUDGET_S", "20"))
    tflops, seconds, cores, desc = oracle_sample(args.steps, budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": seconds * 1e3 / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate",
        "data": "synthetic",
        "config": {"workload": "sgemm 4096^3 (uniform, seed 2) + 8192^3 (uniform, seed 4)",
                   "sample": desc},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def load_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if still current."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except OSError:
        return None
    entry = table.get(kernel_key)
    if not entry:
        return None
    h = hashlib.sha256()
    for rel in entry.get("sources", []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != entry.get("sources_sha256"):
        return None  # the kernel changed since the counters were taken
    return entry.get("bytes_per_launch")


def run_gpu(args):
    import torch
    import tiled_fp32_gemm_gb300 as mt
    from tiled_fp32_gemm_gb300 import build as mt_build

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    mt_build.build()
    mt.lib()

    shapes = [gemm_inputs.WORKLOADS[n] for n in (args.workloads or STEP_WORKLOADS)]
    cfg = mt.make_config(**json.loads(args.config)) if args.config else None
    bufs = []
    for w in shapes:
        A, B = gemm_inputs.make_workload(w)
        a, b = A.cuda(), B.cuda()
        c = torch.empty((w.M, w.N), device="cuda", dtype=torch.float32)
        bufs.append((w, a, b, c, A, B))
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def launch(w, a, b, c):
        st = mt.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K, sptr, cfg)
        if st != mt.MT_OK:
            raise mt.MtError(st, f"mt_sgemm_ex {w.name}")

    plans = {w.name: mt.plan(w.M, w.N, w.K, a=a, b=b, c=c,
                             **(json.loads(args.config) if args.config else {}))
             for (w, a, b, c, _, _) in bufs}

    clocks = ClockSampler(dev).__enter__()
    for _ in range(args.warmup):
        for (w, a, b, c, _, _) in bufs:
            launch(w, a, b, c)
    torch.cuda.synchronize()

    # Timed region: events around every launch on the launching stream.
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in bufs] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("t0")
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        for i, (w, a, b, c, _, _) in enumerate(bufs):
            ev[s][i][0].record(stream)
            launch(w, a, b, c)
            ev[s][i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    clocks.__exit__(None, None, None)
    total_ms = t_start.elapsed_time(t_end)
    per_launch = {w.name: [ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps)]
                  for i, (w, *_r) in enumerate(bufs)}
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    flops_step = sum(w.flops for (w, *_r) in bufs)
    value = world * flops_step * args.steps / (total_ms / 1e3) / 1e12

    clk = clocks.summary()
    peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = clk["sm_max_mhz"] or peaks.get("sm_max_mhz") or SM_MAX_MHZ_FALLBACK
    peak_max = ffma_peak_tflops(sms, sm_max)
    peak_live = ffma_peak_tflops(sms, clk["sm_mhz"]) if clk["sm_mhz"] else None
    per_shape = {}
    for (w, *_r) in bufs:
        ms = statistics.median(per_launch[w.name])
        tf = w.flops / (ms / 1e3) / 1e12
        per_shape[w.name] = {"ms_median": ms, "tflops": tf,
                             "frac_of_ffma_peak_at_max_clock": tf / peak_max,
                             "frac_of_ffma_peak_at_run_clock":
                                 tf / peak_live if peak_live else None,
                             "plan": plans[w.name]}
    # Dominant kernel: the launch with the most device time per step.
    dom = max(bufs, key=lambda x: statistics.mean(per_launch[x[0].name]))[0]
    dom_ms = statistics.mean(per_launch[dom.name])
    achieved = dom.flops / (dom_ms / 1e3) / 1e12
    dom_plan = plans[dom.name]
    kernel_key = (f"ffma_{dom_plan['bm']}x{dom_plan['bn']}x{dom_plan['bk']}_s{dom_plan['stages']}"
                  f"_{dom.name}")

    # End to end through the host-buffer entry point (pinned host memory).
    e2e = None
    if not args.no_e2e:
        hbufs = []
        for (w, _a, _b, _c, A, B) in bufs:
            hA = A.pin_memory()
            hB = B.pin_memory()
            hC = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
            hbufs.append((w, hA, hB, hC))

        def host_step():
            for (w, hA, hB, hC) in hbufs:
                st = mt.mt_sgemm_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), w.M, w.N, w.K,
                                      sptr, cfg)
                if st != mt.MT_OK:
                    raise mt.MtError(st, "mt_sgemm_host")
        host_step()  # warm the stream-ordered pool
        e2e_steps = max(1, min(args.steps, 5))
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        e2e_s = time.perf_counter() - t0
        if world > 1:
            import torch.distributed as dist
            t = torch.tensor([e2e_s], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e = {"value": world * flops_step * e2e_steps / e2e_s / 1e12, "unit": "TFLOP/s",
               "steps": e2e_steps,
               "h2d_bytes_per_step": sum(4 * (w.M * w.K + w.K * w.N) for (w, *_r) in hbufs),
               "d2h_bytes_per_step": sum(4 * w.M * w.N for (w, *_r) in hbufs),
               "api": "mt_sgemm_host"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        budget = float(os.environ.get("MT_ORACLE_BUDGET_S", "15"))
        tfl, secs, cores, desc = oracle_sample(1, budget)
        cpu = {"value": tfl, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc, "seconds": secs}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": " + ".join(f"sgemm {w.M}x{w.N}x{w.K} ({w.dist}, seed {w.seed})"
                                              for (w, *_r) in bufs),
                       "variant": "ffma" if not args.config else args.config,
                       "l2": "inputs larger than L2 (192 MB and 768 MB per GEMM vs 129 MB); "
                             "the 8192^3 GEMM between 4096^3 GEMMs evicts their operands",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "per_shape": per_shape,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_max,
                         "unit": "TFLOP/s", "frac": achieved / peak_max,
                         "traffic": load_traffic(kernel_key),
                         "kernel": kernel_key,
                         "peak_basis": f"{sms} SMs x 128 FP32 lanes x 2 flop x {sm_max:.0f} MHz "
                                       "(max SM clock)",
                         "frac_at_run_clock": achieved / peak_live if peak_live else None},
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": len(bufs) * args.steps,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mt", "reference"], default="mt")
    ap.add_argument("--workloads", nargs="*", help="override the step's workloads (by name)")
    ap.add_argument("--config", help="JSON of mt_config choices, e.g. '{\"bm\":128}'")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "mt":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
