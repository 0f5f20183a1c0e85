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

`variants` holds the other fp32 variant (3xTF32 on tcgen05, or FFMA when
--config selects 3xTF32) measured the same way in the same run.

`--impl reference` times the reference arm instead: the CPU oracle (fp64
accumulation, all host cores) on a bounded sample of rows of the same two
GEMMs, reported in the same metric.

Multi-GPU (torchrun): every rank runs the same step on its own GPU (replicas;
the GEMM has no exchange step), timing is the max over ranks and `value`
counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
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


def reduce_max(x: float, device: str = "cuda") -> float:
    """Max of x over the ranks of the default process group (x itself when
    there is none).  `device` holds the reduction tensor: "cuda" under NCCL,
    "cpu" under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, seconds: float) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return world * flops_per_step * steps / seconds / 1e12


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


# Nominal dense tensor rates (PFLOP/s) of the recipe's table: the TF32 peak
# is the measured bf16 peak scaled by their ratio.
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25

# Dense tf32 tensor throughput per SM and clock: half the bf16 rate of
# 8192 flop/clk/SM (one 128x256x16 bf16 MMA per 128 cycles), the ratio of
# the nominal dense figures above.
TF32_FLOP_PER_CLK_SM = 4096


def device_record(dev: int) -> dict:
    """The GPU, driver and software the run used."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    rec = {"name": props.name, "sms": props.multi_processor_count,
           "compute_capability": f"{props.major}.{props.minor}",
           "memory_gib": round(props.total_memory / 2 ** 30, 1),
           "torch": torch.__version__, "torch_cuda": torch.version.cuda}
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev), "--query-gpu=driver_version",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=20)
        rec["driver"] = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        rec["driver"] = None
    return rec


def tf32_clock_peak(sms: int, mhz: float) -> float:
    return sms * TF32_FLOP_PER_CLK_SM * mhz * 1e6 / 1e12


def launches_per_call(plan) -> int:
    """Kernels one library call launches: the GEMM (tf32x3: pack A, pack B,
    GEMM; FFMA with A staged K-major from a copy: the transposing copy of A,
    then the GEMM), plus the slice reduce when the plan splits K or the
    stream-K fix-up when it deals out stream-K runs."""
    base = 3 if plan["variant"] == 1 else 1
    if plan["variant"] == 0 and plan["pack_a"] == 5:
        base += 1  # the step's operands need no copy of B
    if plan["variant"] == 3 and not plan["vec_ab"]:
        base += 2  # the copy path pads both operands (the step's shapes never take it)
    second_pass = plan["split_k"] > 1 or plan.get("stream_k", 0) > 0
    return base + (1 if second_pass else 0)


def variant_of(cfg_json):
    cfg_json = cfg_json or {}
    if cfg_json.get("dtype"):
        return "tc16"  # 16-bit inputs: the tcgen05 kind::f16 kernel
    return cfg_json.get("variant", "ffma")


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

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, "cuda")

    shapes = [gemm_inputs.WORKLOADS[n] for n in (args.workloads or STEP_WORKLOADS)]
    main_cfg = json.loads(args.config) if args.config else {}
    bufs = []
    for w in shapes:
        A, B = gemm_inputs.make_workload(w)
        a, b = A.cuda(), B.cuda()
        c = torch.empty((w.M, w.N), device="cuda", dtype=torch.float32)
        bufs.append((w, a, b, c, A, B))
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    # SHA-256 of each workload's A then B bytes (fp32, row-major), so a result
    # can be matched to its exact inputs.
    input_hashes = {}
    for (w, _a, _b, _c, A, B) in bufs:
        h = hashlib.sha256()
        h.update(A.numpy().tobytes())
        h.update(B.numpy().tobytes())
        input_hashes[w.name] = h.hexdigest()
    flops_step = sum(w.flops for (w, *_r) in bufs)

    bufs16 = {}

    def operands(dtype):
        """The step's (w, a, b, c) with A and B in `dtype` ("bf16" / "f16",
        rounded from the fp32 inputs before any timing) or fp32 (None)."""
        if dtype is None:
            return [(w, a, b, c) for (w, a, b, c, _, _) in bufs]
        if dtype not in bufs16:
            tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
            bufs16[dtype] = [(w, a.to(tdt), b.to(tdt), c) for (w, a, b, c, _, _) in bufs]
        return bufs16[dtype]

    def measure(cfg_json, steps, warmup, clocks=None):
        """Per-launch CUDA-event times (ms) of every GEMM of `steps` steps.
        A "dtype" key ("bf16" / "f16") runs the 16-bit-input product
        (mt_gemm_mixed_general) on the same shapes."""
        cfg_json = dict(cfg_json or {})
        dtype = cfg_json.pop("dtype", None)
        cfg = mt.make_config(**cfg_json) if cfg_json else None
        ops = operands(dtype)
        code = {"bf16": mt.MT_DTYPE_BF16, "f16": mt.MT_DTYPE_F16}.get(dtype)

        def launch(w, a, b, c):
            if code is None:
                st = mt.mt_sgemm_ex(a.data_ptr(), b.data_ptr(), c.data_ptr(), w.M, w.N, w.K,
                                    sptr, cfg)
            else:
                st = mt.mt_gemm_mixed_general(code, 0, 0, w.M, w.N, w.K, 1.0, a.data_ptr(), w.K,
                                              b.data_ptr(), w.N, 0.0, c.data_ptr(), w.N, sptr,
                                              cfg)
            if st != mt.MT_OK:
                raise mt.MtError(st, f"gemm {w.name}")

        for _ in range(warmup):
            for (w, a, b, c) in ops:
                launch(w, a, b, c)
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in bufs] for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        gc.collect()
        gc.disable()  # no collection pass while the launches are enqueued
        try:
            if clocks:
                clocks.mark("t0")
            t0.record(stream)
            for s_ in range(steps):
                for i, (w, a, b, c) in enumerate(ops):
                    ev[s_][i][0].record(stream)
                    launch(w, a, b, c)
                    ev[s_][i][1].record(stream)
            t1.record(stream)
            torch.cuda.synchronize()
        finally:
            gc.enable()
        if clocks:
            clocks.mark("t1")
        total = max_over_ranks(t0.elapsed_time(t1))
        per = {w.name: [ev[s_][i][0].elapsed_time(ev[s_][i][1]) for s_ in range(steps)]
               for i, (w, *_r) in enumerate(bufs)}
        if mt.mt_device_status(sptr) != mt.MT_OK:
            raise RuntimeError("device status reported a kernel timeout")
        return total, per

    def plans_for(cfg_json):
        cfg_json = dict(cfg_json or {})
        dtype = cfg_json.pop("dtype", None)
        if dtype is None:
            return {w.name: mt.plan(w.M, w.N, w.K, a=a, b=b, c=c, **cfg_json)
                    for (w, a, b, c) in operands(None)}
        code = {"bf16": mt.MT_DTYPE_BF16, "f16": mt.MT_DTYPE_F16}[dtype]
        return {w.name: mt.plan_mixed(code, w.M, w.N, w.K, a=a, b=b, c=c, **cfg_json)
                for (w, a, b, c) in operands(dtype)}

    clocks = ClockSampler(dev).__enter__()
    total_ms, per_launch = measure(main_cfg, args.steps, args.warmup, clocks)
    clocks.__exit__(None, None, None)
    value = job_tflops(world, flops_step, args.steps, total_ms / 1e3)
    plans = plans_for(main_cfg)

    clk = clocks.summary()
    peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = clk["sm_max_mhz"] or peaks.get("sm_max_mhz") or SM_MAX_MHZ_FALLBACK
    ffma_peak = ffma_peak_tflops(sms, sm_max)
    ffma_live = ffma_peak_tflops(sms, clk["sm_mhz"]) if clk["sm_mhz"] else None
    bf16 = peaks.get("bf16_tflops")
    tf32_peak = (bf16 if bf16 else 1900.0) * NOMINAL_TF32_OVER_BF16
    tf32_basis = ("measured bf16 %.0f TFLOP/s (MEASURED_PEAKS.json) x nominal tf32/bf16 "
                  "1.1/2.25" % bf16) if bf16 else "fallback 1.9 PFLOP/s bf16 x 1.1/2.25"

    def shape_summary(per, plans_):
        out = {}
        for (w, *_r) in bufs:
            ms = statistics.median(per[w.name])
            tf = w.flops / (ms / 1e3) / 1e12
            out[w.name] = {"ms_median": ms, "tflops": tf,
                           "frac_of_ffma_peak_at_max_clock": tf / ffma_peak,
                           "frac_of_ffma_peak_at_run_clock": tf / ffma_live if ffma_live else None,
                           "plan": plans_[w.name]}
        return out

    per_shape = shape_summary(per_launch, plans)
    variant = variant_of(main_cfg)
    dom = max(bufs, key=lambda x: statistics.mean(per_launch[x[0].name]))[0]
    dom_ms = statistics.mean(per_launch[dom.name])
    dp = plans[dom.name]
    tf32_measured = {}

    def cublas_tf32_peak():
        """cuBLAS's TF32 GEMM (torch.matmul with TF32 on) on the step's
        largest operands, best of 5 by CUDA events after 3 warm-ups: the
        measured TF32 tensor rate of this GPU in this run."""
        if not tf32_measured:
            w, a, b, c = max(operands(None), key=lambda x: x[0].flops)
            prev = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = True
            try:
                for _ in range(3):
                    torch.matmul(a, b, out=c)
                best = float("inf")
                for _ in range(5):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    torch.matmul(a, b, out=c)
                    e1.record(stream)
                    e1.synchronize()
                    best = min(best, e0.elapsed_time(e1))
            finally:
                torch.backends.cuda.matmul.allow_tf32 = prev
            tf32_measured.update(value=w.flops / (best / 1e3) / 1e12, workload=w.name,
                                 ms=best)
        return tf32_measured

    def tf32_roofline(achieved, key):
        clock_peak = tf32_clock_peak(sms, sm_max)
        m = cublas_tf32_peak()
        return {"bound": "tensor", "achieved": achieved, "peak": m["value"],
                "unit": "TFLOP/s", "frac": achieved / m["value"],
                "traffic": load_traffic(key), "kernel": key,
                "peak_basis": "measured: cuBLAS TF32 GEMM (torch.matmul, TF32 on) on the "
                              f"{m['workload']} operands in this run, best of 5 "
                              f"({m['ms']:.3f} ms)",
                "nominal_peak": tf32_peak, "frac_of_nominal_peak": achieved / tf32_peak,
                "nominal_peak_basis": tf32_basis,
                "clock_peak": clock_peak, "frac_of_clock_peak": achieved / clock_peak,
                "clock_peak_basis": f"{sms} SMs x {TF32_FLOP_PER_CLK_SM} tf32 flop/clk "
                                    f"x {sm_max:.0f} MHz",
                "note": "achieved = 3 x 2MNK tf32 flops / time of the whole call (pack "
                        "kernels included, so it understates the GEMM kernel's own rate); "
                        "traffic is the GEMM kernel's.  cuBLAS's TF32 GEMM is a library "
                        "kernel, not the hardware's limit, so frac can read above 1; "
                        "frac_of_clock_peak is against the tensor pipe's rate at the "
                        "maximum clock"}

    def key_of(v, plan, name):
        return f"{v}_{plan['bm']}x{plan['bn']}x{plan['bk']}_s{plan['stages']}_{name}"

    bf16_peak = bf16 if bf16 else 1900.0
    bf16_basis = ("measured bf16 %.0f TFLOP/s burst (MEASURED_PEAKS.json)" % bf16_peak
                  if bf16 else "fallback 1900 TFLOP/s bf16")

    def tc16_roofline(achieved, key):
        return {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": achieved / bf16_peak, "traffic": load_traffic(key), "kernel": key,
                "peak_basis": bf16_basis,
                "note": "achieved = 2MNK / time of the whole call (split-tail reduce included)"}

    kernel_key = key_of(variant, dp, dom.name)
    if variant == "tf32x3":
        roofline = tf32_roofline(3 * dom.flops / (dom_ms / 1e3) / 1e12, kernel_key)
    elif variant == "tc16":
        roofline = tc16_roofline(dom.flops / (dom_ms / 1e3) / 1e12, kernel_key)
    else:
        achieved = dom.flops / (dom_ms / 1e3) / 1e12
        roofline = {"bound": "alu", "achieved": achieved, "peak": ffma_peak, "unit": "TFLOP/s",
                    "frac": achieved / ffma_peak, "traffic": load_traffic(kernel_key),
                    "kernel": kernel_key,
                    "peak_basis": f"{sms} SMs x 128 FP32 lanes x 2 flop x {sm_max:.0f} MHz "
                                  "(max SM clock)",
                    "note": "achieved = 2MNK / time of the whole call; with A staged "
                            "K-major from a copy the call includes the transposing copy "
                            "kernel, so it understates the GEMM kernel's own rate by that "
                            "kernel's share",
                    "frac_at_run_clock": achieved / ffma_live if ffma_live else None}

    # End to end through the host-buffer entry point (pinned host memory),
    # right after the device timing and before the variants: after the bf16
    # variant's power draw, steps of this loop were seen to stall (one step
    # +27 ms) while the link itself measured normal.
    e2e = None
    if main_cfg.get("dtype"):
        e2e = {"unavailable": "the host-buffer entry point takes fp32 inputs only"}
    elif not args.no_e2e:
        cfg = mt.make_config(**main_cfg) if main_cfg else None
        hbufs = []
        for (w, _a, _b, _c, A, B) in bufs:
            hbufs.append((w, A.pin_memory(), B.pin_memory(),
                          torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()))

        def host_step():
            # Each GEMM through the asynchronous host-buffer entry point (its
            # copies in overlap the previous GEMM's products), then one wait
            # for the step: the results are in the host buffers after it.
            for (w, hA, hB, hC) in hbufs:
                st = mt.mt_sgemm_host_async(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), w.M,
                                            w.N, w.K, sptr, cfg)
                if st != mt.MT_OK:
                    raise mt.MtError(st, "mt_sgemm_host_async")
            stream.synchronize()
        # Untimed warm-up steps, as for the device timing: the first calls on
        # freshly pinned host buffers and pool blocks run slower (measured on
        # GB300: the first two of each shape, up to 2x).
        for _ in range(max(2, args.warmup)):
            host_step()
        # The link this run got: pinned copies of the largest A, each way (the
        # host side of the link is shared with other jobs on the machine, so
        # e2e, which is bound by it, moves with it).
        big = max(hbufs, key=lambda x: x[0].M * x[0].K)
        dev_buf = torch.empty_like(big[1], device="cuda")
        link = {}
        for name, (dst, src) in (("h2d_gbs", (dev_buf, big[1])), ("d2h_gbs", (big[1], dev_buf))):
            dst.copy_(src, non_blocking=True)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            link[name] = big[1].numel() * 4 / (e0.elapsed_time(e1) / 1e3) / 1e9
        del dev_buf
        # The same K steps as the device timing (at most 100, about 2 s): the
        # box's host-copy path pauses for 30-55 ms about every 0.5 s, so a loop
        # much shorter than that meets a pause or not by chance.
        e2e_steps = max(1, min(args.steps, 100))
        barrier()
        step_s = []
        e2e_clocks = ClockSampler(dev).__enter__()
        # No garbage collection inside the timed loop (as timeit does): a
        # collection pass between two asynchronous calls leaves the GPU idle
        # until the next one is enqueued (seen as single steps ~30 ms long).
        gc.collect()
        gc.disable()
        try:
            e2e_clocks.mark("t0")
            t0 = time.perf_counter()
            for _ in range(e2e_steps):
                t_step = time.perf_counter()
                host_step()
                step_s.append(time.perf_counter() - t_step)
            e2e_s = max_over_ranks(time.perf_counter() - t0)
            e2e_clocks.mark("t1")
        finally:
            gc.enable()
        e2e_clocks.__exit__(None, None, None)
        e2e = {"value": job_tflops(world, flops_step, e2e_steps, e2e_s), "unit": "TFLOP/s",
               "steps": e2e_steps,
               "h2d_bytes_per_step": sum(4 * (w.M * w.K + w.K * w.N) for (w, *_r) in hbufs),
               "d2h_bytes_per_step": sum(4 * w.M * w.N for (w, *_r) in hbufs),
               "api": "mt_sgemm_host_async per GEMM, one stream synchronisation per step",
               "link": link,
               "step_ms": [round(t * 1e3, 3) for t in step_s],
               # Context for a step that stalled on the shared host: the same
               # metric over the median step (value stays total work / total time).
               "value_at_median_step": job_tflops(world, flops_step, 1,
                                                  statistics.median(step_s)),
               "clocks": e2e_clocks.summary()}


    # The other fp32 variant, measured in the same run for comparison.
    variants = {}
    if not args.no_variants:
        other = {"variant": "tf32x3"} if variant == "ffma" else {"variant": "ffma"}
        o_steps = max(1, min(args.steps, 10))
        o_total, o_per = measure(other, o_steps, max(1, min(args.warmup, 3)))
        o_val = job_tflops(world, flops_step, o_steps, o_total / 1e3)
        o_plans = plans_for(other)
        variants[other["variant"]] = {
            "value": o_val, "unit": "TFLOP/s", "steps": o_steps,
            "per_shape": shape_summary(o_per, o_plans),
            "tolerance": "5e-5*|A||B|" if other["variant"] == "tf32x3" else "1e-5*|A||B|"}
        if other["variant"] == "tf32x3":
            o_dom = max(bufs, key=lambda x: statistics.mean(o_per[x[0].name]))[0]
            o_ach = 3 * o_dom.flops / (statistics.mean(o_per[o_dom.name]) / 1e3) / 1e12
            variants["tf32x3"]["roofline"] = tf32_roofline(
                o_ach, key_of("tf32x3", o_plans[o_dom.name], o_dom.name))
        # Context, not a target: cuBLAS's fp32 GEMM (torch.matmul with TF32
        # off) on the same operands, timed the same way.
        tf32_prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        try:
            for (w, a, b, c) in operands(None):
                torch.matmul(a, b, out=c)
            cb_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in bufs] for _ in range(o_steps)]
            torch.cuda.synchronize()
            for s_ in range(o_steps):
                for i, (w, a, b, c) in enumerate(operands(None)):
                    cb_ev[s_][i][0].record(stream)
                    torch.matmul(a, b, out=c)
                    cb_ev[s_][i][1].record(stream)
            torch.cuda.synchronize()
        finally:
            torch.backends.cuda.matmul.allow_tf32 = tf32_prev
        cb_per = {w.name: [cb_ev[s_][i][0].elapsed_time(cb_ev[s_][i][1]) for s_ in range(o_steps)]
                  for i, (w, *_r) in enumerate(bufs)}
        variants["cublas_fp32"] = {
            "value": job_tflops(world, flops_step, o_steps,
                                sum(sum(v) for v in cb_per.values()) / 1e3),
            "unit": "TFLOP/s", "steps": o_steps, "impl": "torch.matmul, TF32 off (cuBLAS)",
            "per_shape": {w.name: {"ms_median": statistics.median(cb_per[w.name]),
                                   "tflops": w.flops / (statistics.median(cb_per[w.name]) / 1e3)
                                   / 1e12} for (w, *_r) in bufs}}
        if variant != "tc16":
            # bf16 inputs, fp32 accumulation and output (tcgen05 kind::f16).
            h = {"dtype": "bf16"}
            h_total, h_per = measure(h, o_steps, max(1, min(args.warmup, 3)))
            h_plans = plans_for(h)
            h_dom = max(bufs, key=lambda x: statistics.mean(h_per[x[0].name]))[0]
            variants["tc16_bf16"] = {
                "value": job_tflops(world, flops_step, o_steps, h_total / 1e3),
                "unit": "TFLOP/s", "steps": o_steps, "inputs": "A, B rounded to bf16; C fp32",
                "per_shape": shape_summary(h_per, h_plans),
                "tolerance": "5e-5*|A||B| against the 16-bit oracle",
                "roofline": tc16_roofline(
                    h_dom.flops / (statistics.mean(h_per[h_dom.name]) / 1e3) / 1e12,
                    key_of("tc16", h_plans[h_dom.name], h_dom.name))}

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
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if main_cfg.get("dtype") == "bf16" else
                     "f16" if main_cfg.get("dtype") == "f16" else "f32",
            "data": "synthetic",
            "config": {"workload": " + ".join(f"sgemm {w.M}x{w.N}x{w.K} ({w.dist}, seed {w.seed})"
                                              for (w, *_r) in bufs),
                       "variant": variant, "choices": main_cfg,
                       "l2": "inputs larger than L2 (192 MB and 768 MB per GEMM vs 129 MB); "
                             "the 8192^3 GEMM between 4096^3 GEMMs evicts their operands",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "inputs_sha256": input_hashes},
            "per_shape": per_shape,
            "roofline": roofline,
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": sum(launches_per_call(p) for p in plans.values()) * args.steps,
            "variants": variants,
            "cpu_baseline": cpu,
            "device": device_record(dev),
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
    ap.add_argument("--no-variants", action="store_true",
                    help="skip measuring the other fp32 variant")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "mt":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
