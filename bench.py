#!/usr/bin/env python
"""Benchmark: Stream-K + ABFT GEMM on the square bf16 sweep.

Workload: C = A B with m = n = k in {1024, 2048, 3072, 4096, 5120, 6144},
bf16 inputs drawn N(0,1)/sqrt(k) (seed 1), fp32 accumulation, bf16 output,
ABFT checksum verification on. One step runs the whole hot path on every
shape: skg_gemm calls with ABFT on (the library issues the encode pass and
the persistent Stream-K kernel, or one launch when the encode runs inside
it), each bracketed by CUDA events on the launching stream, with a 256 MiB
write before each call so none starts with its operands in the 129 MB L2.
Each shape is repeated within a step so that over the timed steps it gets
at least 20 launches and 200 ms of timed GEMM time; a shape's time is the
median of its launches. The main kernel alone (pre-encoded checksums) is
timed the same way in a separate loop for the roofline.

Metric: GEMM TFLOPS = 2mnk / time, geomean over the sweep, and its fraction
of the GB300 dense bf16 peak. The JSON line also carries the roofline of the
dominant kernel, the oracle CPU baseline, an end-to-end number through host
buffers, the launch count and the SM clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs the same sweep on its own GPU
(replicas: the GEMM has no exchange step); value aggregates all ranks.
"""
from __future__ import annotations

import argparse
import re
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2mnk/s) and % of GB300 dense bf16 peak; geomean over shape sweep"
WORKLOAD = ("square bf16 sweep m=n=k in {1024,2048,3072,4096,5120,6144}, "
            "N(0,1)/sqrt(k) inputs (seed 1), fp32 accumulate, bf16 out, ABFT verify on")
FLUSH_BYTES = 256 << 20
MIN_LAUNCHES = 20      # per shape, over the timed steps
MIN_TIMED_S = 0.2      # per shape: at least this much timed GEMM time
KERNEL_SOURCES = ("stream_decomposition_abft_gb300/csrc/skg_kernel.cuh",
                  "stream_decomposition_abft_gb300/csrc/skg_ptx.cuh",
                  "stream_decomposition_abft_gb300/csrc/skg_sched.cuh")


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed, so that a
    change to comments alone keeps the hash (the compiled kernel is the same)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), \
            d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


def geomean(xs):
    return math.exp(sum(math.log(x) for x in xs) / len(xs)) if xs else 0.0


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        out = os.environ.get("SKG_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out, f"clocks_rank{index}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index),
                                          f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- ours
def replica_value(sizes, times_ms, world, device):
    """Whole-job throughput of `world` replicas of the square sweep: each
    shape's time is the max over ranks (all_reduce MAX when world > 1), and
    the value is the geomean over shapes of world * 2 s^3 / that time, in
    TFLOPS. Returns (per-shape max times in ms, value)."""
    import torch
    times = list(times_ms)
    if world > 1:
        t = torch.tensor(times, dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        times = t.tolist()
    value = geomean([world * 2.0 * s ** 3 / t / 1e9 for s, t in zip(sizes, times)])
    return times, value


def run_ours(args, rank, world, local_rank):
    import torch
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm

    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    sms = skgemm.device_sm_count()
    opts = skgemm.opts_default(abft=1)                       # one ABFT GEMM call
    main_opts = skgemm.opts_default(abft=1, abft_preencoded=1)  # main kernel alone
    enc_opts = skgemm.opts_default(abft=1)

    problems = []
    for size in inputs.SQUARE_SIZES:
        p = inputs.square(size)
        A = p.A.to(dev)
        B = p.B.to(dev)
        C = torch.empty((size, size), dtype=torch.bfloat16, device=dev)
        ws = skgemm.Workspace(skgemm.workspace_size(size, size, size, opts), dev)
        problems.append(dict(size=size, p=p, A=A, B=B, C=C, ws=ws))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    plans = {pr["size"]: skgemm.launch_plan(pr["size"], pr["size"], pr["size"], opts)
             for pr in problems}
    sched_names = {v: k for k, v in skgemm.SCHED_NAMES.items()}

    def launch(pr, o):
        s = pr["size"]
        st = skgemm.gemm(s, s, s, 1.0, pr["A"].data_ptr(), s, pr["B"].data_ptr(), s, 0.0,
                         pr["C"].data_ptr(), s, skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0, o,
                         pr["ws"].ptr, pr["ws"].nbytes, sh)
        if st != skgemm.OK:
            raise skgemm.SkgError(st, "skg_gemm")

    def step(record):
        # One step: for every shape, pr["per_step"] times an L2 flush, then
        # the whole ABFT GEMM (encode pass + main kernel, issued by the
        # library) between events on the launching stream.
        for pr in problems:
            for _ in range(pr["per_step"] if record else 1):
                flush.zero_()
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                ev[0].record(stream)
                launch(pr, opts)
                ev[1].record(stream)
                pr["events" if record else "warm_events"].append(ev)

    for pr in problems:
        pr["events"], pr["warm_events"] = [], []
        pr["per_step"] = 1
    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    # Launches per shape and step: over the K timed steps every shape gets at
    # least MIN_LAUNCHES launches and MIN_TIMED_S of timed launches (median
    # of them per shape), whatever K is.
    for pr in problems:
        est = statistics.median(a.elapsed_time(b) for a, b in pr["warm_events"]) * 1e-3
        total = max(args.min_launches, math.ceil(args.min_timed_ms * 1e-3 / max(est, 1e-6)))
        pr["per_step"] = max(1, math.ceil(total / args.steps))
    for pr in problems:
        pr["ws"].report(reset=True)

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        step(True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()

    # The dominant kernel alone (roofline): the main kernel on pre-encoded
    # checksums, L2 flushed before each launch, CUDA events on this stream.
    main_reps = max(args.min_launches, 3 * args.steps)
    for pr in problems:
        s = pr["size"]
        st = skgemm.abft_encode(s, s, s, pr["A"].data_ptr(), s, pr["B"].data_ptr(), s,
                                skgemm.IN_BF16, enc_opts, pr["ws"].ptr, pr["ws"].nbytes, sh)
        if st != skgemm.OK:
            raise skgemm.SkgError(st, "skg_abft_encode")
        evs = []
        for _ in range(main_reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(pr, main_opts)
            e1.record(stream)
            evs.append((e0, e1))
        pr["main_events"] = evs
    torch.cuda.synchronize()

    per_shape = []
    total_main_ms = 0.0
    total_main_flops = 0.0
    abft = {"tiles_checked": 0, "detected": 0, "max_ratio_row": 0.0, "max_ratio_col": 0.0}
    for pr in problems:
        s = pr["size"]
        full = [e[0].elapsed_time(e[1]) for e in pr["events"]]
        main = [a.elapsed_time(b) for a, b in pr["main_events"]]
        t_full = statistics.median(full)
        t_main = statistics.median(main)
        flops = 2.0 * s * s * s
        per_shape.append({"m": s, "n": s, "k": s, "ms": round(t_full, 5),
                          "ms_main_kernel": round(t_main, 5), "launches": len(full),
                          "timed_ms": round(sum(full), 2),
                          "tflops": round(flops / t_full / 1e9, 2),
                          "tflops_main_kernel": round(flops / t_main / 1e9, 2)})
        total_main_ms += sum(main)
        total_main_flops += flops * len(main)
        rep = pr["ws"].report()
        abft["tiles_checked"] += rep.tiles_checked
        abft["detected"] += rep.detected
        abft["max_ratio_row"] = max(abft["max_ratio_row"], rep.max_ratio_row)
        abft["max_ratio_col"] = max(abft["max_ratio_col"], rep.max_ratio_col)

    times, value = replica_value([ps["m"] for ps in per_shape], [ps["ms"] for ps in per_shape],
                                 world, dev)

    e2e = measure_e2e(args, problems, dev, stream, opts, enc_opts)

    if rank != 0:
        return
    burst, sustained, hbm, peak_kind = peaks()
    props = torch.cuda.get_device_properties(dev)
    fmax = clocks.get("sm_max_mhz") or 2070.0
    spec_peak = props.multi_processor_count * 8192 * fmax * 1e6 / 1e12
    achieved = total_main_flops / (total_main_ms * 1e-3) / 1e12
    traffic = load_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sum(times), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "plan_per_shape": {str(sz): {"tile": f"{pl.tile_m}x{pl.tile_n}x64",
                                                "ctas": pl.ctas + pl.side_ctas,
                                                "cta_pairs": pl.cta_pair == 2,
                                                "sched": sched_names[pl.sched],
                                                "checksum_tiles": ("fused" if pl.fused_checksums
                                                                   else "separate launches"),
                                                "launches": ((1 if pl.encode_in_kernel else 2)
                                                             if pl.fused_checksums else 4)}
                                      for sz, pl in plans.items()},
                   "sms": sms,
                   "launches_per_shape_per_step": {str(pr["size"]): pr["per_step"]
                                                   for pr in problems},
                   "timing": "per shape: median event time of all its timed launches "
                             f"(>= {args.min_launches} launches and >= {args.min_timed_ms:.0f} ms)",
                   "l2": "flushed between launches (256 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_peak": {"measured_burst": round(100 * value / world / burst, 2),
                        "spec_at_max_clock": round(100 * value / world / spec_peak, 2),
                        "peak_measured_tflops": burst, "peak_spec_tflops": round(spec_peak, 1),
                        "peak_kind": peak_kind},
        "per_shape": per_shape,
        "roofline": {"bound": "tensor", "kernel": "skg_gemm_kernel (Stream-K mainloop + ABFT)",
                     "achieved": round(achieved, 2), "peak": burst,
                     "unit": "TFLOP/s", "frac": round(achieved / burst, 4),
                     "frac_geomean_per_shape": round(geomean(
                         [ps["tflops_main_kernel"] / burst for ps in per_shape]), 4),
                     "peak_source": f"{peak_kind} bf16 burst (MEASURED_PEAKS.json)",
                     "traffic": traffic},
        "abft": abft,
        "gpu_launches": args.steps * sum(
            pr["per_step"] * ((1 if plans[pr["size"]].encode_in_kernel else 2)
                              if plans[pr["size"]].fused_checksums else 4)
            for pr in problems),
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def measure_e2e(args, problems, dev, stream, opts, enc_opts):
    """Same metric through the public C ABI's host-buffer call, skg_gemm_host:
    every step copies that step's A and B from page-locked host memory into
    device staging, runs the ABFT GEMM and copies C back to host memory, all
    inside the timed region. Consecutive steps rotate over `--e2e-streams`
    streams (each with its own staging, workspace and host C), so one step's
    copies overlap the neighbouring steps' GEMM and opposite-direction copy, as
    a stream of independent calls would; the value is the steps' flops over
    the wall time of all of them."""
    import torch
    from stream_decomposition_abft_gb300 import skgemm
    steps = max(6, min(args.steps, 20))
    h2d = d2h = 0
    tf = []
    streams = [stream] + [torch.cuda.Stream(dev) for _ in range(max(1, args.e2e_streams) - 1)]
    ns = len(streams)
    o = skgemm.opts_default(abft=1)
    for pr in problems:
        s = pr["size"]
        hA = pr["p"].A.pin_memory()
        hB = pr["p"].B.pin_memory()
        lanes = []
        for st in streams:
            nst = skgemm.host_staging_size(s, s, s, skgemm.IN_BF16, skgemm.OUT_BF16)
            lanes.append(dict(
                stream=st,
                staging=torch.empty(nst, dtype=torch.uint8, device=dev),
                ws=skgemm.Workspace(skgemm.workspace_size(s, s, s, o), dev),
                hC=torch.empty((s, s), dtype=torch.bfloat16).pin_memory()))

        def issue(i):
            ln = lanes[i % ns]
            rc = skgemm.gemm_host(s, s, s, 1.0, hA.data_ptr(), s, hB.data_ptr(), s, 0.0,
                                  ln["hC"].data_ptr(), s, skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0,
                                  o, ln["staging"].data_ptr(), ln["staging"].numel(),
                                  ln["ws"].ptr, ln["ws"].nbytes, ln["stream"].cuda_stream)
            if rc != skgemm.OK:
                raise skgemm.SkgError(rc, "skg_gemm_host")

        for i in range(2 * ns):  # warm-up, every lane
            issue(i)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t0.record(streams[0])
        for st in streams[1:]:
            st.wait_event(t0)
        for i in range(steps):
            issue(i)
        for st in streams[1:]:
            e1 = torch.cuda.Event()
            e1.record(st)
            streams[0].wait_event(e1)
        t1 = torch.cuda.Event(enable_timing=True)
        t1.record(streams[0])
        torch.cuda.synchronize()
        for ln in lanes:
            rep = ln["ws"].report()
            if rep.detected or rep.status_bits:
                raise RuntimeError(f"e2e run at {s}: ABFT report {rep.detected} {rep.status_bits}")
        tf.append(2.0 * s ** 3 * steps / t0.elapsed_time(t1) / 1e9)
        h2d += hA.numel() * 2 + hB.numel() * 2
        d2h += s * s * 2
    return {"value": round(geomean(tf), 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "per_shape_tflops": [round(x, 2) for x in tf],
            "api": f"skg_gemm_host (host A, B, C; device staging), {ns} streams in turn"}


def load_traffic():
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    or None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "skg_gemm_kernel_square_sweep_traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch_mean")


# ---------------------------------------------------------------------------- oracle
def cpu_baseline(budget_s: float = 15.0, shapes=None):
    """The fp64 oracle as it stands, on a bounded sample of the sweep: for
    each shape, whole rows of C (every entry a k-long dot product), as many
    as fit in budget_s / len(shapes) seconds. Reported in TFLOPS."""
    import oracle
    from stream_decomposition_abft_gb300 import inputs
    shapes = shapes or inputs.SQUARE_SIZES
    oracle.build()
    per = budget_s / len(shapes)
    rates, rows_done = [], []

    def rows_of_c(p, lo, hi):
        s = p.n
        r = [i for i in range(lo, hi) for _ in range(s)]
        c = list(range(s)) * (hi - lo)
        t0 = time.perf_counter()
        oracle.gemm_entries(p.A, p.B, r, c)
        return time.perf_counter() - t0

    for size in shapes:
        p = inputs.square(size)
        dt = rows_of_c(p, 0, 1)                      # calibrate on one row
        more = max(0, min(size - 1, int((per - dt) / max(dt, 1e-6))))
        if more:
            dt += rows_of_c(p, 1, 1 + more)
        rates.append(2.0 * (1 + more) * size * size / dt / 1e12)
        rows_done.append(1 + more)
    return {"value": geomean(rates), "unit": "TFLOPS", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": "fp64 triple-loop oracle (OpenMP) on whole rows of C for each sweep shape: "
                      + ", ".join(f"{s}^3: {r} rows" for s, r in zip(shapes, rows_done)),
            "per_shape_tflops": [round(x, 8) for x in rates]}


def run_reference(args, rank):
    """The reference arm: the oracle timed on the host cores on bounded
    samples of the same workload, K steps after W warm-up steps."""
    if rank != 0:
        return
    import oracle
    from stream_decomposition_abft_gb300 import inputs
    oracle.build()
    probs = [inputs.square(s) for s in inputs.SQUARE_SIZES]
    rows_per_step = 1

    def one_step(i):
        ts = []
        for p in probs:
            s = p.m
            row = (i * 7919) % s
            r = [row] * s
            c = list(range(s))
            t0 = time.perf_counter()
            oracle.gemm_entries(p.A, p.B, r, c)
            ts.append(time.perf_counter() - t0)
        return ts

    for i in range(args.warmup):
        one_step(i)
    per = [[] for _ in probs]
    t0 = time.perf_counter()
    for i in range(args.steps):
        for j, t in enumerate(one_step(args.warmup + i)):
            per[j].append(t)
    wall = time.perf_counter() - t0
    rates = [2.0 * rows_per_step * p.m * p.m / statistics.mean(ts) / 1e12
             for p, ts in zip(probs, per)]
    value = geomean(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * wall / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": "one whole row of C per shape per step",
                       "parallelism": "oracle on the host cores"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.threads(),
                             "kind": "oracle",
                             "sample": "one whole row of C per sweep shape per step"},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def ncu_target(args):
    """Profiling target (no timing): every sweep shape's ABFT GEMM through
    skg_gemm, `--steps` times, with the library's default plan; with
    `--workload hostile`, the quantisation-hostile shapes' plain GEMMs
    (automatic plan) instead."""
    import torch
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    sh = torch.cuda.current_stream().cuda_stream
    if args.workload == "hostile":
        for (m, n, k) in inputs.HOSTILE_SHAPES:
            p = inputs.hostile(m, n, k)
            A, B, C = p.A.to(dev), p.B.to(dev), p.C0.to(dev)
            o = skgemm.opts_default()
            ws = skgemm.Workspace(skgemm.workspace_size(m, n, k, o), dev)
            for _ in range(args.steps):
                st = skgemm.gemm(m, n, k, p.alpha, A.data_ptr(), k, B.data_ptr(), k, p.beta,
                                 C.data_ptr(), n, skgemm.IN_F16, skgemm.OUT_F16, 0, 0, o,
                                 ws.ptr, ws.nbytes, sh)
                if st != skgemm.OK:
                    raise skgemm.SkgError(st, "skg_gemm")
            torch.cuda.synchronize()
            print((m, n, k), skgemm.launch_shape(m, n, k, o), flush=True)
        return
    if args.shape:
        # Given shapes, bf16 with ABFT (or fp16 without, with --plain), the
        # library's default plan.
        for spec in args.shape.split(","):
            m, n, k = (int(x) for x in spec.split("x"))
            dt = "f16" if args.plain else "bf16"
            al, bl = int(args.a_col), int(args.b_nmajor)
            p = inputs.make_problem(m, n, k, seed=5, in_dtype=dt, out_dtype=dt,
                                    law_a="normal", law_b="normal", a_layout=al, b_layout=bl)
            A, B = p.A.to(dev), p.B.to(dev)
            C = torch.empty((m, n), dtype=A.dtype, device=dev)
            o = skgemm.opts_default(abft=0 if args.plain else 1)
            ws = skgemm.Workspace(skgemm.workspace_size_layout(m, n, k, al, bl, o), dev)
            code = skgemm.IN_F16 if args.plain else skgemm.IN_BF16
            out = skgemm.OUT_F16 if args.plain else skgemm.OUT_BF16
            for _ in range(args.steps):
                st = skgemm.gemm(m, n, k, 1.0, A.data_ptr(), A.stride(0), B.data_ptr(),
                                 B.stride(0), 0.0, C.data_ptr(), n, code, out, al, bl, o, ws.ptr,
                                 ws.nbytes, sh)
                if st != skgemm.OK:
                    raise skgemm.SkgError(st, "skg_gemm")
            torch.cuda.synchronize()
            print((m, n, k), skgemm.launch_shape(m, n, k, o), flush=True)
        return
    opts = skgemm.opts_default(abft=1)
    sizes = [int(x) for x in args.sizes.split(",")] if args.sizes else list(inputs.SQUARE_SIZES)
    for size in sizes:
        p = inputs.square(size)
        A, B = p.A.to(dev), p.B.to(dev)
        C = torch.empty((size, size), dtype=torch.bfloat16, device=dev)
        ws = skgemm.Workspace(skgemm.workspace_size(size, size, size, opts), dev)
        for _ in range(args.steps):
            st = skgemm.gemm(size, size, size, 1.0, A.data_ptr(), size, B.data_ptr(), size, 0.0,
                             C.data_ptr(), size, skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0, opts,
                             ws.ptr, ws.nbytes, sh)
            if st != skgemm.OK:
                raise skgemm.SkgError(st, "skg_gemm")
        torch.cuda.synchronize()
        if ws.report().detected:
            raise RuntimeError("ABFT reported a fault on a clean run")
        print(size, skgemm.launch_shape(size, size, size, opts), flush=True)


def write_traffic(csv_path):
    """Turn an ncu CSV of the main kernel over `--ncu-target --steps S` into
    profiles/skg_gemm_kernel_square_sweep_traffic.json, stamped with the
    current kernel-source hash (bench.py reports traffic only while it holds)."""
    import csv
    from collections import defaultdict
    from stream_decomposition_abft_gb300 import inputs
    rows = list(csv.reader(open(csv_path)))
    hi = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    hdr, data = rows[hi], rows[hi + 1:]
    idi, mi, vi = hdr.index("ID"), hdr.index("Metric Name"), hdr.index("Metric Value")
    per = defaultdict(dict)
    for r in data:
        per[int(r[idi])][r[mi]] = float(r[vi].replace(",", ""))
    launches = [per[i] for i in sorted(per)]
    reps = len(launches) // len(inputs.SQUARE_SIZES)
    out = {"kernel_hash": kernel_hash(), "source_csv": os.path.basename(csv_path),
           "per_shape": []}
    tot = []
    for j, size in enumerate(inputs.SQUARE_SIZES):
        ls = launches[j * reps:(j + 1) * reps]
        rd = statistics.mean(x["dram__bytes_read.sum"] for x in ls)
        wr = statistics.mean(x["dram__bytes_write.sum"] for x in ls)
        alg = 2 * size * size * 2 + size * size * 2
        out["per_shape"].append({"size": size, "dram_read": rd, "dram_write": wr,
                                 "algorithmic_bytes": alg, "ratio": (rd + wr) / alg})
        tot.append(rd + wr)
    out["dram_bytes_per_launch_mean"] = statistics.mean(tot)
    path = os.path.join(ROOT, "profiles", "skg_gemm_kernel_square_sweep_traffic.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(path)


# ---------------------------------------------------------------------------- other workloads
def _time_launch(fn, flush, reps, stream):
    """Median event time (ms) of fn() over reps launches, L2 flushed before each."""
    import torch
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts)


def workload_hostile(args):
    """Quantisation-hostile fp16 shapes (alpha 1.5, beta 0.5): time, plan and
    the spread of per-CTA busy time ((max - min) / max of end - start, from
    %globaltimer; median over 7 launches), for the automatic plan, for
    128 x 128 tiles with the model's schedule and grid (the tile the
    workload is stated for), and for the page's evaluated configuration
    (two-tile hybrid on every SM, 128 x 128 tiles)."""
    import torch
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sms = skgemm.device_sm_count()
    burst = peaks()[0]
    names = {v: k for k, v in skgemm.SCHED_NAMES.items()}
    out = []
    for (m, n, k) in inputs.HOSTILE_SHAPES:
        p = inputs.hostile(m, n, k)
        A, B = p.A.to(dev), p.B.to(dev)
        C0 = p.C0.to(dev)
        C = C0.clone()
        for label, kw in (("auto", {}), ("model_128x128", dict(tile_n=128, cta_pair=1)),
                          ("sk2_dp_all_sms_128x128",
                           dict(sched="sk2_dp", grid=sms, tile_n=128, cta_pair=1))):
            opts = skgemm.opts_default(**kw)
            tn, g, sc = skgemm.launch_shape(m, n, k, opts)
            pl = skgemm.launch_plan(m, n, k, opts)
            nclk = 7
            clk = torch.zeros(nclk, 2 * g, dtype=torch.int64, device=dev)
            ws = skgemm.Workspace(skgemm.workspace_size(m, n, k, opts), dev)

            def launch():
                C.copy_(C0)
                st = skgemm.gemm(m, n, k, p.alpha, A.data_ptr(), k, B.data_ptr(), k, p.beta,
                                 C.data_ptr(), n, skgemm.IN_F16, skgemm.OUT_F16, 0, 0, opts,
                                 ws.ptr, ws.nbytes, sh)
                if st != skgemm.OK:
                    raise skgemm.SkgError(st, "skg_gemm")

            ms = _time_launch(launch, flush, max(5, args.steps // 10), stream)
            # Per-CTA busy time of nclk launches issued back to back (as the
            # timed ones are), each with its own clock buffer.
            for i in range(nclk):
                opts.cta_clock = clk[i].data_ptr()
                flush.zero_()
                launch()
            opts.cta_clock = None
            torch.cuda.synchronize()
            spreads, spreads90 = [], []
            for i in range(nclk):
                c = clk[i].view(g, 2).cpu().double()
                busy = (c[:, 1] - c[:, 0])
                spreads.append(float((busy.max() - busy.min()) / busy.max()))
                q = torch.quantile(busy, torch.tensor([0.05, 0.95], dtype=busy.dtype))
                spreads90.append(float((q[1] - q[0]) / busy.max()))
            spread = statistics.median(spreads)
            spread90 = statistics.median(spreads90)
            out.append({"m": m, "n": n, "k": k, "plan": label,
                        "tile": f"{pl.tile_m}x{tn}x64", "cta_pairs": pl.cta_pair == 2,
                        "grid": g, "sched": names[sc], "ms": round(ms, 4),
                        "tflops": round(2.0 * m * n * k / ms / 1e9, 1),
                        "pct_of_peak_measured": round(100 * 2.0 * m * n * k / ms / 1e9 / burst, 1),
                        "sm_busy_spread": round(spread, 4),
                        "sm_busy_spread_p5_p95": round(spread90, 4), "sms_used": g,
                        "status_bits": ws.report().status_bits})
    print(json.dumps({"workload": "hostile fp16 shapes, alpha 1.5 beta 0.5 (C0 U[-1,1])",
                      "unit": "TFLOPS", "results": out}), flush=True)


def workload_random(args):
    """The 1000-shape random fp16 sweep (m, n, k log-uniform on [128, 8192],
    rounded up to 128, seed 3): geomean and 5th percentile of the fraction of
    the measured bf16 peak. Timing only (inputs drawn on the device); parity
    on a subset is in the GPU tests."""
    import torch
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    burst = peaks()[0]
    shapes = inputs.random_shapes(1000)
    if args.limit:
        shapes = shapes[:args.limit]
    opts = skgemm.opts_default()
    big = max(max(m * k, n * k, m * n) for (m, n, k) in shapes)
    pool = torch.empty(3 * big, dtype=torch.float16, device=dev).uniform_(-1, 1)
    ws = skgemm.Workspace(max(skgemm.workspace_size(m, n, k, opts) for (m, n, k) in shapes), dev)
    fracs = []
    for (m, n, k) in shapes:
        A = pool[:m * k]
        B = pool[big:big + n * k]
        C = pool[2 * big:2 * big + m * n]

        def launch():
            st = skgemm.gemm(m, n, k, 1.0, A.data_ptr(), k, B.data_ptr(), k, 0.0, C.data_ptr(), n,
                             skgemm.IN_F16, skgemm.OUT_F16, 0, 0, opts, ws.ptr, ws.nbytes, sh)
            if st != skgemm.OK:
                raise skgemm.SkgError(st, "skg_gemm")

        ms = _time_launch(launch, flush, 3, stream)
        fracs.append(2.0 * m * n * k / ms / 1e9 / burst)
    fs = sorted(fracs)
    p5 = fs[max(0, int(0.05 * len(fs)) - 1)]
    print(json.dumps({"workload": f"random fp16 sweep, {len(shapes)} shapes (seed 3)",
                      "geomean_frac_of_peak_measured": round(geomean(fracs), 4),
                      "p5_frac_of_peak_measured": round(p5, 4),
                      "median_frac": round(statistics.median(fracs), 4),
                      "peak_tflops_measured": burst}), flush=True)


def workload_mlp(args):
    """Transformer-MLP bf16 shapes with ABFT on: time with ABFT on and off,
    and a fault-injection campaign of `--launches` launches per shape with one
    seeded single-bit flip of one fp32 accumulator per 100 launches (launch
    ids, tile, row, column and bit drawn from seed 4). Each injected flip is
    classified in advance with the oracle's fault model (must-detect /
    harmless / grey) from the oracle's value of that accumulator."""
    import torch
    import oracle
    from oracle import abft_ref as ab
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    results = []
    for (m, n, k) in inputs.MLP_SHAPES:
        p = inputs.mlp(m, n, k)
        A, B = p.A.to(dev), p.B.to(dev)
        C = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        o_on = skgemm.opts_default(abft=1)
        o_off = skgemm.opts_default()
        ws = skgemm.Workspace(skgemm.workspace_size(m, n, k, o_on), dev)
        tn, g, sc = skgemm.launch_shape(m, n, k, o_on)

        def launch(o):
            st = skgemm.gemm(m, n, k, 1.0, A.data_ptr(), k, B.data_ptr(), k, 0.0, C.data_ptr(), n,
                             skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0, o, ws.ptr, ws.nbytes, sh)
            if st != skgemm.OK:
                raise skgemm.SkgError(st, "skg_gemm")

        t_on = _time_launch(lambda: launch(o_on), flush, 5, stream)
        t_off = _time_launch(lambda: launch(o_off), flush, 5, stream)
        ws.report(reset=True)
        ids, gen = inputs.fault_plan(args.launches, seed=4)
        tiles_m, tiles_n = (m + 127) // 128, (n + tn - 1) // tn
        Anp, Bnp = p.A.double().numpy(), p.B.double().numpy()
        camp = {"injected": 0, "must_detect": 0, "detected": 0, "located": 0, "corrected": 0,
                "harmless_or_grey": 0}
        for launch_id in range(args.launches):
            if launch_id not in ids:
                launch(o_on)
                continue
            while True:
                tile = int(torch.randint(0, tiles_m * tiles_n, (1,), generator=gen))
                row = int(torch.randint(0, 128, (1,), generator=gen))
                col = int(torch.randint(0, tn, (1,), generator=gen))
                bit = int(torch.randint(0, 32, (1,), generator=gen))
                tm, tnn = tile // tiles_n, tile % tiles_n     # row-major raster for the campaign
                gi, gj = tm * 128 + row, tnn * tn + col
                if gi >= m or gj >= n:
                    continue
                v = float(oracle.gemm_entries(p.A, p.B, [gi], [gj])[0])
                ma, mb = ab.tile_maxima(Anp, Bnp, tm, tnn, 128, tn)
                kind, _ = ab.classify_flip(v, bit, ab.default_tau(k, tn, ma, mb), 1e-6 * abs(v))
                if kind != ab.GREY:
                    break
            oi = skgemm.opts_default(abft=1, inject_tile=tile, inject_row=row, inject_col=col,
                                     inject_bit=bit, raster_band=tiles_n)
            launch(oi)
            rep = ws.report(reset=True)
            camp["injected"] += 1
            if kind == ab.MUST_DETECT:
                camp["must_detect"] += 1
                recs = [rep.records[i] for i in range(min(rep.n_records, skgemm.MAX_RECORDS))]
                hit = [r for r in recs if r.injected]
                if rep.detected:
                    camp["detected"] += 1
                if hit and (hit[0].tile, hit[0].row, hit[0].col) == (tile, row, col):
                    camp["located"] += 1
                    after = float(hit[0].after)
                    if abs(after - float(hit[0].clean_value)) <= 1e-3 * math.sqrt(k) * \
                            float(p.A.abs().max()) * float(p.B.abs().max()):
                        camp["corrected"] += 1
            else:
                camp["harmless_or_grey"] += 1
        pl = skgemm.launch_plan(m, n, k, o_on)
        results.append({"m": m, "n": n, "k": k,
                        "plan": f"{pl.tile_m}x{tn}x64 ctas={g}"
                                + (" (CTA pairs)" if pl.cta_pair == 2 else ""),
                        "ms_abft_on": round(t_on, 4), "ms_abft_off": round(t_off, 4),
                        "abft_overhead_pct": round(100 * (t_on / t_off - 1), 2),
                        "tflops_abft_on": round(2.0 * m * n * k / t_on / 1e9, 1),
                        "campaign": camp, "launches": args.launches})
    print(json.dumps({"workload": "MLP bf16 shapes, ABFT on, one seeded bit flip per 100 "
                                  "launches", "results": results}), flush=True)


def workload_fp64(args):
    """fp64 GEMM rate: skg_gemm_f64 against the library DGEMM (torch.matmul on
    double, which is cuBLAS), m = n = k in {2048, 4096, 8192}, inputs resident
    (the fp64 peak the fp64 kernel is compared with)."""
    import torch
    from stream_decomposition_abft_gb300 import _build, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    res = []
    for s in (2048, 4096, 8192):
        gen = torch.Generator(device=dev).manual_seed(s)
        a = torch.randn(s, s, dtype=torch.float64, device=dev, generator=gen)
        b = torch.randn(s, s, dtype=torch.float64, device=dev, generator=gen)
        c = torch.empty(s, s, dtype=torch.float64, device=dev)
        o = skgemm.opts_default()
        ws = skgemm.Workspace(skgemm.workspace_size_f64(s, s, s, o), dev)

        def ours():
            st = skgemm.gemm_f64(s, s, s, 1.0, a.data_ptr(), s, b.data_ptr(), s, 0.0, c.data_ptr(),
                                 s, o, ws.ptr, ws.nbytes, sh)
            if st != skgemm.OK:
                raise skgemm.SkgError(st, "skg_gemm_f64")

        row = {"size": s}
        for name, fn in (("torch_matmul_fp64", lambda: torch.matmul(a, b)), ("skg_gemm_f64", ours)):
            for _ in range(3):
                fn()
            ts = []
            for _ in range(max(5, args.steps // 20)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3)
            row[name + "_tflops"] = round(2.0 * s ** 3 / statistics.median(ts) / 1e12, 3)
        res.append(row)
    print(json.dumps({"workload": "fp64 GEMM rate (inputs resident)", "results": res}), flush=True)


def workload_stagger(args):
    """k staggering (skg_opts_t.stagger) A/B on the power-of-two square shapes,
    bf16, with and without ABFT, L2 flushed before each launch: median
    event time (us) per stagger value."""
    import torch
    from stream_decomposition_abft_gb300 import _build, inputs, skgemm
    if not os.path.exists(skgemm.LIB_PATH):
        _build.build()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    out = []
    for size in (1024, 2048, 4096, 8192):
        p = inputs.make_problem(size, size, size, seed=1, in_dtype="bf16", out_dtype="bf16",
                                law_a="normal", law_b="normal", scale_a=size ** -0.5,
                                scale_b=size ** -0.5)
        A, B = p.A.to(dev), p.B.to(dev)
        C = torch.empty((size, size), dtype=torch.bfloat16, device=dev)
        row = {"size": size}
        for abft in (0, 1):
            for sg in (0, 2, 4, 8):
                o = skgemm.opts_default(abft=abft, stagger=sg)
                ws = skgemm.Workspace(skgemm.workspace_size(size, size, size, o), dev)

                def launch():
                    st = skgemm.gemm(size, size, size, 1.0, A.data_ptr(), size, B.data_ptr(), size,
                                     0.0, C.data_ptr(), size, skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0,
                                     o, ws.ptr, ws.nbytes, sh)
                    if st != skgemm.OK:
                        raise skgemm.SkgError(st, "skg_gemm")

                for _ in range(4):
                    flush.zero_()
                    launch()
                row[f"{'abft' if abft else 'plain'}_stagger{sg}_us"] = round(
                    1e3 * _time_launch(launch, flush, 30, stream), 2)
                if ws.report().detected:
                    raise RuntimeError("ABFT reported a fault on a clean run")
        out.append(row)
    print(json.dumps({"workload": "k staggering A/B, square bf16", "results": out}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--min-launches", type=int, default=MIN_LAUNCHES,
                    help="square sweep: timed launches per shape, at least")
    ap.add_argument("--min-timed-ms", type=float, default=MIN_TIMED_S * 1e3,
                    help="square sweep: timed GEMM time per shape, at least (ms); 0 for "
                         "profiling runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end leg's host-buffer calls rotate over")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ncu-target", action="store_true",
                    help="run the sweep GEMMs untimed (profiling target)")
    ap.add_argument("--sizes", default="", help="with --ncu-target: comma-separated sizes")
    ap.add_argument("--shape", default="",
                    help="with --ncu-target: MxNxK[,MxNxK...] (bf16 with ABFT, or --plain)")
    ap.add_argument("--a-col", action="store_true",
                    help="with --ncu-target --shape: A stored column-major (k x m)")
    ap.add_argument("--b-nmajor", action="store_true",
                    help="with --ncu-target --shape: B stored k x n")
    ap.add_argument("--plain", action="store_true",
                    help="with --ncu-target --shape: fp16 without ABFT")
    ap.add_argument("--write-traffic", default="",
                    help="write the traffic JSON from an ncu CSV of the main kernel")
    ap.add_argument("--workload", choices=["square", "hostile", "random", "mlp", "fp64", "stagger"],
                    default="square", help="square = the metric's sweep (default)")
    ap.add_argument("--limit", type=int, default=0, help="random: first N shapes only")
    ap.add_argument("--launches", type=int, default=300, help="mlp: launches per shape")
    args = ap.parse_args()
    if args.write_traffic:
        write_traffic(args.write_traffic)
        return
    if args.ncu_target:
        ncu_target(args)
        return
    if args.workload != "square":
        {"hostile": workload_hostile, "random": workload_random, "mlp": workload_mlp,
         "fp64": workload_fp64, "stagger": workload_stagger}[args.workload](args)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
