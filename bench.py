#!/usr/bin/env python
"""Throughput benchmark of the tiled tensor-core GEMM (one JSON line on stdout).

Default workload: bf16 GEMM 8192 x 8192 x 8192, A row-major, B column-major,
alpha = 1, beta = 0, fp32 accumulation, bf16 out; A, B i.i.d. uniform[-1, 1]
(SplitMix64 stream, seed 1).  One step = one ttc_gemm call (the whole hot
path: tile scheduling, TMA staging, tcgen05 mainloop, fused epilogue).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ttc|reference]

--impl reference times the CPU oracle (the plain triple loop) on the host
cores, on a bounded sample of the same workload, in the same metric.
For N > 1 (torchrun) each rank runs an independent replica (the GEMM has no
exchange step); the value is the work of all ranks over the slowest rank's time.
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

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_spec(name):
    import synth
    if name in synth.TRANSPOSE_WORKLOADS:
        return dict(synth.TRANSPOSE_WORKLOADS[name], kind="transpose")
    if name in synth.CONV_WORKLOADS:
        return dict(synth.CONV_WORKLOADS[name], kind="conv")
    try:
        return synth.workload(name)
    except (KeyError, ValueError):
        names = synth.all_workload_names() + sorted(synth.TRANSPOSE_WORKLOADS) + sorted(synth.CONV_WORKLOADS)
        raise SystemExit(f"unknown workload {name}; choose from {names}")


def algorithmic_bytes(spec):
    """Bytes the GEMM must move at least once: A, B, D, plus C when beta != 0 and the bias
    (for every batch of a batched workload; the bias once)."""
    return spec.get("batch", 1) * single_problem_bytes(spec) + (spec["N"] * 4 if spec.get("dist_bias") else 0)


def single_problem_bytes(spec):
    M, N, K = spec["M"], spec["N"], spec["K"]
    ein = 1 if spec["dtype"] == "i8" else 2
    eout = 4 if spec["dtype"] == "i8" else 2
    b = (M * K + K * N) * ein + M * N * eout
    if spec.get("beta", 0.0) != 0.0:
        b += M * N * eout
    return b


L2_BYTES = 129e6


def rotation_copies(nbytes):
    """Input copies the timed loop cycles through: 1 when one step's data is
    already beyond twice the L2, else enough copies to cycle ~3x the L2, so
    every step starts with its inputs evicted and no foreign kernel (an L2
    flush) runs between the timed launches."""
    if nbytes > 2 * L2_BYTES:
        return 1
    return int(-(-3 * L2_BYTES // nbytes))


def l2_note(nbytes):
    n = rotation_copies(nbytes)
    if n == 1:
        return "inputs larger than L2 (no flush)"
    return f"inputs rotated over {n} copies ({n * nbytes / 1e6:.0f} MB, > 2x L2), no flush"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def timed_loops(steps, launch, stream):
    """The timed region: `steps` launches back to back with one event pair
    around the loop (the throughput `value` comes from this pass), then the
    same loop with an event pair around every launch (the per-launch kernel
    durations the roofline uses; the events' own cost stays out of `value`).
    launch(i) enqueues step i.  Returns (total_ms, kern_ms, launches of the
    first pass)."""
    import torch
    import tiled_tensor_core_02_gb300 as ttc
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = ttc.ttc_launch_count()
    t0.record(stream)
    for i in range(steps):
        launch(i)
    t1.record(stream)
    torch.cuda.synchronize()
    launches = ttc.ttc_launch_count() - n0
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        starts[i].record(stream)
        launch(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in zip(starts, ends)], launches


# Below this per-launch time the back-to-back pass is replayed from a CUDA
# graph: the host cannot submit launches that short as fast as they run.
GRAPH_BELOW_MS = 0.05


def timed_graph(steps, launch_on, stream):
    """The back-to-back pass from a CUDA graph holding the K steps' launches:
    captured on a side stream, replayed once untimed, then replayed on
    `stream` between one event pair.  launch_on(i, h) enqueues step i on the
    stream whose handle is h.  Returns (total_ms, launches in the graph)."""
    import torch
    import tiled_tensor_core_02_gb300 as ttc
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    n0 = ttc.ttc_launch_count()
    with torch.cuda.graph(g, stream=cap):
        for i in range(steps):
            launch_on(i, cap.cuda_stream)
    launches = ttc.ttc_launch_count() - n0
    stream.wait_stream(cap)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), launches


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample_rate(p, spec, budget_s, threads=0):
    """Times the oracle on a bounded sample of whole output rows (full K each).

    The sample grows by 4x until it takes a quarter of the budget, then is
    scaled to the budget.  Returns (flop/s, description, threads used, seconds)."""
    import numpy as np

    import oracle
    alpha, beta, act = spec["alpha"], spec["beta"], spec["act"]
    total = p.M * p.N

    def timed(n):
        ii = (np.arange(n, dtype=np.int64) // p.N) % p.M
        jj = np.arange(n, dtype=np.int64) % p.N
        t0 = time.perf_counter()
        _, _, used = oracle.gemm_elements(p, ii, jj, alpha=alpha, beta=beta, act=act, nthreads=threads)
        return time.perf_counter() - t0, used

    n = min(256, total)
    dt, used = timed(n)
    while dt < budget_s / 4 and n < total:
        n = min(total, n * 4)
        dt, used = timed(n)
    if dt < budget_s and n < total:
        n = int(min(total, n * budget_s / max(dt, 1e-6)))
        dt, used = timed(n)
    flops = 2.0 * n * p.K
    desc = f"{n} output elements ({n / p.N:.2f} rows x {p.N} cols, full K={p.K}) in {dt:.2f} s"
    return flops / dt, desc, used, dt


def run_reference(args, spec, name):
    """The CPU oracle, as it stands, on a bounded sample of the workload (rank 0 only)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth
    p, alpha, beta, act = synth.make(spec)
    import oracle
    oracle.build()
    import numpy as np
    # Calibrate once, then give every step the same fixed sample of output
    # elements, sized so the whole run takes about a minute and a half.
    rate, _, used, _ = oracle_sample_rate(p, spec, 3.0)
    per_step_s = min(10.0, max(0.01, 90.0 / max(1, args.steps + args.warmup)))
    n = int(max(64, min(p.M * p.N, rate * per_step_s / (2.0 * p.K))))
    ii = (np.arange(n, dtype=np.int64) // p.N) % p.M
    jj = np.arange(n, dtype=np.int64) % p.N
    rates = []
    t_all = None
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            t_all = time.perf_counter()
        t0 = time.perf_counter()
        _, _, used = oracle.gemm_elements(p, ii, jj, alpha=alpha, beta=beta, act=act)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            rates.append(2.0 * n * p.K / dt)
    wall = time.perf_counter() - t_all
    value = statistics.median(rates) / 1e12
    descs = [f"{n} output elements per step ({n / p.N:.3f} rows x {p.N} cols, full K={p.K})"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[spec["dtype"]],
        "data": "synthetic", "config": config_of(spec, name, world),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": used, "kind": "oracle",
                         "sample": descs[-1] if descs else ""},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


METRIC = "GEMM TFLOPS (bf16 8192^3) and % of GB300 dense tensor peak, 1 GPU"
DTYPE_NAME = {"bf16": "bf16", "f16": "f16", "i8": "int8"}


def config_of(spec, name, world):
    return {"workload": name, "batch": spec.get("batch", 1), "M": spec["M"], "N": spec["N"], "K": spec["K"],
            "dtype": spec["dtype"],
            "layoutA": spec["layoutA"], "layoutB": spec["layoutB"], "alpha": spec["alpha"],
            "beta": spec["beta"], "act": spec["act"], "bias": bool(spec.get("dist_bias")),
            "seed": spec["seed"], "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": l2_note(algorithmic_bytes(spec))}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="bf16_8192")
    ap.add_argument("--impl", default="ttc", choices=["ttc", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pair", type=int, default=0, choices=[0, 1, 2],
                    help="kernel choice: 0 planner, 1 CTA-pair kernel where it applies, 2 single-CTA kernel")
    ap.add_argument("--pair-tile-n", type=int, default=0, choices=[0, 256, 224, 192, 128],
                    help="CTA-pair tile width: 0 planner, else forced")
    ap.add_argument("--group-m", type=int, default=0, help="tile rows per rasterization group (0: default)")
    ap.add_argument("--graph", default="auto", choices=["auto", "on", "off"],
                    help="GEMM workloads: replay the back-to-back pass from a CUDA graph (auto: when a "
                         "launch takes under 50 us)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    spec = workload_spec(args.workload)
    name = args.workload
    if spec.get("kind") == "transpose":
        return run_transpose_reference(args, spec, name) if args.impl == "reference" else \
            run_transpose(args, spec, name)
    if spec.get("kind") == "conv":
        return run_conv_reference(args, spec, name) if args.impl == "reference" else run_conv(args, spec, name)
    if args.impl == "reference":
        return run_reference(args, spec, name)

    import numpy as np
    import torch

    world, rank, local = dist_setup()
    import synth
    import tiled_tensor_core_02_gb300 as ttc
    from tiled_tensor_core_02_gb300 import _build
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    ttc.load()
    ttc.ttc_set_knob("pair", args.pair)
    ttc.ttc_set_knob("pair_tile_n", args.pair_tile_n)
    ttc.ttc_set_knob("group_m", args.group_m)

    p, alpha, beta, act = synth.make(spec)
    M, N, K = p.M, p.N, p.K
    nbatch = spec.get("batch", 1)
    flops = 2.0 * M * N * K * nbatch
    esz_out = 4 if p.dtype == "i8" else 2

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    if nbatch > 1:
        # batches packed back to back (strides = one matrix each)
        probs = synth.make_batch(spec)
        hA = np.concatenate([q.A for q in probs])
        hB = np.concatenate([q.B for q in probs])
        hC = np.concatenate([q.C for q in probs]) if p.C is not None else None
    else:
        hA, hB, hC = p.A, p.B, p.C
    ncopy = rotation_copies(algorithmic_bytes(spec))
    copies = []
    for _ in range(ncopy):
        copies.append((dev(hA), dev(hB), dev(hC) if hC is not None else None,
                       torch.empty(nbatch * M * N, dtype=torch.int32 if p.dtype == "i8" else torch.int16,
                                   device="cuda")))
    A, B, C, D = copies[0]
    bias = dev(p.bias) if p.bias is not None else None
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    stream_h = s
    lay = {"row": ttc.ROW_MAJOR, "col": ttc.COL_MAJOR}

    # Operands TMA cannot read (odd pitches) are repacked by ttc_gemm_ws into a
    # caller-owned workspace, and a D whose rows are not 16-byte aligned is
    # staged through an aligned copy there; the workspace is allocated here,
    # outside the timed region, the copies themselves run inside every step.
    ws_bytes = ttc.ttc_gemm_workspace_size_staged(M, N, K, A.data_ptr(), p.lda, lay[p.layoutA], B.data_ptr(),
                                                  p.ldb, lay[p.layoutB], D.data_ptr(), N, ttc.DTYPE[p.dtype])
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")

    def step(Ap=A, Bp=B, Cp=C, Dp=D, h=None):
        s = stream_h if h is None else h
        if nbatch > 1:
            st = ttc.ttc_gemm_strided_batched(
                nbatch, M, N, K, Ap.data_ptr(), p.lda, p.A.size, lay[p.layoutA], Bp.data_ptr(), p.ldb, p.B.size,
                lay[p.layoutB], Cp.data_ptr() if (Cp is not None and beta != 0.0) else None, p.ldc,
                p.C.size if p.C is not None else 0, Dp.data_ptr(), N, M * N, alpha, beta,
                bias.data_ptr() if bias is not None else None, ttc.ACT[act], ttc.DTYPE[p.dtype], s)
            if st != 0:
                raise ttc.TTCError(st)
            return
        st = ttc.ttc_gemm_ws(M, N, K, Ap.data_ptr(), p.lda, lay[p.layoutA], Bp.data_ptr(), p.ldb,
                             lay[p.layoutB], Cp.data_ptr() if (Cp is not None and beta != 0.0) else None,
                             p.ldc, Dp.data_ptr(), N, alpha, beta,
                             bias.data_ptr() if bias is not None else None, ttc.ACT[act],
                             ttc.DTYPE[p.dtype], ws.data_ptr() if ws_bytes else None, ws_bytes, s)
        if st != 0:
            raise ttc.TTCError(st)

    for i in range(args.warmup):
        step(*copies[i % ncopy])
    torch.cuda.synchronize()
    if ttc.ttc_get_device_error(s) != 0:
        raise SystemExit("device error during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    total_ms, kern_ms, launches = timed_loops(args.steps, lambda i: step(*copies[(args.warmup + i) % ncopy]),
                                              stream)
    launch_mode = "stream"
    if args.graph == "on" or (args.graph == "auto" and statistics.median(kern_ms) < GRAPH_BELOW_MS):
        total_ms, launches = timed_graph(args.steps,
                                         lambda i, h: step(*copies[(args.warmup + i) % ncopy], h=h), stream)
        launch_mode = "cuda_graph"

    barrier(world)
    clocks = sampler.stop()
    if ttc.ttc_get_device_error(stream_h) != 0:
        raise SystemExit("device error during the timed region")
    total_ms = max_over_ranks(total_ms, world)
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    avg_kernel_s = statistics.mean(kern_ms) * 1e-3

    peaks, peak_src = load_peaks()
    # fp16 and bf16 share the dense tensor rate; int8 runs on the same fp16
    # tensor pipe (exact for int8 values).  A timed region of a second or more
    # of back-to-back launches runs under the power cap: compare it with the
    # sustained figure, a shorter one with the burst figure.
    sustained = total_ms >= 1000.0
    peak_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = peaks[peak_key]
    alg_bytes = algorithmic_bytes(spec)
    ridge = peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / alg_bytes >= ridge:
        achieved = flops / avg_kernel_s / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "peak_source": f"{peak_src} {peak_key}"}
    else:
        achieved = alg_bytes / avg_kernel_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs"}
    roofline.update({"traffic": load_traffic(name), "alg_bytes": alg_bytes,
                     "alg_flops": flops, "intensity_flop_per_byte": flops / alg_bytes,
                     "tflops": flops / avg_kernel_s / 1e12, "achieved_gbs": alg_bytes / avg_kernel_s / 1e9,
                     "kernel_ms_mean": statistics.mean(kern_ms),
                     "kernel_ms_median": statistics.median(kern_ms), "kernel_ms_min": min(kern_ms)})
    # the same ratio over the back-to-back pass (its launches overlap their
    # prologues with the previous launch's tail): the steady-state rate
    b2b_s = total_ms * 1e-3 / args.steps
    b2b = flops / b2b_s / 1e12 if roofline["bound"] == "tensor" else alg_bytes / b2b_s / 1e9
    roofline.update({"achieved_back_to_back": b2b, "frac_back_to_back": b2b / roofline["peak"]})

    # ---------------------------------------------------------------- end to end
    # Every step uploads its inputs from pinned host memory, runs the GEMM and
    # reads the result back.  Copies run on their own streams so that step
    # i+1's upload and step i-1's download overlap step i's kernel.
    hA = torch.empty(A.numel(), dtype=A.dtype, pin_memory=True).copy_(A)
    hB = torch.empty(B.numel(), dtype=B.dtype, pin_memory=True).copy_(B)
    use_c = C is not None and beta != 0.0
    hC = torch.empty(C.numel(), dtype=C.dtype, pin_memory=True).copy_(C) if use_c else None
    hD = [torch.empty(D.numel(), dtype=D.dtype, pin_memory=True) for _ in range(2)]
    dA = [torch.empty_like(A) for _ in range(2)]
    dB = [torch.empty_like(B) for _ in range(2)]
    dC = [torch.empty_like(C) for _ in range(2)] if use_c else [None, None]
    dD = [D, torch.empty_like(D)]
    h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size() + \
        (hC.numel() * hC.element_size() if use_c else 0)
    d2h = hD[0].numel() * hD[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used_once = [False, False]

    def e2e_step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if used_once[j]:
                s_in.wait_event(comp_done[j])
            dA[j].copy_(hA, non_blocking=True)
            dB[j].copy_(hB, non_blocking=True)
            if use_c:
                dC[j].copy_(hC, non_blocking=True)
            in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        if used_once[j]:
            stream.wait_event(out_done[j])
        step(dA[j], dB[j], dC[j], dD[j])
        comp_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            hD[j].copy_(dD[j], non_blocking=True)
            out_done[j].record(s_out)
        used_once[j] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    stream.wait_event(out_done[(args.e2e_steps - 1) & 1])
    stream.wait_event(out_done[args.e2e_steps & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = flops * args.e2e_steps * world / (e2e_ms * 1e-3) / 1e12
    if not np.array_equal(hD[(args.e2e_steps - 1) & 1].numpy(), D.cpu().numpy()):
        raise SystemExit("end-to-end result differs from the device-timed result")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, used, _ = oracle_sample_rate(p, spec, args.cpu_budget)
        cpu = {"value": rate / 1e12, "unit": "TFLOPS", "cores": used, "kind": "oracle", "sample": desc}
        # the same oracle on one host core
        rate1, desc1, _, _ = oracle_sample_rate(p, spec, args.cpu_budget / 3, threads=1)
        cpu["single_core"] = {"value": rate1 / 1e12, "unit": "TFLOPS", "cores": 1, "sample": desc1}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[p.dtype], "data": "synthetic",
            "config": config_of(spec, name, world), "launch": launch_mode,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "workspace_bytes": ws_bytes,
            "input_copies": ncopy,
            "clocks": clocks,
            "frac_of_peak": value / peak,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def kernel_source_hash(kind="gemm"):
    """Hash of the sources the workload's kernel is built from: the transpose
    kernel's own two files, or every other file under csrc/ for the GEMM."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "tiled_tensor_core_02_gb300", "csrc", "*"))):
        is_t = os.path.basename(f).startswith("transpose.")
        if is_t != (kind == "transpose"):
            continue
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(name, kind="gemm"):
    """DRAM bytes (read + write) per launch of the workload's kernel from the
    committed ncu summary; None when there is none or the kernel sources
    changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f).get(name)
    except (OSError, ValueError):
        return None
    if not d or d.get("source_hash") != kernel_source_hash(kind):
        return None
    return d.get("bytes_per_launch")


# ---------------------------------------------------------------- transpose workload

T_METRIC = "transpose GB/s (read + write), 1 GPU"
T_DTYPE = {1: "u8", 2: "bf16 bits (u16)", 4: "f32 bits (u32)", 8: "u64"}


def t_config(spec, name, world):
    return {"workload": name, "rows": spec["rows"], "cols": spec["cols"], "elem_bytes": spec["elem_bytes"],
            "seed": spec["seed"], "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "inputs larger than L2 (no flush)"}


def oracle_transpose_rate(spec, budget_s):
    """Times oracle.transpose on whole source rows, growing the sample until it
    takes about the budget.  Returns (bytes/s, description, seconds)."""
    import oracle
    import synth
    rows, cols, eb = spec["rows"], spec["cols"], spec["elem_bytes"]
    n = 1
    while True:
        src = synth.transpose_input(n, cols, eb, seed=spec["seed"])
        t0 = time.perf_counter()
        oracle.transpose(src, n, cols, cols, n)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or n >= rows:
            break
        n = min(rows, n * 4)
    if dt < budget_s and n < rows:
        n = int(min(rows, max(1, n * budget_s / max(dt, 1e-6))))
        src = synth.transpose_input(n, cols, eb, seed=spec["seed"])
        t0 = time.perf_counter()
        oracle.transpose(src, n, cols, cols, n)
        dt = time.perf_counter() - t0
    nbytes = 2.0 * n * cols * eb
    return nbytes / dt, f"{n} source rows x {cols} cols ({nbytes / 1e6:.1f} MB moved) in {dt:.2f} s", dt


def run_transpose_reference(args, spec, name):
    """The oracle's transpose, as it stands, on a bounded sample (rank 0 only)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import oracle
    import synth
    rows, cols, eb = spec["rows"], spec["cols"], spec["elem_bytes"]
    rate, _, _ = oracle_transpose_rate(spec, 2.0)
    per_step_s = min(10.0, max(0.01, 90.0 / max(1, args.steps + args.warmup)))
    n = int(max(1, min(rows, rate * per_step_s / (2.0 * cols * eb))))
    src = synth.transpose_input(n, cols, eb, seed=spec["seed"])
    rates, t_all = [], None
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            t_all = time.perf_counter()
        t0 = time.perf_counter()
        oracle.transpose(src, n, cols, cols, n)
        if i >= args.warmup:
            rates.append(2.0 * n * cols * eb / (time.perf_counter() - t0))
    wall = time.perf_counter() - t_all
    value = statistics.median(rates) / 1e9
    line = {
        "impl": "reference", "metric": T_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": T_DTYPE[eb],
        "data": "synthetic", "config": t_config(spec, name, world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} source rows x {cols} cols per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_transpose(args, spec, name):
    """Out-of-place transpose of a rows x cols matrix, one ttc_transpose call per step."""
    import numpy as np
    import torch

    world, rank, local = dist_setup()
    import synth
    import tiled_tensor_core_02_gb300 as ttc
    from tiled_tensor_core_02_gb300 import _build
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    ttc.load()
    rows, cols, eb = spec["rows"], spec["cols"], spec["elem_bytes"]
    tdt = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[eb]
    sdt = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}[eb]
    src_np = synth.transpose_input(rows, cols, eb, seed=spec["seed"])
    S = torch.from_numpy(src_np.view(sdt)).cuda()
    D = torch.empty(rows * cols, dtype=tdt, device="cuda")
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    nbytes = 2.0 * rows * cols * eb

    def step(Sp=S, Dp=D):
        st = ttc.ttc_transpose(rows, cols, Sp.data_ptr(), cols, Dp.data_ptr(), rows, eb, s)
        if st != 0:
            raise ttc.TTCError(st, "ttc_transpose")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    total_ms, kern_ms, launches = timed_loops(args.steps, lambda i: step(), stream)
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, world)
    value = nbytes * args.steps * world / (total_ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    achieved = nbytes / (statistics.mean(kern_ms) * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs",
                "traffic": load_traffic(name, "transpose"), "alg_bytes": nbytes,
                "kernel_ms_mean": statistics.mean(kern_ms), "kernel_ms_median": statistics.median(kern_ms),
                "kernel_ms_min": min(kern_ms)}

    # end to end: upload the source from pinned memory, transpose, read back;
    # copies on their own streams overlap the neighbouring steps' kernels
    hS = torch.empty(S.numel(), dtype=tdt, pin_memory=True).copy_(S)
    hD = [torch.empty(D.numel(), dtype=tdt, pin_memory=True) for _ in range(2)]
    dS = [torch.empty_like(S) for _ in range(2)]
    dD = [D, torch.empty_like(D)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done, comp_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    used_once = [False, False]

    def e2e_step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if used_once[j]:
                s_in.wait_event(comp_done[j])
            dS[j].copy_(hS, non_blocking=True)
            in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        if used_once[j]:
            stream.wait_event(out_done[j])
        step(dS[j], dD[j])
        comp_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            hD[j].copy_(dD[j], non_blocking=True)
            out_done[j].record(s_out)
        used_once[j] = True

    e2e_steps = max(4, min(args.e2e_steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(out_done[0])
    stream.wait_event(out_done[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = nbytes * e2e_steps * world / (e2e_ms * 1e-3) / 1e9
    if not torch.equal(hD[(e2e_steps - 1) & 1], D.cpu()):
        raise SystemExit("end-to-end result differs from the device-timed result")
    if ttc.ttc_get_device_error(s) != 0:
        raise SystemExit("device error")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, _ = oracle_transpose_rate(spec, args.cpu_budget)
        cpu = {"value": rate / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {
            "metric": T_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": T_DTYPE[eb], "data": "synthetic",
            "config": t_config(spec, name, world), "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": rows * cols * eb,
                    "d2h_bytes_per_step": rows * cols * eb},
            "gpu_launches": launches, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0



# ---------------------------------------------------------------- convolution workload

C_METRIC = "implicit-GEMM convolution TFLOPS, 1 GPU"


def conv_problem(spec):
    import synth
    kw = {k: v for k, v in spec.items() if k != "kind"}
    return synth.ConvProblem(**kw)


def conv_config(cp, name, world):
    return {"workload": name, "N": cp.N, "H": cp.H, "W": cp.W, "C": cp.C, "K": cp.K, "R": cp.R, "S": cp.S,
            "pad": list(cp.pad), "stride": list(cp.stride), "dil": list(cp.dil), "dtype": cp.dtype,
            "gemm_view": {"M": cp.M, "N": cp.K, "K": cp.R * cp.S * cp.C},
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": l2_note(conv_bytes(cp))}


def conv_bytes(cp):
    """Bytes the convolution must move at least once: X, the filters and D."""
    return 2 * (cp.N * cp.H * cp.W * cp.C + cp.K * cp.R * cp.S * cp.C + cp.M * cp.K)


def conv_oracle_rate(cp, budget_s, threads=0):
    """Times oracle.conv_elements on whole output rows; returns (flop/s, description, threads)."""
    import numpy as np

    import oracle
    kg = cp.R * cp.S * cp.C

    def timed(n):
        mm = (np.arange(n, dtype=np.int64) // cp.K) % cp.M
        kk = np.arange(n, dtype=np.int64) % cp.K
        t0 = time.perf_counter()
        _, _, used = oracle.conv_elements(cp, mm, kk, nthreads=threads)
        return time.perf_counter() - t0, used

    n = min(256, cp.M * cp.K)
    dt, used = timed(n)
    while dt < budget_s / 4 and n < cp.M * cp.K:
        n = min(cp.M * cp.K, n * 4)
        dt, used = timed(n)
    if dt < budget_s and n < cp.M * cp.K:
        n = int(min(cp.M * cp.K, n * budget_s / max(dt, 1e-6)))
        dt, used = timed(n)
    return 2.0 * n * kg / dt, f"{n} output elements ({n / cp.K:.2f} pixels x {cp.K} channels, R S C = {kg}) in {dt:.2f} s", used


def run_conv_reference(args, spec, name):
    """The oracle's convolution, as it stands, on a fixed per-step sample (rank 0 only)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import numpy as np

    import oracle
    oracle.build()
    cp = conv_problem(spec)
    kg = cp.R * cp.S * cp.C
    rate, _, used = conv_oracle_rate(cp, 3.0)
    per_step_s = min(10.0, max(0.01, 90.0 / max(1, args.steps + args.warmup)))
    n = int(max(64, min(cp.M * cp.K, rate * per_step_s / (2.0 * kg))))
    mm = (np.arange(n, dtype=np.int64) // cp.K) % cp.M
    kk = np.arange(n, dtype=np.int64) % cp.K
    rates, t_all = [], None
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            t_all = time.perf_counter()
        t0 = time.perf_counter()
        _, _, used = oracle.conv_elements(cp, mm, kk)
        if i >= args.warmup:
            rates.append(2.0 * n * kg / (time.perf_counter() - t0))
    wall = time.perf_counter() - t_all
    value = statistics.median(rates) / 1e12
    line = {
        "impl": "reference", "metric": C_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cp.dtype, "data": "synthetic",
        "config": conv_config(cp, name, world),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": used, "kind": "oracle",
                         "sample": f"{n} output elements per step ({n / cp.K:.2f} pixels x {cp.K} channels)"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_conv(args, spec, name):
    """One ttc_conv2d_fprop call per step."""
    import numpy as np
    import torch

    world, rank, local = dist_setup()
    import tiled_tensor_core_02_gb300 as ttc
    from tiled_tensor_core_02_gb300 import _build
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    ttc.load()
    cp = conv_problem(spec)
    kg = cp.R * cp.S * cp.C
    flops = 2.0 * cp.M * cp.K * kg

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()

    ncopy = rotation_copies(conv_bytes(cp))
    copies = [(dev(cp.X), dev(cp.Wt), torch.empty(cp.M * cp.K, dtype=torch.int16, device="cuda"))
              for _ in range(ncopy)]
    X, Wt, D = copies[0]
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream

    def step(Xp=X, Wp=Wt, Dp=D):
        st = ttc.ttc_conv2d_fprop(*cp.dims(), Xp.data_ptr(), Wp.data_ptr(), None, cp.K, Dp.data_ptr(), cp.K,
                                  1.0, 0.0, None, ttc.ACT["none"], ttc.DTYPE[cp.dtype], s)
        if st != 0:
            raise ttc.TTCError(st, "ttc_conv2d_fprop")

    for i in range(args.warmup):
        step(*copies[i % ncopy])
    torch.cuda.synchronize()
    if ttc.ttc_get_device_error(s) != 0:
        raise SystemExit("device error during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    total_ms, kern_ms, launches = timed_loops(args.steps, lambda i: step(*copies[(args.warmup + i) % ncopy]),
                                              stream)
    barrier(world)
    clocks = sampler.stop()
    if ttc.ttc_get_device_error(s) != 0:
        raise SystemExit("device error during the timed region")
    total_ms = max_over_ranks(total_ms, world)
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak_key = "bf16_tflops_sustained" if total_ms >= 1000.0 else "bf16_tflops"
    achieved = flops / (statistics.mean(kern_ms) * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks[peak_key], "unit": "TFLOP/s",
                "frac": achieved / peaks[peak_key], "peak_source": f"{peak_src} {peak_key}",
                "traffic": load_traffic(name), "alg_bytes": conv_bytes(cp), "alg_flops": flops,
                "intensity_flop_per_byte": flops / conv_bytes(cp),
                "kernel_ms_mean": statistics.mean(kern_ms), "kernel_ms_median": statistics.median(kern_ms),
                "kernel_ms_min": min(kern_ms)}

    # end to end: upload input and filters from pinned memory, convolve, read D back
    hX = torch.empty(X.numel(), dtype=X.dtype, pin_memory=True).copy_(X)
    hW = torch.empty(Wt.numel(), dtype=Wt.dtype, pin_memory=True).copy_(Wt)
    hD = [torch.empty(D.numel(), dtype=D.dtype, pin_memory=True) for _ in range(2)]
    dX, dW = [torch.empty_like(X) for _ in range(2)], [torch.empty_like(Wt) for _ in range(2)]
    dD = [D, torch.empty_like(D)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done, comp_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    used_once = [False, False]

    def e2e_step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if used_once[j]:
                s_in.wait_event(comp_done[j])
            dX[j].copy_(hX, non_blocking=True)
            dW[j].copy_(hW, non_blocking=True)
            in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        if used_once[j]:
            stream.wait_event(out_done[j])
        step(dX[j], dW[j], dD[j])
        comp_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            hD[j].copy_(dD[j], non_blocking=True)
            out_done[j].record(s_out)
        used_once[j] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    stream.wait_event(out_done[0])
    stream.wait_event(out_done[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = flops * args.e2e_steps * world / (e2e_ms * 1e-3) / 1e12
    if not torch.equal(hD[(args.e2e_steps - 1) & 1], D.cpu()):
        raise SystemExit("end-to-end result differs from the device-timed result")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, used = conv_oracle_rate(cp, args.cpu_budget)
        cpu = {"value": rate / 1e12, "unit": "TFLOPS", "cores": used, "kind": "oracle", "sample": desc}
        rate1, desc1, _ = conv_oracle_rate(cp, args.cpu_budget / 3, threads=1)
        cpu["single_core"] = {"value": rate1 / 1e12, "unit": "TFLOPS", "cores": 1, "sample": desc1}
    if rank == 0:
        line = {
            "metric": C_METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cp.dtype, "data": "synthetic",
            "config": conv_config(cp, name, world), "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": 2 * (X.numel() + Wt.numel()),
                    "d2h_bytes_per_step": 2 * D.numel()},
            "gpu_launches": launches, "clocks": clocks, "input_copies": ncopy,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
