"""Benchmark of the single-GPU Purlin collective datapath.

Default workload: AllGather bf16, R = 8 rank buffers x 8 Mi elements each
(16 MiB per rank; each of the 8 outputs holds all 8 contributions, 128 MiB).
A step is one collective call over inputs already resident in HBM.

Metric: effective HBM GB/s = (bytes every rank buffer must read + bytes every
rank buffer must write) / device time.  Timing: W warm-up steps, then K
steps on the library's stream, timed with CUDA events.  When the step's
inputs are larger than the L2 the device reports (the ReduceScatter and
AllToAllV workloads), the K steps run back to back between one pair of
events, since no input can survive in L2 from one step to the next;
otherwise (the default AllGather: 128 MiB of inputs) every step has its own
events and an L2 flush (a 512 MiB write) comes before it, outside the events
(``--flush`` forces this mode).  Barrier + synchronize around the whole timed
loop; max over ranks.

Extra keys: ``roofline`` (the throughput kernel against the measured HBM
copy bandwidth), ``cpu_baseline`` (the CPU oracle on a bounded sample),
``e2e`` (the same metric with host buffers: pinned H2D of the inputs, the
call, D2H of every output, all inside the timed region), ``clocks``
(nvidia-smi samples taken during the timed region).

``--impl reference`` times the CPU oracle instead (the pages publish no
runnable reference; the oracle is the reference arm).  ``--all`` also runs
every workload and the latency sweep and writes them to ``--report``.
"""
from __future__ import annotations

import argparse
import hashlib
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

import workloads  # noqa: E402

L2_FLUSH_BYTES = 512 << 20
# purlin_launch_info.variant -> the kernel that ran
KERNEL_OF_VARIANT = {1: "purlin_latency_kernel", 2: "purlin_throughput_kernel",
                     3: "purlin_throughput_kernel", 4: "purlin_vcounts_kernel",
                     5: "purlin_packet_ar_kernel"}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ["collective_datapath_atom_gb300/csrc/kernels.cu",
                  "collective_datapath_atom_gb300/csrc/ring_kernel.cuh",
                  "collective_datapath_atom_gb300/csrc/snac.cuh",
                  "collective_datapath_atom_gb300/csrc/atom.cuh"]


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    e = d.get(workload_name)
    if not e or e.get("kernel_src_sha") != kernel_source_sha():
        return None
    return int(e["dram_bytes_per_launch"])


# ------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sms.append(float(parts[0]))
                maxs.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs),
                "reasons": sorted(reasons), "samples": len(sms)}


# --------------------------------------------------------------- setup ----

def setup_workload(name: str, device, elements: int = 0):
    """Device inputs/outputs and a closure that runs one call.  `elements`
    (if set) replaces the elements per rank of the AllGather, ReduceScatter
    or AllReduce workload, or the tokens per rank of the MoE dispatch: a
    smaller case of the same kernel for profiling."""
    import dataclasses

    import torch

    if name == workloads.AG_BF16_R8_8MI.name:
        w = workloads.AG_BF16_R8_8MI
        if elements:
            w = dataclasses.replace(w, n=elements, name=f"allgather_bf16_R8_n{elements}")
        ins = workloads.inputs_for(w)
        out_elems = [w.R * w.n] * w.R
        call = ("all_gather", w.n)
    elif name == workloads.RS_BF16_R8_128MI.name:
        w = workloads.RS_BF16_R8_128MI
        if elements:
            w = dataclasses.replace(w, n=elements - elements % 8,
                                    name=f"reducescatter_bf16_R8_n{elements}")
        ins = workloads.inputs_for(w)
        out_elems = [w.n // w.R] * w.R
        call = ("reduce_scatter", w.n)
    elif name == workloads.A2AV_BF16_R8_MOE.name:
        w = workloads.A2AV_BF16_R8_MOE
        tokens = elements or workloads.MOE_TOKENS   # `elements`: tokens per rank here
        if elements:
            w = dataclasses.replace(w, n=tokens * workloads.MOE_HIDDEN,
                                    name=f"alltoallv_bf16_R8_{tokens}tok_x7168_zipf1.2")
        C, ins = workloads.moe_dispatch(tokens=tokens)
        counts = (C * workloads.MOE_HIDDEN).reshape(-1)
        out_elems = [int(counts.reshape(8, 8)[:, d].sum()) for d in range(8)]
        call = ("all_to_all_v", counts.tolist())
    elif name == workloads.AR_F32_R8_4096.name:
        w = workloads.AR_F32_R8_4096
        ins = workloads.inputs_for(w)
        out_elems = [w.n] * w.R
        call = ("all_reduce", w.n)
    elif name.startswith("allreduce_bf16_R8_b"):
        batch = int(name.rsplit("_b", 1)[1].split("x")[0])
        w = workloads.ar_sweep_workload(batch)
        ins = workloads.inputs_for(w)
        out_elems = [w.n] * w.R
        call = ("all_reduce", w.n)
    else:
        raise SystemExit(f"unknown workload {name}")
    tdt = torch.float32 if w.dtype == workloads.F32 else torch.int16
    src = [torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).to(device)
           for x in ins]
    dst = [torch.empty(m, dtype=tdt, device=device) for m in out_elems]
    in_bytes = sum(x.nbytes for x in ins)
    out_bytes = sum(m * workloads.ELEM_BYTES[w.dtype] for m in out_elems)
    return w, ins, src, dst, call, in_bytes + out_bytes, in_bytes, out_bytes


def make_runner(P, ctx, w, call):
    coll, arg = call
    f = getattr(P, "purlin_" + coll)

    def run(src, dst):
        f(ctx, src, dst, arg, w.dtype)
    return run


# ---------------------------------------------------------- CPU oracle ----

def oracle_sample(w, per_rank: int):
    """A bounded sample of workload `w` for the CPU oracle: the same
    collective, dtype and R with `per_rank` elements per rank (the AllToAllV
    count matrix scaled down in proportion).  Returns (fn, bytes, desc)."""
    import oracle

    R = w.R
    if w.collective == "all_gather":
        ins = workloads.normals(w.seed, R, per_rank, w.dtype)
        return (lambda: oracle.all_gather(ins, w.dtype), R * per_rank * 2 * (1 + R),
                f"AllGather bf16 R=8, {per_rank} elements per rank")
    if w.collective == "reduce_scatter":
        n = per_rank - per_rank % R
        ins = workloads.normals(w.seed, R, n, w.dtype)
        return (lambda: oracle.reduce_scatter(ins, w.dtype), R * n * 2 + n * 2,
                f"ReduceScatter bf16 R=8, {n} elements per rank")
    if w.collective == "all_to_all_v":
        C, _ = workloads.moe_dispatch(payload=False)
        scale = per_rank / float(workloads.MOE_TOKENS * workloads.MOE_HIDDEN)
        counts = np.floor(C * workloads.MOE_HIDDEN * scale).astype(np.int64)
        ins = [workloads.normals(w.seed + s, 1, int(counts[s].sum()), w.dtype)[0]
               for s in range(R)]
        return (lambda: oracle.all_to_all_v(ins, counts, w.dtype), 2 * int(counts.sum()) * 2,
                f"AllToAllV bf16 R=8, MoE count matrix scaled to {per_rank} elements per rank")
    n = min(w.n, per_rank)
    ins = (workloads.normals(w.seed, R, n, w.dtype) if w.dtype == workloads.BF16
           else workloads.int_values_f32(w.seed, R, n))
    return (lambda: oracle.all_reduce(ins, w.dtype),
            2 * R * n * workloads.ELEM_BYTES[w.dtype],
            f"AllReduce R=8, {n} elements per rank")


def calibrated_sample(w, seconds: float):
    """Pick the per-rank sample size whose oracle run takes about `seconds`."""
    n0 = 1 << 14
    fn, _, _ = oracle_sample(w, n0)
    fn()
    t0 = time.perf_counter()
    fn()
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(n0 * seconds / dt)
    n = max(4096, min(n, w.n))
    return oracle_sample(w, n)


def oracle_sample_time(w, budget_s: float = 10.0):
    """The oracle as it stands on a bounded sample, repeated for about
    `budget_s` seconds; returns (GB/s, description, seconds per rep, reps)."""
    fn, nbytes, desc = calibrated_sample(w, min(2.0, budget_s / 4))
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = (time.perf_counter() - t0) / reps
    return nbytes / dt / 1e9, desc, dt, reps


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed as it stands, on the host's
    cores (its OpenMP build over every core this process may use).  Each
    step is one oracle run over a sample sized so the whole run takes about
    a minute."""
    if rank != 0:
        return
    w = _workload_by_name(args.workload)
    import oracle

    cores = len(os.sched_getaffinity(0))
    oracle.build(openmp=True)
    with oracle.openmp(cores) as omp:
        threads = omp.threads
        per_step = max(0.02, 60.0 / max(1, args.steps + args.warmup))
        fn, nbytes, desc = calibrated_sample(w, per_step)
        for _ in range(args.warmup):
            fn()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            fn()
            times.append(time.perf_counter() - t0)
    total = float(np.sum(times))
    value = nbytes * args.steps / total / 1e9
    line = {
        "impl": "reference",
        "metric": "effective HBM GB/s (algorithmic read+write bytes / device time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == workloads.BF16 else "f32", "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "elements_per_rank": w.n},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "build": f"OpenMP, {threads} threads", "cpu_model": cpu_model(),
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _workload_by_name(name):
    for w in (workloads.AR_F32_R8_4096, workloads.AG_BF16_R8_8MI, workloads.RS_BF16_R8_128MI,
              workloads.A2AV_BF16_R8_MOE):
        if w.name == name:
            return w
    if name.startswith("allreduce_bf16_R8_b"):
        return workloads.ar_sweep_workload(int(name.rsplit("_b", 1)[1].split("x")[0]))
    raise SystemExit(f"unknown workload {name}")


# ------------------------------------------------------- multi-rank ------
# Replicas only: every rank runs its own in-HBM collective on its own GPU;
# ranks meet only at the barriers around the timed region and in the max.

def max_over_ranks(x: float) -> float:
    """The largest `x` over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, steps: int, world: int, slowest_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time, in GB/s."""
    return world * bytes_per_step_per_rank * steps / (slowest_ms / 1e3) / 1e9


# ------------------------------------------------------------ GPU arm ----

def time_steps(torch, stream, run, src, dst, steps, flush_buf, events_out, back_to_back=False):
    """Per-step device time in ms.  back_to_back (inputs larger than L2): the
    steps run one after another between one pair of CUDA events on `stream`
    and each gets the average; otherwise every step has its own events and
    the L2 is flushed (a 512 MiB write) before it, outside the events."""
    if back_to_back:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                run(src, dst)
            e1.record(stream)
        stream.synchronize()
        ms = [e0.elapsed_time(e1) / steps] * steps
        events_out.extend(ms)
        return ms
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_buf.zero_()
            starts[i].record(stream)
            run(src, dst)
            ends[i].record(stream)
    stream.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    events_out.extend(ms)
    return ms


def _graph_per_call_us(torch, stream, fn, k, reps=5):
    """Device time per call from a CUDA graph of k calls (median of reps
    replays): the host's launch cost drops out."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(k):
            fn()
    g.replay()
    stream.synchronize()
    t = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        t.append(e0.elapsed_time(e1) * 1e3 / k)
    del g
    return float(np.median(t))


def _graph_flushed_us(torch, stream, fn, flush, k):
    """Device time per call with the L2 flushed before every call and no
    launch cost: a graph of k (flush, call) pairs minus a graph of k
    flushes, per call."""
    both = _graph_per_call_us(torch, stream, lambda: (flush.zero_(), fn()), k)
    only = _graph_per_call_us(torch, stream, lambda: flush.zero_(), k)
    return both - only


def _back_to_back_us(torch, stream, fn, k):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / k


def config_rows(P, ctx, torch, device, stream, flush, peak):
    """Every workload of the measurement table, at its full size, timed on
    this GPU in this run (the bench line's ``configs``).  Per row: the
    median of single launches with the L2 flushed before each (the launch
    floor included), the average of back-to-back launches where the inputs
    exceed the L2, and for messages of up to 32 MiB per rank the device time
    per call in a CUDA graph, L2 flushed and warm.  Effective GB/s =
    algorithmic read+write bytes / time; frac = that / the measured copy
    peak; algbw = the pages' totalBytes (one rank's input) / the
    single-launch time.  Inputs: the small exact-integer AllReduce from the host
    generator; the large ones N(0,1) drawn on the device from a seeded
    generator (the values do not change the work; the parity tests use the
    host-generated workloads)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(4)
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or 0)
    rows = []

    def normals(n):
        return torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)

    def measure(name, fn, algo, in_bytes, reps, graph=False):
        # none of these rows is an AllGather: the pages' totalBytes is the
        # input size of one rank (every rank's input has the same size here)
        total = in_bytes // 8
        fn()
        P.purlin_check(ctx)
        info = P.purlin_last_launch(ctx)
        single = _events_us(torch, stream, fn, reps, flush)[0]
        row = {"config": name, "variant": info["variant"], "grid": info["grid"],
               "algorithmic_bytes": algo, "us_single_flushed": single,
               "gbs_single_flushed": algo / (single * 1e-6) / 1e9}
        row["frac_single_flushed"] = row["gbs_single_flushed"] / peak
        row.update({"total_bytes": total, "algbw_gbs_single_flushed": total / (single * 1e-6) / 1e9})
        traffic = recorded_traffic(name)   # DRAM bytes per launch, ncu, this kernel source
        if traffic is not None:
            row.update({"traffic": traffic, "traffic_over_algorithmic": traffic / algo})
        if in_bytes > l2:
            b2b = _back_to_back_us(torch, stream, fn, max(3, reps // 2))
            row.update({"us_back_to_back": b2b, "gbs_back_to_back": algo / (b2b * 1e-6) / 1e9,
                        "frac_back_to_back": algo / (b2b * 1e-6) / 1e9 / peak})
        if graph:
            k = 100 if algo < (64 << 20) else 20
            gf = _graph_flushed_us(torch, stream, fn, flush, k)
            gw = _graph_per_call_us(torch, stream, fn, k)
            row.update({"us_graph_flushed": gf, "gbs_graph_flushed": algo / (gf * 1e-6) / 1e9,
                        "frac_graph_flushed": algo / (gf * 1e-6) / 1e9 / peak,
                        "us_graph_warm": gw, "gbs_graph_warm": algo / (gw * 1e-6) / 1e9})
        P.purlin_check(ctx)
        rows.append(row)

    # config 1: AllReduce fp32 8 x 4096, exact integer values (latency-bound)
    w = workloads.AR_F32_R8_4096
    src = [torch.from_numpy(x).to(device) for x in workloads.inputs_for(w)]
    dst = [torch.empty(w.n, dtype=torch.float32, device=device) for _ in range(8)]
    torch.cuda.synchronize()
    measure(w.name, lambda: P.purlin_all_reduce(ctx, src, dst, w.n, 0), 2 * 8 * w.n * 4,
            8 * w.n * 4, 200, graph=True)
    del src, dst

    # config 3: ReduceScatter bf16 8 x 128 Mi
    w = workloads.RS_BF16_R8_128MI
    src = [normals(w.n) for _ in range(8)]
    dst = [torch.empty(w.n // 8, dtype=torch.bfloat16, device=device) for _ in range(8)]
    torch.cuda.synchronize()
    measure(w.name, lambda: P.purlin_reduce_scatter(ctx, src, dst, w.n, 1),
            8 * w.n * 2 + w.n * 2, 8 * w.n * 2, 10)
    del src, dst
    torch.cuda.empty_cache()

    # config 4: AllToAllV bf16, MoE dispatch (Zipf(1.2) count matrix)
    C, _ = workloads.moe_dispatch(payload=False)
    counts = (C * workloads.MOE_HIDDEN).reshape(-1)
    Cm = counts.reshape(8, 8)
    src = [normals(int(Cm[s].sum())) for s in range(8)]
    dst = [torch.empty(int(Cm[:, d].sum()), dtype=torch.bfloat16, device=device)
           for d in range(8)]
    torch.cuda.synchronize()
    cl = counts.tolist()
    measure(workloads.A2AV_BF16_R8_MOE.name, lambda: P.purlin_all_to_all_v(ctx, src, dst, cl, 1),
            2 * int(counts.sum()) * 2, int(counts.sum()) * 2, 10)
    del src, dst
    torch.cuda.empty_cache()

    # config 5: AllReduce bf16, batch x 4096 per rank, the whole sweep
    for b in workloads.AR_BF16_SWEEP_BATCHES:
        n = b * workloads.HIDDEN
        src = [normals(n) for _ in range(8)]
        dst = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(8)]
        torch.cuda.synchronize()
        measure(workloads.ar_sweep_workload(b).name,
                lambda: P.purlin_all_reduce(ctx, src, dst, n, 1), 2 * 8 * n * 2, 8 * n * 2,
                100 if n <= (1 << 20) else 20, graph=2 * n <= (32 << 20))
        del src, dst
        torch.cuda.empty_cache()
    return rows


def small_message_rows():
    """Messages of 2 KiB per rank and less against the two launch floors,
    timed from C through the public ABI (no Python in the timed path): per
    collective one call between events (median of 200) and the device time
    per call in a CUDA graph of 1000 calls; the floors are an empty kernel
    and a kernel whose one thread loads and stores 16 bytes, timed the same
    two ways."""
    exe = os.path.join(ROOT, "collective_datapath_atom_gb300", "purlin_bench")
    rows = []
    for coll in ("AR", "RS", "AG", "A2A", "AGV", "RSV", "A2AV"):
        lo = "256" if coll in ("AR", "AG") else "2048"
        res = subprocess.run([exe, coll, lo, "2048", "1000", "200", "10", "42"],
                             capture_output=True, text=True, check=True)
        for line in res.stdout.splitlines():
            r = json.loads(line)
            rows.append({k: r[k] for k in (
                "coll", "bytes_per_rank", "single_us", "graph_us", "floor_single_us",
                "floor_graph_us", "x_floor_single", "x_floor_graph", "touch_single_us",
                "touch_graph_us", "x_touch_single", "x_touch_graph")})
    return rows


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def cpu_baseline_legs(w, seconds: float):
    """The oracle as it stands on the host: its single-threaded build, then
    its OpenMP build over every core this process may run on."""
    import oracle

    oracle.build()
    gbs1, desc1, dt1, reps1 = oracle_sample_time(w, budget_s=seconds)
    cores = len(os.sched_getaffinity(0))
    try:
        oracle.build(openmp=True)
        with oracle.openmp(cores) as omp:
            gbsn, descn, dtn, repsn = oracle_sample_time(w, budget_s=seconds)
            used = omp.threads
    except (OSError, subprocess.CalledProcessError) as e:
        return {"value": gbs1, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"{desc1}; {reps1} reps, {dt1 * 1e3:.1f} ms each",
                "openmp": f"unavailable: {e}", "cpu_model": cpu_model()}
    return {"value": gbsn, "unit": "GB/s", "cores": used, "kind": "oracle",
            "build": f"OpenMP, {used} threads (sched_getaffinity: {cores} cores)",
            "sample": f"{descn}; {repsn} reps, {dtn * 1e3:.1f} ms each",
            "cpu_model": cpu_model(),
            "single_core": {"value": gbs1, "unit": "GB/s", "cores": 1,
                            "sample": f"{desc1}; {reps1} reps, {dt1 * 1e3:.1f} ms each"}}


def run_gpu(args, rank, world, local_rank):
    import torch

    import collective_datapath_atom_gb300 as P

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    ctx = P.purlin_init(8, stream)
    w, ins, src, dst, call, algo_bytes, in_bytes, out_bytes = setup_workload(
        args.workload, device, args.elements)
    run = make_runner(P, ctx, w, call)
    if args.device_counts:
        # the count matrix stays on the GPU: the device-count entry point,
        # with every output sized for the largest column
        if w.collective != "all_to_all_v":
            raise SystemExit("--device-counts applies to the AllToAllV workload")
        Cm = np.asarray(call[1]).reshape(w.R, w.R)
        in_cap, out_cap = int(Cm.sum(1).max()), int(Cm.sum(0).max())
        dst = [torch.empty(out_cap, dtype=d.dtype, device=device) for d in dst]
        d_counts = torch.tensor(call[1], dtype=torch.int64, device=device)

        def run(src_, dst_):
            P.purlin_all_to_all_v_device_counts(ctx, src_, dst_, d_counts, in_cap, out_cap,
                                                w.dtype)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    torch.cuda.synchronize()   # inputs were uploaded on another stream

    # warm-up (also checks the first call for device errors)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run(src, dst)
    P.purlin_check(ctx)
    info = P.purlin_last_launch(ctx)

    dist = None
    if world > 1:
        import torch.distributed as dist
    sampler = ClockSampler(local_rank) if not args.no_clocks else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    # Inputs larger than the L2 cannot carry over from one step to the next
    # (each step also writes its outputs through L2), so such workloads run
    # back to back; smaller ones get the L2 flushed before every step.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or 0)
    back_to_back = (not args.flush) and l2_bytes > 0 and in_bytes > l2_bytes
    l2_note = (f"not flushed: inputs ({in_bytes} B) larger than L2 ({l2_bytes} B), steps back to back"
               if back_to_back else f"flushed between steps (512 MiB write; L2 {l2_bytes} B)")
    ms = time_steps(torch, stream, run, src, dst, args.steps, flush_buf, [], back_to_back)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None
    P.purlin_check(ctx)
    total_ms = max_over_ranks(float(np.sum(ms)))
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(algo_bytes, args.steps, world, total_ms)

    # the pages' "algorithm bandwidth": totalBytes / time, with totalBytes the
    # output size of one rank for AllGather and the input size of one rank
    # otherwise (the largest rank's, where V counts make them differ)
    total_bytes = (max(d.numel() * d.element_size() for d in dst) if call[0] == "all_gather"
                   else max(x.nbytes for x in ins))

    # roofline of the dominant (only) kernel: one launch per step
    peak, peak_kind = measured_peaks()
    achieved = algo_bytes / (float(np.mean(ms)) / 1e3) / 1e9
    traffic = recorded_traffic(w.name)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        h_in = [torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).pin_memory()
                for x in ins]
        h_out = [torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in dst]
        e2e_steps = max(3, min(args.steps, 20))
        with torch.cuda.stream(stream):
            for i in range(2):
                for hs, ds in zip(h_in, src):
                    ds.copy_(hs, non_blocking=True)
                run(src, dst)
                for ho, dd in zip(h_out, dst):
                    ho.copy_(dd, non_blocking=True)
        stream.synchronize()
        # Steps are pipelined across the two directions of the host link:
        # step i+1's inputs go up (second stream) while step i's outputs come
        # down.  Every step still copies its own inputs in and its outputs
        # out; the upload of step i+1 only waits for step i's call to finish
        # reading the inputs, and step i+1's call waits for its upload.
        up = torch.cuda.Stream(stream.device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        read_done = [torch.cuda.Event() for _ in range(e2e_steps)]
        uploaded = [torch.cuda.Event() for _ in range(e2e_steps)]
        e0.record(stream)
        for i in range(e2e_steps):
            up.wait_event(e0 if i == 0 else read_done[i - 1])
            with torch.cuda.stream(up):
                for hs, ds in zip(h_in, src):
                    ds.copy_(hs, non_blocking=True)
            uploaded[i].record(up)
            stream.wait_event(uploaded[i])
            with torch.cuda.stream(stream):
                run(src, dst)
                read_done[i].record(stream)
                for ho, dd in zip(h_out, dst):
                    ho.copy_(dd, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        e2e = {"value": world * algo_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": e2e_ms}

    # the headline workload back to back (no flush between steps): the
    # output left dirty in the L2 by one step is written back during the next
    b2b = None
    if not args.no_configs:
        k = max(10, min(args.steps, 200))
        b2b_us = _back_to_back_us(torch, stream, lambda: run(src, dst), k)
        b2b = {"us": b2b_us, "steps": k, "gbs": algo_bytes / (b2b_us * 1e-6) / 1e9,
               "frac": algo_bytes / (b2b_us * 1e-6) / 1e9 / peak}
        P.purlin_check(ctx)

    configs = small = None
    if rank == 0 and not args.no_configs:
        # Extra rows: a failure here is recorded in the line, never loses it.
        try:
            configs = config_rows(P, ctx, torch, device, stream, flush_buf, peak)
        except Exception as e:   # noqa: BLE001
            configs = {"error": f"{type(e).__name__}: {e}"}
        try:
            small = small_message_rows()
        except Exception as e:   # noqa: BLE001
            small = {"error": f"{type(e).__name__}: {e}"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        try:
            cpu = cpu_baseline_legs(w, args.cpu_seconds)
        except Exception as e:   # noqa: BLE001
            cpu = {"error": f"{type(e).__name__}: {e}"}

    line = {
        "metric": "effective HBM GB/s (algorithmic read+write bytes / device time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == 1 else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "elements_per_rank": w.n,
                   "algorithmic_bytes_per_step": algo_bytes, "l2": l2_note,
                   "variant": info["variant"], "grid": info["grid"], "block": info["block"],
                   "stages": info["stages"], "chunk_bytes": info["chunk_bytes"],
                   "parallelism": f"replicas x{world}",
                   **({"counts": "device"} if args.device_counts else {})},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                     "kernel": KERNEL_OF_VARIANT.get(info["variant"], "none")},
        "algbw": {"total_bytes": total_bytes, "gbs": total_bytes / (ms_per_step / 1e3) / 1e9,
                  "note": "pages-style algorithm bandwidth (totalBytes / device time per step), "
                          "not the headline metric"},
        "back_to_back": b2b,
        "configs": configs,
        "small_messages": small,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
        "p10_p50_p90_us": [float(np.percentile(ms, q)) * 1e3 for q in (10, 50, 90)],
    }
    ctx.close()
    return line


# --------------------------------------------------------------- sweep ----

def _events_us(torch, stream, fn, reps, flush=None):
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for i in range(reps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    stream.synchronize()
    us = np.array([a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends)])
    return float(np.median(us)), float(np.percentile(us, 10)), float(np.percentile(us, 90))


def _graph_us(torch, stream, fn, k):
    """Device time per launch from a CUDA graph of k launches."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(k):
            fn()
    g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(5):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (5 * k)


def sweep(args):
    """Every workload, both variants across the AllReduce sweep, composed vs
    fused AllReduce, and small-message latency against the empty-kernel
    floor.  Timing inputs are seeded N(0,1) values drawn on the device (the
    values do not change the work); the parity tests use the CPU-generated
    workloads."""
    import torch

    import collective_datapath_atom_gb300 as P

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    ctx = P.purlin_init(8, stream)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    peak, peak_kind = measured_peaks()
    gen = torch.Generator(device=device)
    gen.manual_seed(4)
    rows = []

    def emit(row):
        rows.append(row)
        print(json.dumps(row), flush=True)

    sections = set(args.rows.split(",")) if args.rows else None

    def want(name):
        return sections is None or name in sections

    def bufs(n_in, n_out, dtype=1):
        tdt = torch.float32 if dtype == 0 else torch.bfloat16
        src = [torch.randn(n_in, generator=gen, device=device, dtype=torch.float32).to(tdt)
               for _ in range(8)]
        dst = [torch.empty(n_out, device=device, dtype=tdt) for _ in range(8)]
        torch.cuda.synchronize()   # drawn on the default stream; the library uses `stream`
        return src, dst

    def setopt(variant, mode=0):
        P.purlin_set_option(ctx, P.PURLIN_OPT_VARIANT, variant)
        P.purlin_set_option(ctx, P.PURLIN_OPT_AR_MODE, mode)

    # ---- small messages (<= 2 KiB per rank) against the empty-kernel floor,
    # timed from C through the public ABI (no Python in the timed path)
    exe = os.path.join(ROOT, "collective_datapath_atom_gb300", "purlin_bench")
    for coll in ("AR", "RS", "AG", "A2A", "AGV", "RSV", "A2AV") if want("small") else ():
        res = subprocess.run([exe, coll, "256", "2048", "200", "200", "10", "42"],
                             capture_output=True, text=True, check=True)
        for line in res.stdout.splitlines():
            r = json.loads(line)
            r["row"] = "small"
            emit(r)

    # ---- the pages' V-collective sweep ("Purlin: Separating Orchestration from the Datapath of Collectives"
    # §C.4): Zipf(0.125)
    # split of a total T per rank, 1 KiB .. 1 GiB, through the C ABI
    for coll in ("AGV", "RSV", "A2AV") if want("vsweep") else ():
        res = subprocess.run([exe, coll, "1024", str(1 << 30), "10", "10", "2", "42"],
                             capture_output=True, text=True, check=True)
        for line in res.stdout.splitlines():
            r = json.loads(line)
            r["row"] = "vsweep"
            r["frac"] = r["eff_gbs"] / peak
            emit(r)

    # ---- AllReduce bf16 sweep, batch x 4096, both variants, L2 flushed
    for b in workloads.AR_BF16_SWEEP_BATCHES if want("ar_sweep") else ():
        n = b * workloads.HIDDEN
        src, dst = bufs(n, n)
        algo = 2 * 8 * n * 2
        reps = 200 if n <= (1 << 20) else 30
        for variant, mode in ((1, 0), (2, 1), (2, 2), (0, 3), (0, 0)):
            if mode == 3 and 2 * n > (1 << 20):   # packets: up to 1 MiB per rank
                continue
            setopt(variant, mode)
            call = lambda: P.purlin_all_reduce(ctx, src, dst, n, 1)   # noqa: E731
            call()
            P.purlin_check(ctx)
            info = P.purlin_last_launch(ctx)
            med, p10, p90 = _events_us(torch, stream, call, reps, flush)
            warm = _events_us(torch, stream, call, reps)[0] if n <= (8 << 20) else None
            emit({"row": "ar_sweep", "batch": b, "bytes_per_rank": 2 * n,
                  "mode": {(1, 0): "latency", (2, 1): "throughput fused",
                           (2, 2): "throughput composed", (0, 3): "composed packets",
                           (0, 0): "auto"}[(variant, mode)],
                  "chosen_variant": info["variant"], "us_cold": med, "p10": p10, "p90": p90,
                  "us_warm": warm, "gbs_cold": algo / (med * 1e-6) / 1e9,
                  "frac_cold": algo / (med * 1e-6) / 1e9 / peak})
        del src, dst
        torch.cuda.empty_cache()
    setopt(0)

    # ---- the large workloads, L2 flushed
    for name in (workloads.AG_BF16_R8_8MI.name, workloads.RS_BF16_R8_128MI.name,
                 workloads.A2AV_BF16_R8_MOE.name,
                 workloads.AR_F32_R8_4096.name) if want("workload") else ():
        w, ins, src, dst, call, algo, _, _ = setup_workload(name, device)
        torch.cuda.synchronize()
        run = make_runner(P, ctx, w, call)
        for variant in (0, 1, 2):
            setopt(variant)
            run(src, dst)
            P.purlin_check(ctx)
            info = P.purlin_last_launch(ctx)
            med, p10, p90 = _events_us(torch, stream, lambda: run(src, dst), 20, flush)
            emit({"row": "workload", "workload": w.name, "variant_opt": variant,
                  "variant": info["variant"], "us": med, "p10": p10, "p90": p90,
                  "gbs": algo / (med * 1e-6) / 1e9, "frac": algo / (med * 1e-6) / 1e9 / peak,
                  "grid": info["grid"], "block": info["block"], "stages": info["stages"]})
        del ins, src, dst
        torch.cuda.empty_cache()

    # ---- the device-side API: the same collectives entered from a user
    # kernel (examples/), and the Atom's copy bandwidth against CTA count
    from collective_datapath_atom_gb300 import examples as X

    sms = torch.cuda.get_device_properties(device).multi_processor_count
    dev_cases = [(workloads.AG_BF16_R8_8MI.name, 0), (workloads.RS_BF16_R8_128MI.name, 0),
                 (workloads.ar_sweep_workload(32768).name, 1),
                 (workloads.ar_sweep_workload(32768).name, 2)]
    for name, mode in dev_cases if want("device_api") else ():
        w, ins, src, dst, call, algo, _, _ = setup_workload(name, device)
        torch.cuda.synchronize()
        setopt(2, mode)
        coll = {"all_gather": P.PURLIN_COLL_ALL_GATHER, "reduce_scatter": P.PURLIN_COLL_REDUCE_SCATTER,
                "all_reduce": P.PURLIN_COLL_ALL_REDUCE}[w.collective]
        run = make_runner(P, ctx, w, call)
        run(src, dst)
        P.purlin_check(ctx)
        host_us = _events_us(torch, stream, lambda: run(src, dst), 20, flush)[0]
        grid = P.purlin_last_launch(ctx)["grid"]
        d = P.purlin_device_prepare(ctx, coll, src, dst, n=w.n, dtype=w.dtype, blocks=grid)
        fn = lambda: X.collective(d, stream=stream)   # noqa: E731
        fn()
        assert P.purlin_device_check(d, stream) == P.PURLIN_OK
        med, p10, p90 = _events_us(torch, stream, fn, 20, flush)
        emit({"row": "device_api", "workload": w.name,
              "mode": {0: "", 1: "fused", 2: "composed"}[mode], "blocks": grid,
              "threads": d.threads, "us": med, "p10": p10, "p90": p90,
              "gbs": algo / (med * 1e-6) / 1e9, "frac": algo / (med * 1e-6) / 1e9 / peak,
              "host_call_us": host_us})
        P.purlin_device_release(ctx, d)
        del ins, src, dst
        torch.cuda.empty_cache()
    setopt(0)

    # ---- V collectives with device-resident counts: the MoE dispatch with
    # the count matrix already on the GPU, against the host-count call and
    # against what a host-count caller must do with GPU counts (copy them
    # to the host first); also a decode-size dispatch (64 tokens per rank)
    if want("device_counts"):
        w, ins, src, dst, call, algo, _, _ = setup_workload(workloads.A2AV_BF16_R8_MOE.name,
                                                            device)
    H = workloads.MOE_HIDDEN
    for label, tokens in (("moe_16384tok", workloads.MOE_TOKENS),
                          ("moe_64tok", 64)) if want("device_counts") else ():
        if tokens == workloads.MOE_TOKENS:
            counts = call[1]
            s_in = src
        else:
            Cs = np.stack([np.random.default_rng(7 + r).multinomial(tokens, workloads.zipf_weights(8))
                           for r in range(8)])
            counts = (Cs * H).reshape(-1).tolist()
            s_in = [x[:tokens * H] for x in src]
        Cm = np.asarray(counts).reshape(8, 8)
        in_cap, out_cap = int(Cm.sum(1).max()), int(Cm.sum(0).max())
        d_out = [torch.empty(out_cap, dtype=torch.int16, device=device) for _ in range(8)]
        d_counts = torch.tensor(counts, dtype=torch.int64, device=device)
        torch.cuda.synchronize()
        algo_c = 2 * int(Cm.sum()) * 2
        for path, fn in (
                ("host_counts", lambda: P.purlin_all_to_all_v(ctx, s_in, d_out, counts, 1)),
                ("device_counts", lambda: P.purlin_all_to_all_v_device_counts(
                    ctx, s_in, d_out, d_counts, in_cap, out_cap, 1)),
                ("device_counts_copied_to_host", lambda: P.purlin_all_to_all_v(
                    ctx, s_in, d_out, d_counts.cpu().tolist(), 1))):
            fn()
            P.purlin_check(ctx)
            med, p10, p90 = _events_us(torch, stream, fn, 30, flush)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(30):
                fn()
            torch.cuda.synchronize()
            wall = (time.perf_counter() - t0) / 30 * 1e6
            emit({"row": "device_counts", "workload": label, "path": path, "us": med, "p10": p10,
                  "p90": p90, "wall_us_per_call": wall, "gbs": algo_c / (med * 1e-6) / 1e9,
                  "frac": algo_c / (med * 1e-6) / 1e9 / peak})
        del d_out
    if want("device_counts"):
        del ins, src, dst
    torch.cuda.empty_cache()

    # ---- the packet channel (latency path, 16-byte payload+flag packets)
    # against the chunk-flag path, both inside a user kernel that computes
    # relu of its inputs and AllReduces the result: the packet-streaming
    # kernel (no grid barrier; each unit moves as soon as it is computed)
    # against relu, grid barrier, then the device-side composed AllReduce
    # (per-chunk flags) or the fused one (no cross-CTA flags).  Single
    # launches with the L2 flushed (median of 100), and per call in a CUDA
    # graph of 100 (L2 warm).
    if want("packet_channel"):
        ch = P.purlin_packet_channel_create(ctx, 1 << 20, 2 * sms)
        for per_rank in (256, 2048, 16 << 10, 64 << 10, 256 << 10, 1 << 20):
            n = per_rank // 2
            src, dst = bufs(n, n)
            ptr_s, ptr_d = [t.data_ptr() for t in src], [t.data_ptr() for t in dst]
            cases = [("packets", lambda: X.packet_stream(ch, ptr_s, ptr_d, n, 1, True,
                                                         stream=stream))]
            descs = []
            for mode, label in ((2, "chunk_flags"), (1, "fused")):
                setopt(2, mode)
                d = P.purlin_device_prepare(ctx, P.PURLIN_COLL_ALL_REDUCE, src, dst, n=n, dtype=1,
                                            blocks=sms)
                descs.append(d)
                cases.append((label, (lambda d=d: X.relu_collective(d, n, stream=stream))))
            setopt(0)
            for label, fn in cases:
                fn()
                torch.cuda.synchronize()
                med, p10, p90 = _events_us(torch, stream, fn, 100, flush)
                g_us = _graph_us(torch, stream, fn, 100)
                emit({"row": "packet_channel", "bytes_per_rank": per_rank, "path": label,
                      "us_single": med, "p10": p10, "p90": p90, "us_graph": g_us})
            assert P.purlin_packet_channel_check(ch, stream) == P.PURLIN_OK
            for d in descs:
                assert P.purlin_device_check(d, stream) == P.PURLIN_OK
                P.purlin_device_release(ctx, d)
            del src, dst
        P.purlin_packet_channel_release(ctx, ch)

    nbytes = 1 << 30 if want("atom_copy") else 16
    a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for ctas in (1, 2, 4, 8, 16, 38, 76, sms, 2 * sms, 3 * sms) if want("atom_copy") else ():
        per = (nbytes + ctas - 1) // ctas
        per = (per + 15) // 16 * 16
        fn = lambda: X.atom_copy(b, a, nbytes, per, status, stream=stream)   # noqa: E731
        fn()
        stream.synchronize()
        assert int(status.item()) == 0
        med = _events_us(torch, stream, fn, 5 if ctas < 16 else 20, flush)[0]
        emit({"row": "atom_copy", "ctas": ctas, "bytes": nbytes, "us": med,
              "gbs": 2 * nbytes / (med * 1e-6) / 1e9,
              "frac": 2 * nbytes / (med * 1e-6) / 1e9 / peak})
    del a, b
    ctx.close()
    if args.report:
        with open(args.report, "w") as f:
            for r in rows:
                f.write(json.dumps(r) + "\n")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="purlin", choices=["purlin", "reference"])
    ap.add_argument("--workload", default=workloads.AG_BF16_R8_8MI.name)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="only the headline workload (no per-config rows, no small messages)")
    ap.add_argument("--flush", action="store_true",
                    help="flush L2 before every timed step even when the inputs exceed it")
    ap.add_argument("--device-counts", action="store_true",
                    help="AllToAllV workload: counts in device memory (the device-count call)")
    ap.add_argument("--elements", type=int, default=0,
                    help="elements per rank (a smaller case of the same kernel)")
    ap.add_argument("--sweep", action="store_true",
                    help="measure every workload, both variants and the launch floor")
    ap.add_argument("--report", default="", help="with --sweep: also write the rows here")
    ap.add_argument("--rows", default="",
                    help="with --sweep: comma-separated sections to run (small, vsweep, ar_sweep, "
                         "workload, device_api, device_counts, packet_channel, atom_copy)")
    args = ap.parse_args()
    if args.sweep:
        sweep(args)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
