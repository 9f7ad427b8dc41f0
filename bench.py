"""Bench of the virtual-rank collectives: HBM GB/s and fraction of the
measured copy peak.

One step = the whole path once over the workload: the fused AllReduce
(vc_all_reduce, one kernel) and the decomposed AllReduce
(vc_all_reduce_decomposed: ReduceScatter kernel, then AllGather kernel).
Default workload: four virtual ranks of 256 MiB fp32 (67,108,864 elements,
normal(0, 1)), SUM, ring order.

Algorithmic bytes (s = element size, q = ceil(M/N)):
  ReduceScatter  N*M*s read + M*s written
  AllGather      M*s read   + N*M*s written
  fused AR       N*M*s read + N*M*s written
  decomposed AR  RS + AG
The step moves 4*N*M*s + 2*M*s bytes; value = those bytes / step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(the path shards by index range with no exchange; weak scaling), the step
time is the max over ranks, and value counts the bytes of all ranks.
--impl reference times the CPU oracle instead, on a bounded window of the
same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "AR/RS/AG HBM GB/s over N virtual ranks; % of GB300 HBM copy peak"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 10**6  # GB300 L2
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, the vendor's figure (context only)
ESIZE = {"int32": 4, "int64": 8, "float32": 4, "bfloat16": 2}
DTYPE_TAG = {"int32": "i32", "int64": "i64", "float32": "f32", "bfloat16": "bf16"}


# ----------------------------------------------------------------- helpers --

def step_bytes(n: int, M: int, es: int) -> dict:
    rs = n * M * es + M * es
    ag = M * es + n * M * es
    ar = 2 * n * M * es
    return {"reduce_scatter": rs, "all_gather": ag, "fused_ar": ar, "decomposed_ar": rs + ag,
            "step": ar + rs + ag}


def measured_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and blank lines: a comment edit does not
    change the kernels, so it does not void a recorded ncu figure."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


# The sources that build and launch the measured kernels (vc_ar_kernel,
# vc_rs_kernel, vc_ag_kernel): the kernels and folds, the instance dispatch,
# and the host side that sizes the grids.
KERNEL_SOURCES = ("vc_device.cuh", "vc_launch.cuh", "vc_reduce_inst.cu",
                  "vc_reduce_dispatch.cu", "vc_api.cu")


def source_digest() -> str:
    """Digest of the code (comments and blank lines removed) of the sources
    that build and launch the measured kernels."""
    h = hashlib.sha256()
    csrc = ROOT / "allreduce_reducescatter_allgather_gb300" / "csrc"
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        h.update(_code_only((csrc / name).read_text()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = ROOT / "profiles" / "dram_traffic.txt"
    if not p.exists():
        return None
    rec = {}
    for line in p.read_text().splitlines():
        if line.startswith("#") or ":" not in line:
            continue
        k, _, v = line.partition(":")
        rec[k.strip()] = v.strip()
    key = f"{kernel}@{workload}"
    if rec.get("source_sha") != source_digest() or key not in rec:
        return None
    return float(rec[key])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index  # nvidia-smi --id: an index or a GPU UUID
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append({"sm": float(parts[2]), "max": float(parts[3]),
                             "power": float(parts[4]) if parts[4] not in ("[N/A]", "") else 0.0,
                             "hw_slowdown": parts[6], "hw_thermal": parts[7],
                             "sw_thermal": parts[8], "sw_power_cap": parts[9]})
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] >= 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for k in ("hw_slowdown", "hw_thermal", "sw_thermal", "sw_power_cap"):
                if r[k] == "Active":
                    reasons.add(k if k != "hw_thermal" else "hw_thermal_slowdown")
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "samples": len(loaded),
                "reasons": sorted(reasons)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(torch, local_ms: float, local_bytes: int, world: int):
    """Max step time and total bytes over ranks (control plane only)."""
    if world == 1:
        return local_ms, local_bytes
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() \
        else torch.device("cpu")
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


# ------------------------------------------------------------ CPU oracle --

class OracleStep:
    """One oracle step over host windows: fused AR then decomposed AR, into
    output arrays allocated once (so the timing is the oracle's arithmetic,
    not the host's page faults)."""

    def __init__(self, xs, dtype, op, order):
        import numpy as np
        import oracle
        self.oracle, self.xs, self.dtype, self.op, self.order = oracle, xs, dtype, op, order
        n, M = len(xs), xs[0].size
        st = oracle.NP_STORAGE[dtype]
        q = oracle.shard_count(M, n)
        self.y = [np.zeros(M, st) for _ in range(n)]
        self.y2 = [np.zeros(M, st) for _ in range(n)]
        self.z = [np.zeros(q, st) for _ in range(n)]

    def __call__(self):
        o = self.oracle
        o.all_reduce(self.xs, self.dtype, self.op, self.order, out=self.y)
        o.all_reduce_decomposed(self.xs, self.dtype, self.op, self.order, shards=self.z,
                                out=self.y2)


def host_window(workload: dict, window: int, start: int = 0):
    """Elements start .. start+window-1 of every rank of the workload (the
    same values the full workload holds there)."""
    import synthetic_inputs as si
    w = dict(workload)
    n, M = w.pop("n"), w.pop("M")
    dtype, dist_, seed = w.pop("dtype"), w.pop("dist"), w.pop("seed")
    W = min(window, M - start)
    return [si.generate_rank(dtype, dist_, seed, r, W, start=start, **w) for r in range(n)]


def time_oracle(workload: dict, op: str, order: str, seconds: float, window: int,
                start: int = 0):
    """Run oracle steps over a window of `window` elements per rank until
    `seconds` of CPU time have passed; returns (GB/s, steps, seconds)."""
    xs = host_window(workload, window, start)
    n, dtype = workload["n"], workload["dtype"]
    W = xs[0].size
    b = step_bytes(n, W, ESIZE[dtype])["step"]
    step = OracleStep(xs, dtype, op, order)
    step()
    steps, t0 = 0, time.perf_counter()
    while True:
        step()
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return b * steps / el / 1e9, steps, el


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or ""."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def _oracle_worker(job):
    """One process of the all-cores oracle timing: its own window."""
    workload, op, order, seconds, window, start = job
    g, steps, secs = time_oracle(workload, op, order, seconds, window, start)
    return g * secs * 1e9, steps, secs  # bytes, steps, seconds


def time_oracle_all_cores(workload: dict, op: str, order: str, seconds: float, window: int):
    """The oracle as it stands on every host core this process may use: one
    spawned process per core, each timing oracle steps on its own window of
    the workload (windows side by side from element 0, wrapping if the
    workload is shorter).  The oracle is single-threaded and unchanged;
    splitting the index range is exact because every element's reduction
    is independent.  Returns (GB/s, cores, steps, seconds)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    M = workload["M"]
    W = min(window, M)
    slots = max(1, M // W)
    jobs = [(workload, op, order, seconds, W, (k % slots) * W) for k in range(cores)]
    # an executor (not a Pool): a worker that dies raises here instead of
    # being replaced forever; the timeout bounds the whole measurement
    with ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        res = list(ex.map(_oracle_worker, jobs, timeout=3 * seconds + 300))
    total = sum(r[0] for r in res)
    secs = max(r[2] for r in res)
    return total / secs / 1e9, cores, sum(r[1] for r in res), secs


def run_reference(args, workload: dict):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    n, dtype = workload["n"], workload["dtype"]
    # size the window so that warmup + steps take about a minute: time two
    # steps on a 2^18-element window (outputs preallocated, as in the run)
    calib = OracleStep(host_window(workload, 1 << 18), dtype, args.op, args.order)
    calib()
    t0 = time.perf_counter()
    calib()
    calib()
    per_elem = (time.perf_counter() - t0) / 2 / calib.xs[0].size
    budget = 60.0 / max(1, args.steps + args.warmup)
    window = 1 << 12
    while window * 2 * per_elem <= budget and window * 2 <= workload["M"]:
        window *= 2
    step = OracleStep(host_window(workload, window), dtype, args.op, args.order)
    W = step.xs[0].size
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    b = step_bytes(n, W, ESIZE[dtype])["step"]
    value = b * args.steps / el / 1e9
    sample = (f"the first {W} of {workload['M']} elements of each of the {n} ranks; "
              f"each step = oracle fused AR + decomposed AR on that window")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_TAG[dtype], "data": "synthetic",
        "config": config_block(args, workload, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_note(input_bytes: int) -> str:
    """How the timed steps meet the 129 MB L2 (no flush between steps)."""
    if input_bytes >= 2 * L2_BYTES:
        return (f"no flush: every call streams {input_bytes / 2**30:.2f} GiB of inputs and as "
                "much output, far larger than the 129 MB L2")
    return (f"no flush, and the {input_bytes / 2**20:.0f} MiB of inputs are not larger than "
            "twice the 129 MB L2: a small case, its rates include L2 hits")


def config_block(args, workload, world):
    n, M, dtype = workload["n"], workload["M"], workload["dtype"]
    return {
        "workload": args.workload,
        "virtual_ranks": n, "elements_per_rank": M, "bytes_per_rank": M * ESIZE[dtype],
        "op": args.op, "order": args.order,
        "step": "fused AllReduce + decomposed AllReduce (ReduceScatter then AllGather)",
        "l2": l2_note(n * M * ESIZE[dtype]),
        "parallelism": f"{world} GPU(s), each with its own {n} virtual ranks (index-range "
                       "shards, no exchange)",
    }


# ------------------------------------------------------------ GPU arm ----

def run_ours(args, workload: dict):
    import torch

    import allreduce_reducescatter_allgather_gb300 as vc
    import synthetic_inputs as si

    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import datetime

        import torch.distributed as dist
        # a rank that dies or never arrives ends the others' next collective
        # with an error after this long, instead of leaving them waiting
        dist.init_process_group("nccl", device_id=dev,
                                timeout=datetime.timedelta(seconds=args.dist_timeout))

    w = dict(workload)
    n, M, dtype = w.pop("n"), w.pop("M"), w.pop("dtype")
    d = si.generate_device(torch, dtype, w.pop("dist"), n, M, w.pop("seed") + rank, dev, **w)
    q = vc.vc_shard_count(M, n)
    es = ESIZE[dtype]
    y = [torch.empty_like(t) for t in d]
    y2 = [torch.empty_like(t) for t in d]
    sh = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
    by = step_bytes(n, M, es)
    stream = torch.cuda.current_stream(dev)

    def step():
        vc.vc_all_reduce(d, y, op=args.op, order=args.order, stream=stream)
        vc.vc_all_reduce_decomposed(d, sh, y2, op=args.op, order=args.order, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        gpu_id = local
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    # per-call events on the launching stream: [AR start, AR end = dec start, dec end]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        e = evs[k]
        e[0].record(stream)
        vc.vc_all_reduce(d, y, op=args.op, order=args.order, stream=stream)
        e[1].record(stream)
        vc.vc_all_reduce_decomposed(d, sh, y2, op=args.op, order=args.order, stream=stream)
        e[2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    ar_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    max_ms, all_bytes = aggregate(torch, total_ms, by["step"] * args.steps, world)
    ms_per_step = max_ms / args.steps
    value = all_bytes / (max_ms / 1e3) / 1e9

    # RS alone and AG alone (outside the timed region), for the per-path table
    def time_calls(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fn()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    reps = max(10, min(200, args.steps))
    rs_ms = time_calls(lambda: vc.vc_reduce_scatter(d, sh, op=args.op, order=args.order,
                                                    stream=stream), reps)
    ag_ms = time_calls(lambda: vc.vc_all_gather(sh, y2, stream=stream), reps)

    peak, peak_kind = measured_peak()
    ar_avg = statistics.mean(ar_ms)
    dec_avg = statistics.mean(dec_ms)

    def path(bytes_, ms):
        g = bytes_ / (ms / 1e3) / 1e9
        return {"us": round(ms * 1e3, 2), "gbs": round(g, 1), "frac": round(g / peak, 4)}

    paths = {"fused_ar": path(by["fused_ar"], ar_avg),
             "decomposed_ar": path(by["decomposed_ar"], dec_avg),
             "reduce_scatter": path(by["reduce_scatter"], rs_ms),
             "all_gather": path(by["all_gather"], ag_ms)}
    ar_gbs = by["fused_ar"] / (ar_avg / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "vc_ar_kernel", "achieved": round(ar_gbs, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(ar_gbs / peak, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(ar_gbs / NOMINAL_HBM_GBS, 4),
                # recorded for the workload's own size only
                "traffic": (recorded_traffic("vc_ar_kernel", args.workload)
                            if M == si.WORKLOADS[args.workload]["M"] else None),
                "algorithmic_bytes_per_launch": by["fused_ar"]}

    memory = memory_report(torch, vc, d, args, dev) if not args.no_memory else None
    buckets = bucket_report(torch, vc, args, dev) if not args.no_memory else None
    latency = latency_table(torch, vc, args, dev) if not args.no_memory else None
    e2e = e2e_measure(torch, vc, d, y, y2, sh, args, dev, stream, by["step"])

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_TAG[dtype], "data": "synthetic",
        "config": config_block(args, workload, world),
        "roofline": roofline,
        "paths": paths,
        "gpu_launches": 3 * args.steps,
        "e2e": e2e,
    }
    if clk is not None:
        line["clocks"] = {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                          "reasons": clk["reasons"], "samples": clk["samples"]}
    if memory is not None:
        line["memory_mib"] = memory
    if buckets is not None:
        line["gradient_buckets"] = buckets
    if latency is not None:
        line["direct_vs_decomposed"] = latency
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        g, steps, secs = time_oracle(workload, args.op, args.order, args.cpu_seconds,
                                     window=1 << 22)
        line["cpu_baseline"] = {
            "value": round(g, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{steps} oracle steps (fused AR + decomposed AR) over the first "
                      f"{min(1 << 22, M)} elements of each of the {n} ranks, "
                      f"{secs:.1f} s on one host core"}
        try:
            gp, cores, psteps, psecs = time_oracle_all_cores(workload, args.op, args.order,
                                                            args.cpu_seconds, window=1 << 22)
            line["cpu_baseline"]["all_cores"] = {
                "value": round(gp, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"{psteps} oracle steps in {cores} spawned processes, each on its "
                          f"own {min(1 << 22, M)}-element window of every rank, "
                          f"{psecs:.1f} s"}
        except Exception as e:  # the single-core figure above still stands
            line["cpu_baseline"]["all_cores"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def e2e_measure(torch, vc, d, y, y2, sh, args, dev, stream, step_bytes_):
    """The same step through the public API with the inputs in pinned host
    memory: each step copies the N inputs in, runs both AllReduce paths and
    copies every output of both back.  Steps are pipelined the way a user
    would run them: two sets of device buffers and of host outputs, one
    stream per direction, so step k+1's inputs travel while step k's
    outputs come back (the two link directions run concurrently)."""
    n = len(d)
    host_in = [t.cpu().pin_memory() for t in d]
    sets = [(d, y, y2, sh),
            ([torch.empty_like(t) for t in d], [torch.empty_like(t) for t in d],
             [torch.empty_like(t) for t in d], [torch.empty_like(t) for t in sh])]
    host_out = [([torch.empty_like(t, device="cpu").pin_memory() for t in d],
                 [torch.empty_like(t, device="cpu").pin_memory() for t in d]) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = 2 * h2d
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(steps):
        for k in range(steps):
            j = k % 2
            di, dy, dy2, dsh = sets[j]
            hy, hy2 = host_out[j]
            if k >= 2:
                s_in.wait_event(comp_done[j])  # set j's inputs no longer read
            with torch.cuda.stream(s_in):
                for r in range(n):
                    di[r].copy_(host_in[r], non_blocking=True)
            in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            if k >= 2:
                stream.wait_event(out_done[j])  # set j's outputs already copied out
            vc.vc_all_reduce(di, dy, op=args.op, order=args.order, stream=stream)
            vc.vc_all_reduce_decomposed(di, dsh, dy2, op=args.op, order=args.order,
                                        stream=stream)
            comp_done[j].record(stream)
            s_out.wait_event(comp_done[j])
            with torch.cuda.stream(s_out):
                for r in range(n):
                    hy[r].copy_(dy[r], non_blocking=True)
                    hy2[r].copy_(dy2[r], non_blocking=True)
            out_done[j].record(s_out)

    run(2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(args.e2e_steps)
    s_in.wait_stream(s_out)
    s_in.wait_stream(stream)
    b.record(s_in)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.e2e_steps
    wall_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    # every output of the last step came back intact
    ref = sets[(args.e2e_steps - 1) % 2][1][0].cpu()
    assert torch.equal(host_out[(args.e2e_steps - 1) % 2][0][n - 1], ref)
    del sets, host_out
    return {"value": round(step_bytes_ / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "host_wall_ms_per_step": round(wall_ms, 3), "steps": args.e2e_steps,
            "pipelined": True}


def memory_report(torch, vc, d, args, dev):
    """Peak device memory (MiB above the baseline) of the buffer lifetimes of
    "NCCL 专家课程 07" 显存实验, with all N virtual ranks on one GPU: inputs
    are copies of the workload made inside each measurement.  The page's
    optimised lifetime frees the input after a synchronize; the stream-
    ordered one (lifetimes.all_reduce_decomposed_low_peak) needs none."""
    n, M = len(d), d[0].numel()
    q = vc.vc_shard_count(M, n)
    MiB = float(1 << 20)
    out = {}

    def measure(name, fn):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        kept = fn()
        torch.cuda.synchronize()
        peak = torch.cuda.max_memory_allocated(dev) - base
        steady = torch.cuda.memory_allocated(dev) - base
        out[name] = {"peak": round(peak / MiB, 1), "steady": round(steady / MiB, 1)}
        del kept

    def ar_in_place():
        full = [t.clone() for t in d]
        vc.vc_all_reduce(full, None, op=args.op, order=args.order)
        return full

    def ar_out_of_place():
        full = [t.clone() for t in d]
        res = [torch.empty_like(t) for t in full]
        vc.vc_all_reduce(full, res, op=args.op, order=args.order)
        del full
        return res

    def rs_only():
        full = [t.clone() for t in d]
        shard = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
        vc.vc_reduce_scatter(full, shard, op=args.op, order=args.order)
        torch.cuda.synchronize()
        del full
        return shard

    def rs_ag_naive():
        full = [t.clone() for t in d]
        shard = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
        gathered = [torch.empty_like(t) for t in full]
        vc.vc_reduce_scatter(full, shard, op=args.op, order=args.order)
        vc.vc_all_gather(shard, gathered)
        torch.cuda.synchronize()
        del full, shard
        return gathered

    def rs_ag_optimized():
        full = [t.clone() for t in d]
        shard = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
        vc.vc_reduce_scatter(full, shard, op=args.op, order=args.order)
        torch.cuda.synchronize()
        del full
        gathered = [torch.empty(M, dtype=d[0].dtype, device=dev) for _ in range(n)]
        vc.vc_all_gather(shard, gathered)
        torch.cuda.synchronize()
        del shard
        return gathered

    def rs_ag_stream_ordered():
        from allreduce_reducescatter_allgather_gb300 import lifetimes
        return lifetimes.all_reduce_decomposed_low_peak([t.clone() for t in d], op=args.op,
                                                        order=args.order)

    for name, fn in (("allreduce_in_place", ar_in_place),
                     ("allreduce_out_of_place", ar_out_of_place),
                     ("reduce_scatter_only", rs_only), ("rs_ag_naive", rs_ag_naive),
                     ("rs_ag_optimized", rs_ag_optimized),
                     ("rs_ag_stream_ordered", rs_ag_stream_ordered)):
        measure(name, fn)
    return out


def latency_table(torch, vc, args, dev):
    """p1's direct-vs-decomposed experiment on four virtual ranks ("NCCL 专家
    课程 07", 性能实验为什么交替执行顺序 / 严格处理不稳定点): per-rank sizes 1 KiB,
    64 KiB, 1 MiB, 16 MiB, 256 MiB of fp32; 3 warm-ups, then 10 cycles that
    alternate which path runs first; inputs reset and synchronised outside
    each timed call; median / P95 / CV of the per-call CUDA-event times; the
    decomposed / direct ratio is given only when both CVs are at most 5 %."""
    import numpy as np
    n = 4
    stream = torch.cuda.current_stream(dev)
    rows = []
    for nbytes in (1 << 10, 64 << 10, 1 << 20, 16 << 20, 256 << 20):
        M = nbytes // 4
        g = torch.Generator(device=dev)
        g.manual_seed(nbytes)
        base = [torch.randn(M, generator=g, device=dev) for _ in range(n)]
        work = [t.clone() for t in base]
        shards = [torch.empty(vc.vc_shard_count(M, n), device=dev) for _ in range(n)]

        def reset():
            for w, b in zip(work, base):
                w.copy_(b)
            torch.cuda.synchronize()

        # prepared calls: checked once, one C call each (the first C call on
        # the stream, as a user with persistent buffers would issue it)
        ar = vc.prepare_all_reduce(work, None, op=args.op, order=args.order)
        dec = vc.prepare_all_reduce_decomposed(work, shards, None, op=args.op,
                                               order=args.order)

        def direct():
            ar(stream=stream)

        def decomposed():
            dec(stream=stream)

        def timed(fn):
            reset()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b) * 1e3  # µs

        for _ in range(3):
            timed(direct)
            timed(decomposed)
        t = {"direct": [], "decomposed": []}
        for cycle in range(10):
            order = ("direct", "decomposed") if cycle % 2 == 0 else ("decomposed", "direct")
            for mode in order:
                t[mode].append(timed(direct if mode == "direct" else decomposed))
        row = {"bytes_per_rank": nbytes}
        for mode, v in t.items():
            a = np.array(v)
            med = float(np.median(a))
            row[mode] = {"median_us": round(med, 3), "p95_us": round(float(np.percentile(a, 95)), 3),
                         "cv": round(float(a.std() / a.mean()), 4),
                         "payload_gbs": round(nbytes * n / med / 1e3, 2),
                         "hbm_gbs": round(step_bytes(n, M, 4)["fused_ar" if mode == "direct"
                                                               else "decomposed_ar"] / med / 1e3, 1)}
        stable = row["direct"]["cv"] <= 0.05 and row["decomposed"]["cv"] <= 0.05
        row["decomposed_over_direct"] = (round(row["decomposed"]["median_us"]
                                               / row["direct"]["median_us"], 3)
                                         if stable else "unstable")
        rows.append(row)
        del base, work, shards, ar, dec
    torch.cuda.empty_cache()
    return rows


def transformer_grad_shapes(layers: int = 12, hidden: int = 1024, vocab: int = 32000):
    """Gradient shapes of a small synthetic transformer (forward order):
    token embedding, then per layer two layer norms and four linear layers
    with biases."""
    h = hidden
    shapes = [(vocab, h)]
    for _ in range(layers):
        shapes += [(h,), (h,), (3 * h, h), (3 * h,), (h, h), (h,),
                   (h,), (h,), (4 * h, h), (4 * h,), (h, 4 * h), (h,)]
    return shapes


def bucket_report(torch, vc, args, dev):
    """One AllReduce per gradient tensor against one per 25 MiB bucket (the
    pages' DDP buckets), on 8 virtual ranks of bf16 gradients: with the
    gradients as bucket views (no copy), with packing (three launches per
    bucket) and fused (one launch per bucket, the tensors reduced where they
    are); the per-tensor and bucket loops also replayed from a CUDA graph
    (launch cost amortised); the buckets' ReduceScatter into per-rank
    shards (ZeRO), from the views, packed, and fused; and the fused
    AllGather of the shards back into the tensors (FSDP's unpack)."""
    from allreduce_reducescatter_allgather_gb300 import bucketing
    n = 8
    shapes = transformer_grad_shapes()
    gb = bucketing.GradientBuckets(shapes, torch.bfloat16, n, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(99)
    grads = [[torch.randn(s, generator=g, device=dev).to(torch.bfloat16) for s in shapes]
             for _ in range(n)]
    gb.bind(grads)
    total = sum(t.numel() for t in grads[0]) * 2
    stream = torch.cuda.current_stream(dev)

    singles = [vc.prepare_all_reduce([grads[r][t] for r in range(n)], None, op=args.op,
                                     order=args.order) for t in range(len(shapes))]

    # each loop runs on the current stream: the bench's, or the capture
    # stream while a CUDA graph records it
    def per_tensor():
        for c in singles:
            c()

    def views():
        gb.all_reduce(op=args.op, order=args.order)

    def packed():
        gb.all_reduce_tensors(op=args.op, order=args.order, fused=False)

    def fused():
        gb.all_reduce_tensors(op=args.op, order=args.order, fused=True)

    def t_ms(fn, reps=10):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def graphed(fn):
        """The loop captured once in a CUDA graph; each call replays it."""
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
        return g.replay

    graphs = []

    def rs_views():
        gb.reduce_scatter(op=args.op, order=args.order)

    def rs_packed():
        gb.reduce_scatter_tensors(op=args.op, order=args.order, fused=False)

    def rs_fused():
        gb.reduce_scatter_tensors(op=args.op, order=args.order, fused=True)

    def ag_fused():
        gb.all_gather_tensors()

    ar_bytes = 2 * n * total
    rs_bytes = n * total + total
    out = {"ranks": n, "dtype": "bf16", "tensors": len(shapes), "buckets": len(gb.buckets),
           "bytes_per_rank": total}
    for name, fn, launches in (("per_tensor", per_tensor, len(shapes)),
                               ("per_tensor_graph", graphed(per_tensor), len(shapes)),
                               ("bucket_views", views, len(gb.buckets)),
                               ("bucket_views_graph", graphed(views), len(gb.buckets)),
                               ("bucket_packed", packed, 3 * len(gb.buckets))) + (
            (("bucket_fused", fused, len(gb.buckets)),) if gb.fused_supported(args.order)
            else ()):
        ms = t_ms(fn)
        out[name] = {"us": round(ms * 1e3, 1), "allreduce_gbs": round(ar_bytes / ms / 1e6, 1),
                     "launches": launches}
    # ZeRO: the buckets' ReduceScatter into per-rank shards
    for name, fn, launches in (("rs_bucket_views", rs_views, len(gb.buckets)),
                               ("rs_bucket_packed", rs_packed, 2 * len(gb.buckets))) + (
            (("rs_bucket_fused", rs_fused, len(gb.buckets)),) if gb.fused_supported(args.order)
            else ()):
        ms = t_ms(fn)
        out[name] = {"us": round(ms * 1e3, 1),
                     "reduce_scatter_gbs": round(rs_bytes / ms / 1e6, 1), "launches": launches}
    # FSDP's unpack: the shards gathered back into the tensors
    gb.reduce_scatter(op=args.op, order=args.order)
    ms = t_ms(ag_fused)
    out["ag_bucket_fused"] = {"us": round(ms * 1e3, 1),
                              "all_gather_gbs": round(rs_bytes / ms / 1e6, 1),
                              "launches": len(gb.buckets)}
    del grads, gb, singles, graphs
    torch.cuda.empty_cache()
    return out


def run_sweep(args):
    """The size x rank-count sweep (per-rank bytes 8 KiB * 4^k and 1 GiB, N in
    {2, 4, 8, 16, 64}, N * bytes <= 64 GiB) over the four element types: one
    JSON line per point with RS / AG / fused AR GB/s and their fraction of the
    measured copy peak (SUM, the order given by --order).  Inputs are made on
    the device; each kernel's time is the median of 5 single calls after 3
    warm-ups.  Before each call a read of twice the L2 evicts the last
    call's data, and it keeps the GPU busy while the host issues the call:
    the events then time the call on the device, launch latency included,
    without the host's time to reach the launch.  (A write would leave the
    L2 full of dirty lines, up to 126 MB that the timed call would have to
    write back: measured, that cost N = 2 ReduceScatter at 64 MiB per rank
    a fifth of its rate.  After a read the lines are clean, and at 256 MiB
    per rank a single call then measures what the back-to-back bench does.)
    Points with 64 MiB to 4 GiB of input per call also get "sustained":
    back-to-back calls over enough buffer sets that every call reads from
    HBM and meets the previous calls' dirty lines in L2, as in a training
    loop."""
    import torch

    import allreduce_reducescatter_allgather_gb300 as vc
    import synthetic_inputs as si
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = measured_peak()
    stream = torch.cuda.current_stream(dev)

    # a buffer twice the L2: reading it between calls evicts the last call's
    # data, so points whose data would fit in L2 are still timed from HBM
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def t_ms(fn, reps=5):
        for _ in range(3):
            fn()
        times = []
        for _ in range(reps):
            torch.sum(flush, dim=0, out=sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        return sorted(times)[len(times) // 2]

    def sustained(n, M, dtype, dist, kw, d, z, b, set_bytes):
        """Back-to-back calls, the way a training loop issues them: K sets
        of buffers whose inputs together exceed twice the L2 are taken in
        turn, so every call reads from HBM and finds the L2 full of the
        previous calls' dirty lines.  Per-call average over 3 rounds."""
        K = -(-2 * l2 // set_bytes) + 1
        sets = [(d, z)]
        for k in range(1, K):
            dk = si.generate_device(torch, dtype, dist, n, M, si.SEED_BASE + 40 + k, dev, **kw)
            sets.append((dk, [torch.empty_like(t) for t in z]))
        out = {"sets": K}
        for name, key in (("reduce_scatter", "reduce_scatter"), ("all_gather", "all_gather"),
                          ("all_reduce", "fused_ar")):
            calls = []
            for dk, zk in sets:
                if name == "reduce_scatter":
                    calls.append(vc.prepare_reduce_scatter(dk, zk, op=args.op, order=args.order))
                elif name == "all_gather":
                    calls.append(vc.prepare_all_gather(zk, dk))
                else:
                    calls.append(vc.prepare_all_reduce(dk, None, op=args.op, order=args.order))
            for c in calls:  # warm-up round
                c(stream=stream)
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(3):
                for c in calls:
                    c(stream=stream)
            e.record(stream)
            e.synchronize()
            ms = a.elapsed_time(e) / (3 * K)
            g = b[key] / (ms / 1e3) / 1e9
            out[name] = {"us": round(ms * 1e3, 2), "gbs": round(g, 1), "frac": round(g / peak, 4)}
        del sets
        return out

    for n, nbytes in si.sweep_points():
        if args.order == "recursive_halving" and n & (n - 1):
            continue
        for dtype in ("float32", "bfloat16", "int32", "int64"):
            es = ESIZE[dtype]
            M = nbytes // es
            dist = "uniform_pm1" if dtype in ("float32", "bfloat16") else "uniform_int"
            kw = {} if dist == "uniform_pm1" else {"lo": -100, "hi": 100}
            d = si.generate_device(torch, dtype, dist, n, M, si.SEED_BASE + 4, dev, **kw)
            q = vc.vc_shard_count(M, n)
            z = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
            rs = vc.prepare_reduce_scatter(d, z, op=args.op, order=args.order)
            ag = vc.prepare_all_gather(z, d)  # AG writes over the inputs, after RS
            ar = vc.prepare_all_reduce(d, None, op=args.op, order=args.order)  # in place
            b = step_bytes(n, M, es)
            line = {"sweep": "size_x_ranks", "n": n, "bytes_per_rank": nbytes, "dtype": dtype,
                    "op": args.op, "order": args.order, "peak": peak, "peak_kind": kind,
                    "timing": "median of 5 single calls, each after an L2-evicting read"}
            for name, fn, key in (("reduce_scatter", rs, "reduce_scatter"),
                                  ("all_gather", ag, "all_gather"),
                                  ("all_reduce", ar, "fused_ar")):
                ms = t_ms(lambda: fn(stream=stream))
                g = b[key] / (ms / 1e3) / 1e9
                line[name] = {"us": round(ms * 1e3, 2), "gbs": round(g, 1),
                              "frac": round(g / peak, 4)}
            set_bytes = n * nbytes
            if 64 << 20 <= set_bytes <= 4 << 30:
                line["sustained"] = sustained(n, M, dtype, dist, kw, d, z, b, set_bytes)
            print(json.dumps(line), flush=True)
            del d, z, rs, ag, ar
            torch.cuda.empty_cache()
    return 0


def main(argv=None):
    import synthetic_inputs as si
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="n4_256mib_f32_normal", choices=sorted(si.WORKLOADS))
    ap.add_argument("--op", default="sum", choices=["sum", "prod", "max", "min", "avg"])
    ap.add_argument("--order", default="ring",
                    choices=["ring", "recursive_halving", "pairwise_tree"])
    ap.add_argument("--elements", type=int, default=0,
                    help="override the elements per rank (small cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--dist-timeout", type=float, default=300.0,
                    help="seconds a rank waits in a collective for the others (torchrun)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="run the size x rank-count sweep instead (one JSON line per point)")
    ap.add_argument("--no-memory", action="store_true",
                    help="skip the memory-lifetime, gradient-bucket and latency reports")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    workload = dict(si.WORKLOADS[args.workload])
    if args.elements > 0:
        workload["M"] = args.elements
    if args.impl == "reference":
        return run_reference(args, workload)
    if args.sweep:
        import __graft_entry__
        __graft_entry__.build()
        return run_sweep(args)
    if dist_info()[0] == 1:
        import __graft_entry__
        __graft_entry__.build()  # under torchrun the library must be built beforehand
    return run_ours(args, workload)


if __name__ == "__main__":
    sys.exit(main())
