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

Beside the headline the line carries (one GPU only):
  configs               every workload: the worked example, 8 x 1,000,003
                        fp32, the 25 MiB bf16 bucket, 4 x 256 MiB fp32 and
                        4 x 512 MiB int64, and a 64 MiB / 1 GiB per rank
                        summary of the size x rank-count sweep.  Each path
                        with per-call median / P95 / CV (path order
                        alternating each cycle), algorithmic bytes, GB/s and
                        fraction of the copy peak, and an oracle check of
                        that run's outputs (every element, or sampled
                        indices with every chunk boundary at full size);
  direct_vs_decomposed  single calls and CUDA-graph loops of 16 calls from
                        1 KiB to 256 MiB per rank;
  e2e                   the step from pinned host buffers, with the host
                        link probed in the same run;
  memory_mib, gradient_buckets, cpu_baseline, cpu_baseline_all_cores.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(the path shards by index range with no exchange; weak scaling), the step
time is the max over ranks, and value counts the bytes of all ranks.  The
ranks talk only over a host-side gloo group (a barrier, a max and a sum).
--impl reference times the CPU oracle instead, on a bounded window of the
same workload (rank 0 only).  Single cases for profiling: --one (one
collective on one shape), --bucket-path (one gradient-bucket collective),
--sweep (the size x rank-count sweep).
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
    """Max step time and total bytes over ranks (control plane only: two
    host scalars over the gloo process group; no GPU collective)."""
    if world == 1:
        return local_ms, local_bytes
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64)
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
        # The control plane (a barrier around the timed region and the
        # max / sum of two scalars) runs on the host over gloo: the ranks
        # exchange no data, so no GPU collective library is involved.  A rank
        # that dies or never arrives ends the others' next collective with an
        # error after this long, instead of leaving them waiting.
        dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=args.dist_timeout))

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

    del y, y2, sh
    torch.cuda.empty_cache()
    memory = memory_report(torch, vc, d, args, dev) if not args.no_memory else None
    buckets = bucket_report(torch, vc, args, dev) if not args.no_memory else None
    latency = latency_table(torch, vc, args, dev, peak) if not args.no_memory else None
    e2e = e2e_measure(torch, vc, d, args, dev, stream, by["step"])
    configs = (configs_report(torch, vc, args, dev, stream, peak, d, memory)
               if (world == 1 and not args.no_configs
                   and M == si.WORKLOADS[args.workload]["M"]) else None)

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
    if configs is not None:
        line["configs"] = configs
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
            line["cpu_baseline_all_cores"] = {
                "value": round(gp, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                "cpu": line["cpu_baseline"]["cpu"],
                "sample": f"{psteps} oracle steps in {cores} spawned processes, each on its "
                          f"own {min(1 << 22, M)}-element window of every rank, "
                          f"{psecs:.1f} s"}
        except Exception as e:  # the single-core figure above still stands
            line["cpu_baseline_all_cores"] = {"error": f"{type(e).__name__}: {e}"[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def link_probe(torch, dev, nbytes: int = 1 << 30, reps: int = 3) -> dict:
    """The host link in this run: pinned 1 GiB host-to-device and device-to-
    host copies alone, and both at once on two streams (best of `reps`, CUDA
    events), in GB/s."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    h_in.fill_(1)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def best(kind):
        out = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(s1)
            if kind in ("h2d", "both"):
                with torch.cuda.stream(s1):
                    d_a.copy_(h_in, non_blocking=True)
            if kind in ("d2h", "both"):
                s2.wait_event(a)
                with torch.cuda.stream(s2):
                    h_out.copy_(d_b, non_blocking=True)
                s1.wait_stream(s2)
            b.record(s1)
            b.synchronize()
            moved = nbytes * (2 if kind == "both" else 1)
            out.append(moved / (a.elapsed_time(b) / 1e3) / 1e9)
        return round(max(out), 1)

    res = {"h2d_gbs": best("h2d"), "d2h_gbs": best("d2h"), "both_gbs": best("both"),
           "bytes": nbytes, "how": f"pinned {nbytes >> 20} MiB copies, best of {reps}"}
    del h_in, h_out, d_a, d_b
    torch.cuda.empty_cache()
    return res


def e2e_measure(torch, vc, d, args, dev, stream, step_bytes_):
    """The same step through the public API with the inputs in pinned host
    memory: each step copies the N inputs in, runs both AllReduce paths and
    copies every output of both back.  Each buffer set's N rank buffers are
    views of one contiguous allocation (host and device alike), so a step
    issues one host-to-device copy and two device-to-host copies (the fused
    and the decomposed outputs).  Steps are pipelined the way a user would
    run them: two sets of device buffers and of host outputs, one stream per
    direction, so step k+1's inputs travel while step k's outputs come back.
    The host link is probed in the same run, and the step's host traffic is
    reported as a fraction of the both-directions rate."""
    n, M = len(d), d[0].numel()
    dt = d[0].dtype
    q = vc.vc_shard_count(M, n)
    link = link_probe(torch, dev)
    host_in = torch.empty(n * M, dtype=dt, pin_memory=True)
    for r in range(n):
        host_in[r * M:(r + 1) * M].copy_(d[r])

    def views(flat, count):
        return [flat[r * count:(r + 1) * count] for r in range(n)]

    sets = []
    for _ in range(2):
        flat = [torch.empty(n * M, dtype=dt, device=dev) for _ in range(3)]
        sh = torch.empty(n * q, dtype=dt, device=dev)
        sets.append((flat, views(flat[0], M), views(flat[1], M), views(sh, q), views(flat[2], M)))
    host_out = [(torch.empty(n * M, dtype=dt, pin_memory=True),
                 torch.empty(n * M, dtype=dt, pin_memory=True)) for _ in range(2)]
    h2d = host_in.numel() * host_in.element_size()
    d2h = 2 * h2d
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    calls = [(vc.prepare_all_reduce(di, dy, op=args.op, order=args.order),
              vc.prepare_all_reduce_decomposed(di, dsh, dy2, op=args.op, order=args.order))
             for _, di, dy, dsh, dy2 in sets]

    phases = []  # per timed step: events around its host-to-device and device-to-host copies

    def run(steps, timed=False):
        for k in range(steps):
            j = k % 2
            flat = sets[j][0]
            hy, hy2 = host_out[j]
            marks = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if timed else None
            if k >= 2:
                s_in.wait_event(comp_done[j])  # set j's inputs no longer read
            with torch.cuda.stream(s_in):
                if marks:
                    marks[0].record(s_in)
                flat[0].copy_(host_in, non_blocking=True)
                if marks:
                    marks[1].record(s_in)
            in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            if k >= 2:
                stream.wait_event(out_done[j])  # set j's outputs already copied out
            ar, dec = calls[j]
            ar(stream=stream)
            dec(stream=stream)
            comp_done[j].record(stream)
            s_out.wait_event(comp_done[j])
            with torch.cuda.stream(s_out):
                if marks:
                    marks[2].record(s_out)
                hy.copy_(flat[1], non_blocking=True)
                hy2.copy_(flat[2], non_blocking=True)
                if marks:
                    marks[3].record(s_out)
            out_done[j].record(s_out)
            if marks:
                phases.append(marks)

    run(2)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(args.e2e_steps, timed=True)
    s_in.wait_stream(s_out)
    s_in.wait_stream(stream)
    b.record(s_in)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.e2e_steps
    wall_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    # the last step's outputs came back intact: both paths, every rank
    last = (args.e2e_steps - 1) % 2
    assert torch.equal(host_out[last][0], sets[last][0][1].cpu())
    assert torch.equal(host_out[last][1], sets[last][0][2].cpu())
    del sets, host_out, calls
    torch.cuda.empty_cache()
    host_gbs = (h2d + d2h) / (ms / 1e3) / 1e9
    link["e2e_host_gbs"] = round(host_gbs, 1)
    link["e2e_frac_of_both"] = round(host_gbs / link["both_gbs"], 4) if link["both_gbs"] else None
    serial_ms = (h2d / link["h2d_gbs"] + d2h / link["d2h_gbs"]) / 1e6
    link["serial_link_ms_per_step"] = round(serial_ms, 3)
    # where the step's time goes: each direction's copy time per step (its
    # events on its own stream) and the share of the step the device-to-host
    # stream spent copying (1.0: the outbound link never waited for compute)
    h2d_ms = sum(m[0].elapsed_time(m[1]) for m in phases) / len(phases)
    d2h_ms = sum(m[2].elapsed_time(m[3]) for m in phases) / len(phases)
    link["h2d_ms_per_step"] = round(h2d_ms, 3)
    link["d2h_ms_per_step"] = round(d2h_ms, 3)
    link["d2h_busy_frac"] = round(d2h_ms / ms, 4)
    # the rates the copies reached inside the step, against the probe's
    # best-of-3 above: the host link is shared with whatever else runs on
    # the host, and the step gets what is left of it
    link["h2d_gbs_in_step"] = round(h2d / (h2d_ms / 1e3) / 1e9, 1)
    link["d2h_gbs_in_step"] = round(d2h / (d2h_ms / 1e3) / 1e9, 1)
    return {"value": round(step_bytes_ / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3),
            "host_wall_ms_per_step": round(wall_ms, 3), "steps": args.e2e_steps,
            "pipelined": True, "copies_per_step": {"h2d": 1, "d2h": 2}, "link": link}


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


def latency_table(torch, vc, args, dev, peak, K: int = 16):
    """p1's direct-vs-decomposed experiment on four virtual ranks ("NCCL 专家
    课程 07", 性能实验为什么交替执行顺序 / 严格处理不稳定点): per-rank sizes 1 KiB,
    64 KiB, 1 MiB, 16 MiB, 256 MiB of fp32, out of place (the inputs never
    change, so no reset is needed); 3 warm-ups, then 10 cycles that
    alternate which path runs first; median / P95 / CV per path; the
    decomposed / direct ratio only when both CVs are at most 5 %.  Two
    timings per size:
      single  one call per event pair, after an L2-evicting read that keeps
              the GPU busy while the host issues the call (device time of one
              call, launch included);
      graph   a CUDA graph of K back-to-back calls per event pair, the time
              divided by K (what a loop of calls costs per call; the host's
              per-call jitter does not enter)."""
    n = 4
    stream = torch.cuda.current_stream(dev)
    single = CallTimer(torch, dev, stream)
    plain = CallTimer(torch, dev, stream, evict=False)
    rows = []
    for nbytes in (1 << 10, 64 << 10, 1 << 20, 16 << 20, 256 << 20):
        M = nbytes // 4
        g = torch.Generator(device=dev)
        g.manual_seed(nbytes)
        x = [torch.randn(M, generator=g, device=dev) for _ in range(n)]
        y = [torch.empty_like(t) for t in x]
        y2 = [torch.empty_like(t) for t in x]
        shards = [torch.empty(vc.vc_shard_count(M, n), device=dev) for _ in range(n)]
        ar = vc.prepare_all_reduce(x, y, op=args.op, order=args.order)
        dec = vc.prepare_all_reduce_decomposed(x, shards, y2, op=args.op, order=args.order)
        b = step_bytes(n, M, 4)
        row = {"bytes_per_rank": nbytes}

        def finish(t, scale):
            r = {"direct": call_stats([v / scale for v in t["direct"]], b["fused_ar"], peak),
                 "decomposed": call_stats([v / scale for v in t["decomposed"]],
                                          b["decomposed_ar"], peak)}
            for mode in ("direct", "decomposed"):
                r[mode]["payload_gbs"] = round(nbytes * n / r[mode]["mean_us"] / 1e3, 2)
            stable = r["direct"]["stable"] and r["decomposed"]["stable"]
            r["decomposed_over_direct"] = (round(r["decomposed"]["mean_us"]
                                                 / r["direct"]["mean_us"], 3)
                                           if stable else "unstable")
            return r

        row["single"] = finish(single.alternating([("direct", lambda: ar(stream=stream)),
                                                   ("decomposed", lambda: dec(stream=stream))]), 1)
        graphs = {name: graph_loop(torch, fn, K) for name, fn in (("direct", ar),
                                                                   ("decomposed", dec))}
        row["graph"] = finish(plain.alternating([("direct", graphs["direct"].replay),
                                                 ("decomposed", graphs["decomposed"].replay)]), K)
        row["graph"]["calls_per_replay"] = K
        rows.append(row)
        del x, y, y2, shards, ar, dec, graphs
    torch.cuda.empty_cache()
    return rows


# ------------------------------------------------- every configuration --

class CallTimer:
    """Per-call CUDA-event times on one stream, the method of "NCCL 专家课程
    07", 性能实验: warm-ups, then cycles in which the order of the paths
    alternates (forward on even cycles, reversed on odd ones).  Before every
    timed call a read of twice the L2 evicts the last call's data (so small
    configurations are timed from HBM too) and keeps the GPU busy while the
    host issues the call, so the events time the call on the device, launch
    included, without the host's time to reach it.  (A read leaves the lines
    clean; an evicting write would leave dirty lines for the timed call to
    write back.)"""

    def __init__(self, torch, dev, stream, evict: bool = True):
        self.torch, self.stream = torch, stream
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.flush = (torch.ones(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)
                      if evict else None)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def alternating(self, paths, cycles: int = 10, warmup: int = 3) -> dict:
        """paths: [(name, fn)], each fn issuing one call on the stream.
        Returns {name: [ms per call, one per cycle]}."""
        torch = self.torch
        for _ in range(warmup):
            for _, fn in paths:
                fn()
        torch.cuda.synchronize()
        out = {name: [] for name, _ in paths}
        for k in range(cycles):
            seq = paths if k % 2 == 0 else paths[::-1]
            evs = []
            for name, fn in seq:
                if self.flush is not None:
                    torch.sum(self.flush, dim=0, out=self.sink)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                fn()
                b.record(self.stream)
                evs.append((name, a, b))
            torch.cuda.synchronize()
            for name, a, b in evs:
                out[name].append(a.elapsed_time(b))
        return out


def graph_loop(torch, fn, K: int):
    """fn (one call on the current stream) captured K times back to back in
    a CUDA graph; returns the graph's replay (one launch of K calls)."""
    fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(K):
            fn()
    return gr


def call_stats(ms: list, nbytes: int, peak: float) -> dict:
    """Median / P95 / CV of per-call times, and the HBM rate against the copy
    peak.  "stable" (CV <= 5 %) marks the figures a ratio may be claimed from
    ("NCCL 专家课程 07", 严格处理不稳定点).  The rate (and every ratio taken
    from these figures) uses mean_us, the mean of the calls left after the
    fastest and the slowest tenth are dropped: on the GB300 machines measured
    here the CUDA event clock advances in steps of 2.048 us, so each call's
    time is a multiple of that step and a median sits on that grid (up to
    1 us off, a few per cent of a 30 us call), while the mean over calls
    that start at varying phases of the clock does not."""
    import numpy as np
    a = np.sort(np.asarray(ms, dtype=np.float64))
    med = float(np.median(a))
    k = a.size // 10
    t = float(a[k:a.size - k].mean())
    g = nbytes / (t / 1e3) / 1e9
    cv = float(a.std() / a.mean()) if a.mean() > 0 else 0.0
    return {"median_us": round(med * 1e3, 2), "mean_us": round(t * 1e3, 2),
            "p95_us": round(float(np.percentile(a, 95)) * 1e3, 2),
            "cv": round(cv, 4), "calls": int(a.size), "bytes": int(nbytes), "gbs": round(g, 1),
            "frac": round(g / peak, 4), "stable": cv <= 0.05}


def host_bits(t, dtype: str):
    """A device tensor's bytes as a numpy array of the oracle's storage type
    (bf16 as raw uint16 bits)."""
    import numpy as np
    if dtype == "bfloat16":
        import torch
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _bits(a):
    import numpy as np
    a = np.ascontiguousarray(a)
    return a.view({1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[a.itemsize])


class Check:
    """Bitwise comparison of GPU outputs with the oracle, counted."""

    def __init__(self, kind: str):
        self.kind, self.compared, self.mismatches, self.outputs = kind, 0, 0, set()

    def eq(self, name: str, got, want):
        import numpy as np
        g, w = _bits(got), _bits(want)
        self.outputs.add(name)
        self.compared += int(w.size)
        self.mismatches += int(np.count_nonzero(g != w)) if g.shape == w.shape else int(w.size)

    def summary(self, **extra) -> dict:
        return {"kind": self.kind, "outputs": sorted(self.outputs), "elements": self.compared,
                "mismatches": self.mismatches, "bit_exact": self.mismatches == 0, **extra}


def sample_indices(M: int, n: int, q: int, k: int = 4096, seed: int = 0):
    """k random indices of [0, M) plus both sides of every chunk boundary
    and the two ends, sorted."""
    import numpy as np
    rng = np.random.default_rng(seed)
    idx = set(int(i) for i in rng.integers(0, M, size=min(k, M)))
    for c in range(1, n):
        for i in (c * q - 1, c * q):
            if 0 <= i < M:
                idx.add(i)
    idx.update((0, M - 1))
    return np.array(sorted(idx), dtype=np.int64)


def sampled_operands(torch, d, idx, dtype):
    """Every rank's operand at the sampled indices, read from the device."""
    it = torch.from_numpy(idx).to(d[0].device)
    return [host_bits(t[it], dtype) for t in d]


def check_rs_sampled(chk, torch, z, idx, want, n, M, q, dtype, op, name="RS"):
    """Shard c = floor(i/q) at i - cq against the oracle's value at i, and
    the padded tail of the last shard against the op's identity (0 for AVG)."""
    import numpy as np
    import oracle
    for c in range(n):
        sel = np.flatnonzero((idx // q) == c)
        if sel.size == 0:
            continue
        off = torch.from_numpy(idx[sel] - c * q).to(z[c].device)
        chk.eq(name, host_bits(z[c][off], dtype), want[sel])
    tail = n * q - M
    if tail > 0:
        e = np.zeros(1, oracle.NP_STORAGE[dtype]) if op == "avg" else \
            np.full(1, oracle.identity(dtype, op), oracle.NP_STORAGE[dtype])
        chk.eq(name + " padding", host_bits(z[n - 1][q - tail:], dtype), np.repeat(e, tail))


def check_full_sampled(chk, torch, name, outs, idx, want, dtype):
    """Every output tensor at the sampled indices."""
    it = torch.from_numpy(idx).to(outs[0].device)
    for t in outs:
        chk.eq(name, host_bits(t[it], dtype), want)


def config_c1(torch, vc, dev, stream, peak):
    """The pages' worked example: four ranks, twenty int64, x = 100r + i.
    SUM (600 + 4i, shards of five) and MAX (300 + i), ring order, direct
    AllReduce against ReduceScatter + AllGather, every output against the
    oracle and the closed forms; the two negative checks must fail (a rolled
    gather, and MAX with zero padding on M = 19 all-negative inputs).  Tiny:
    latency only."""
    import numpy as np
    import oracle
    import synthetic_inputs as si
    n, M = 4, 20
    xs = si.generate("int64", "rank_linear", n, M, seed=0)
    d = [torch.from_numpy(x.copy()).to(dev) for x in xs]
    q = vc.vc_shard_count(M, n)
    chk = Check("full")
    timer = CallTimer(torch, dev, stream)
    loops = CallTimer(torch, dev, stream, evict=False)
    K = 16
    out = {"config": "N=4, M=20 int64, x = 100r + i; SUM and MAX; ring; direct AR vs RS+AG",
           "q": q, "timing": "single: one call per event pair after an L2-evicting read; "
                             f"graph: {K} calls per CUDA-graph replay, time / {K}", "ops": {}}
    closed = {"sum": 600 + 4 * np.arange(M), "max": 300 + np.arange(M)}
    for op in ("sum", "max"):
        y = [torch.empty_like(t) for t in d]
        z = [torch.empty(q, dtype=torch.int64, device=dev) for _ in range(n)]
        g = [torch.empty_like(t) for t in d]
        ar = vc.prepare_all_reduce(d, y, op=op, order="ring")
        rs = vc.prepare_reduce_scatter(d, z, op=op, order="ring")
        ag = vc.prepare_all_gather(z, g)
        dec = vc.prepare_all_reduce_decomposed(d, [torch.empty_like(t) for t in z], g,
                                               op=op, order="ring")
        ar(stream=stream)
        rs(stream=stream)
        ag(stream=stream)
        torch.cuda.synchronize()
        oy = oracle.all_reduce(xs, "int64", op, "ring")
        oz = oracle.reduce_scatter(xs, "int64", op, "ring")
        for r in range(n):
            chk.eq("AR", y[r].cpu().numpy(), oy[r])
            chk.eq("AR closed form", y[r].cpu().numpy(), closed[op])
            chk.eq("RS", z[r].cpu().numpy(), oz[r])
            chk.eq("RS+AG", g[r].cpu().numpy(), oy[r])
        t = timer.alternating([("all_reduce", lambda: ar(stream=stream)),
                               ("rs_then_ag", lambda: dec(stream=stream))])
        gl = {k: graph_loop(torch, f, K) for k, f in (("all_reduce", ar), ("rs_then_ag", dec))}
        tg = loops.alternating([(k, g.replay) for k, g in gl.items()])
        b = step_bytes(n, M, 8)
        out["ops"][op] = {
            "single": {"all_reduce": call_stats(t["all_reduce"], b["fused_ar"], peak),
                       "rs_then_ag": call_stats(t["rs_then_ag"], b["decomposed_ar"], peak)},
            "graph": {"all_reduce": call_stats([v / K for v in tg["all_reduce"]],
                                               b["fused_ar"], peak),
                      "rs_then_ag": call_stats([v / K for v in tg["rs_then_ag"]],
                                               b["decomposed_ar"], peak)}}
        del gl
    # negative checks: a gather whose shards are rolled by one rank, and MAX
    # shards padded with zero instead of the identity, must both be caught
    z = [torch.empty(q, dtype=torch.int64, device=dev) for _ in range(n)]
    vc.vc_reduce_scatter(d, z, op="sum")
    rolled = [torch.empty_like(t) for t in d]
    vc.vc_all_gather(z[1:] + z[:1], rolled)
    torch.cuda.synchronize()
    oy = oracle.all_reduce(xs, "int64", "sum", "ring")
    rolled_caught = any(not np.array_equal(rolled[r].cpu().numpy(), oy[r]) for r in range(n))
    M2 = 19
    xneg = [-(100 * r + np.arange(M2, dtype=np.int64)) - 1 for r in range(n)]
    dn = [torch.from_numpy(x).to(dev) for x in xneg]
    q2 = vc.vc_shard_count(M2, n)
    zn = [torch.empty(q2, dtype=torch.int64, device=dev) for _ in range(n)]
    vc.vc_reduce_scatter(dn, zn, op="max")
    torch.cuda.synchronize()
    oz = oracle.reduce_scatter(xneg, "int64", "max", "ring")
    for r in range(n):
        chk.eq("RS (M=19, MAX, identity padding)", zn[r].cpu().numpy(), oz[r])
    # the same shards with the padding slot filled with 0 instead of MAX's
    # identity: the comparator must tell them from the GPU's shards
    zero_pad = [o.copy() for o in oz]
    zero_pad[n - 1][q2 - (n * q2 - M2):] = 0
    zero_pad_caught = any(not np.array_equal(zn[r].cpu().numpy(), zero_pad[r]) for r in range(n))
    out["negatives"] = {"rolled_gather_caught": bool(rolled_caught),
                        "max_zero_padding_caught": bool(zero_pad_caught)}
    out["oracle_check"] = chk.summary()
    return out


def config_c2(torch, vc, dev, stream, peak):
    """Eight ranks of 1,000,003 fp32 uniform[-1, 1) (q = 125,001, five
    padding slots): SUM / MAX / MIN x ring / recursive halving x RS, AG, fused
    AR and decomposed AR, every output against the oracle, element by
    element.  The 30.5 MiB of inputs fit in L2: every timed call follows an
    L2-evicting read."""
    import oracle
    import synthetic_inputs as si
    w = si.WORKLOADS["n8_m1000003_f32_uniform"]
    n, M = w["n"], w["M"]
    xs = si.generate("float32", w["dist"], n, M, seed=w["seed"])
    d = [torch.from_numpy(x).to(dev) for x in xs]
    q = vc.vc_shard_count(M, n)
    z = [torch.empty(q, device=dev) for _ in range(n)]
    g = [torch.empty(M, device=dev) for _ in range(n)]
    y = [torch.empty(M, device=dev) for _ in range(n)]
    s2 = [torch.empty(q, device=dev) for _ in range(n)]
    y2 = [torch.empty(M, device=dev) for _ in range(n)]
    timer = CallTimer(torch, dev, stream)
    b = step_bytes(n, M, 4)
    chk = Check("full")
    out = {"config": "N=8, M=1,000,003 fp32 uniform[-1,1); SUM/MAX/MIN x ring/RH; "
                     "RS, AG, AR, decomposed; trimmed to M", "q": q, "cases": {}}
    for order in ("ring", "recursive_halving"):
        for op in ("sum", "max", "min"):
            rs = vc.prepare_reduce_scatter(d, z, op=op, order=order)
            ag = vc.prepare_all_gather(z, g)
            ar = vc.prepare_all_reduce(d, y, op=op, order=order)
            dec = vc.prepare_all_reduce_decomposed(d, s2, y2, op=op, order=order)
            t = timer.alternating([("reduce_scatter", lambda: rs(stream=stream)),
                                   ("all_gather", lambda: ag(stream=stream)),
                                   ("all_reduce", lambda: ar(stream=stream)),
                                   ("decomposed_ar", lambda: dec(stream=stream))])
            torch.cuda.synchronize()
            oz = oracle.reduce_scatter(xs, "float32", op, order)
            oy = oracle.all_reduce(xs, "float32", op, order)
            for r in range(n):
                chk.eq("RS", host_bits(z[r], "float32"), oz[r])
                chk.eq("AG", host_bits(g[r], "float32"), oy[r])
                chk.eq("AR", host_bits(y[r], "float32"), oy[r])
                chk.eq("decomposed shards", host_bits(s2[r], "float32"), oz[r])
                chk.eq("decomposed AR", host_bits(y2[r], "float32"), oy[r])
            out["cases"][f"{op}/{order}"] = {
                "reduce_scatter": call_stats(t["reduce_scatter"], b["reduce_scatter"], peak),
                "all_gather": call_stats(t["all_gather"], b["all_gather"], peak),
                "all_reduce": call_stats(t["all_reduce"], b["fused_ar"], peak),
                "decomposed_ar": call_stats(t["decomposed_ar"], b["decomposed_ar"], peak)}
    out["oracle_check"] = chk.summary()
    return out


def config_c3(torch, vc, dev, stream, peak):
    """One 25 MiB gradient bucket on eight ranks: 13,107,200 bf16 normal(0,
    1e-3) each, SUM then AVG with fp32 accumulation, ring order; the ZeRO
    ReduceScatter (shards only) and the fused AllReduce.  Every output
    against the oracle run on the device's own input bytes."""
    import oracle
    import synthetic_inputs as si
    w = si.WORKLOADS["n8_bucket25mib_bf16_normal"]
    n, M = w["n"], w["M"]
    d = si.generate_device(torch, "bfloat16", w["dist"], n, M, w["seed"], dev,
                           sigma=w["sigma"])
    xs = [host_bits(t, "bfloat16") for t in d]
    q = vc.vc_shard_count(M, n)
    z = [torch.empty(q, dtype=torch.bfloat16, device=dev) for _ in range(n)]
    y = [torch.empty_like(t) for t in d]
    timer = CallTimer(torch, dev, stream)
    b = step_bytes(n, M, 2)
    chk = Check("full")
    out = {"config": "N=8, 13,107,200 bf16 normal(0, 1e-3) (one 25 MiB bucket); SUM then AVG, "
                     "fp32 accumulation; ring; RS-only (ZeRO shards) and fused AR",
           "q": q, "cases": {}}
    for op in ("sum", "avg"):
        rs = vc.prepare_reduce_scatter(d, z, op=op, order="ring")
        ar = vc.prepare_all_reduce(d, y, op=op, order="ring")
        t = timer.alternating([("reduce_scatter_only", lambda: rs(stream=stream)),
                               ("all_reduce", lambda: ar(stream=stream))])
        torch.cuda.synchronize()
        oz = oracle.reduce_scatter(xs, "bfloat16", op, "ring")
        oy = oracle.all_reduce(xs, "bfloat16", op, "ring")
        for r in range(n):
            chk.eq("RS", host_bits(z[r], "bfloat16"), oz[r])
            chk.eq("AR", host_bits(y[r], "bfloat16"), oy[r])
        out["cases"][op] = {
            "reduce_scatter_only": call_stats(t["reduce_scatter_only"], b["reduce_scatter"], peak),
            "all_reduce": call_stats(t["all_reduce"], b["fused_ar"], peak)}
    out["oracle_check"] = chk.summary()
    return out


def config_c4(torch, vc, dev, stream, peak, workload_name, args, d=None, memory=None):
    """Four ranks of 67,108,864 elements (fp32 normal(0, 1): 256 MiB per
    rank; int64 uniform[-2^20, 2^20): 512 MiB): fused AllReduce against
    ReduceScatter + AllGather against RS-only, alternating, with the peak
    device memory of each path's buffer lifetime; sampled indices (every
    chunk boundary included) against the oracle."""
    import oracle
    import synthetic_inputs as si
    w = dict(si.WORKLOADS[workload_name])
    n, M, dtype = w.pop("n"), w.pop("M"), w.pop("dtype")
    if d is None:
        d = si.generate_device(torch, dtype, w.pop("dist"), n, M, w.pop("seed"), dev, **w)
    es = d[0].element_size()
    q = vc.vc_shard_count(M, n)
    y = [torch.empty_like(t) for t in d]
    sh = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
    y2 = [torch.empty_like(t) for t in d]
    op, order = "sum", "ring"
    ar = vc.prepare_all_reduce(d, y, op=op, order=order)
    dec = vc.prepare_all_reduce_decomposed(d, sh, y2, op=op, order=order)
    rs = vc.prepare_reduce_scatter(d, sh, op=op, order=order)
    idx = sample_indices(M, n, q, k=1 << 16)
    xs_at = sampled_operands(torch, d, idx, dtype)
    want = oracle.reduce_points(xs_at, idx, n, M, dtype, op, order)
    timer = CallTimer(torch, dev, stream)
    t = timer.alternating([("all_reduce", lambda: ar(stream=stream)),
                           ("rs_then_ag", lambda: dec(stream=stream)),
                           ("reduce_scatter_only", lambda: rs(stream=stream))])
    torch.cuda.synchronize()
    chk = Check("sampled")
    check_full_sampled(chk, torch, "AR", y, idx, want, dtype)
    check_full_sampled(chk, torch, "RS+AG", y2, idx, want, dtype)
    check_rs_sampled(chk, torch, sh, idx, want, n, M, q, dtype, op)
    b = step_bytes(n, M, es)
    out = {"config": f"N=4, {M:,} {dtype} per rank ({M * es >> 20} MiB), SUM, ring; fused AR vs "
                     "RS+AG vs RS-only", "q": q,
           "paths": {"all_reduce": call_stats(t["all_reduce"], b["fused_ar"], peak),
                     "rs_then_ag": call_stats(t["rs_then_ag"], b["decomposed_ar"], peak),
                     "reduce_scatter_only": call_stats(t["reduce_scatter_only"],
                                                       b["reduce_scatter"], peak)},
           "oracle_check": chk.summary(indices=int(idx.size))}
    med = {k: v["mean_us"] for k, v in out["paths"].items()}
    out["rs_then_ag_over_all_reduce"] = (round(med["rs_then_ag"] / med["all_reduce"], 3)
                                         if out["paths"]["all_reduce"]["stable"]
                                         and out["paths"]["rs_then_ag"]["stable"] else "unstable")
    del y, y2, sh, ar, dec, rs
    torch.cuda.empty_cache()
    if memory is not None:
        out["memory_mib"] = memory
    elif not args.no_memory:
        out["memory_mib"] = memory_report(torch, vc, d, args, dev)
    return out


def config_c5(torch, vc, dev, stream, peak):
    """The size x rank-count sweep, summarised: 64 MiB and 1 GiB per rank,
    N in {2, 4, 8, 16, 64}, int32 / int64 / fp32 / bf16, SUM, ring order.
    Per point RS, AG and the fused AllReduce (in place) alternate, 3 warm-ups
    and 10 cycles, each call after an L2-evicting read (at 2 x 64 MiB the
    data is about the size of the L2, so the previous call's lines would
    otherwise decide the time); before the timing, a sampled check against
    the oracle (RS shards, the AllReduce, and the AllGather of the shards)."""
    import oracle
    import synthetic_inputs as si
    timer = CallTimer(torch, dev, stream)
    rows = []
    for nbytes in (64 << 20, 1 << 30):
        for n in (2, 4, 8, 16, 64):
            for dtype in ("float32", "bfloat16", "int32", "int64"):
                es = ESIZE[dtype]
                M = nbytes // es
                dist = "uniform_pm1" if dtype in ("float32", "bfloat16") else "uniform_int"
                kw = {} if dist == "uniform_pm1" else {"lo": -100, "hi": 100}
                d = si.generate_device(torch, dtype, dist, n, M, si.SEED_BASE + 4, dev, **kw)
                q = vc.vc_shard_count(M, n)
                z = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
                idx = sample_indices(M, n, q, k=1 << 12, seed=n)
                xs_at = sampled_operands(torch, d, idx, dtype)
                rs = vc.prepare_reduce_scatter(d, z, op="sum", order="ring")
                ar = vc.prepare_all_reduce(d, None, op="sum", order="ring")  # in place
                ag = vc.prepare_all_gather(z, d)  # writes over the inputs
                rs(stream=stream)
                ar(stream=stream)
                torch.cuda.synchronize()
                want = oracle.reduce_points(xs_at, idx, n, M, dtype, "sum", "ring")
                chk = Check("sampled")
                check_rs_sampled(chk, torch, z, idx, want, n, M, q, dtype, "sum")
                check_full_sampled(chk, torch, "AR", d, idx, want, dtype)
                ag(stream=stream)
                torch.cuda.synchronize()
                check_full_sampled(chk, torch, "AG", d, idx, want, dtype)
                t = timer.alternating([("rs", lambda: rs(stream=stream)),
                                       ("ag", lambda: ag(stream=stream)),
                                       ("ar", lambda: ar(stream=stream))])
                b = step_bytes(n, M, es)
                row = {"n": n, "bytes_per_rank": nbytes, "dtype": dtype}
                for key, bk in (("rs", "reduce_scatter"), ("ag", "all_gather"), ("ar", "fused_ar")):
                    st = call_stats(t[key], b[bk], peak)
                    row[key] = {k: st[k] for k in ("median_us", "mean_us", "p95_us", "cv", "frac")}
                row["oracle"] = {"indices": int(idx.size), "mismatches": chk.mismatches}
                rows.append(row)
                del d, z, rs, ar, ag
                torch.cuda.empty_cache()
    # every op and order at one point: eight ranks, 64 MiB per rank, the
    # float types (the integer types give the same bits in every order)
    combos = []
    n, nbytes = 8, 64 << 20
    for dtype in ("float32", "bfloat16"):
        M = nbytes // ESIZE[dtype]
        d = si.generate_device(torch, dtype, "uniform_pm1", n, M, si.SEED_BASE + 6, dev)
        q = vc.vc_shard_count(M, n)
        z = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
        y = [torch.empty_like(t) for t in d]
        idx = sample_indices(M, n, q, k=1 << 12, seed=8)
        xs_at = sampled_operands(torch, d, idx, dtype)
        b = step_bytes(n, M, ESIZE[dtype])
        for order in ("ring", "recursive_halving", "pairwise_tree", "double_binary_tree"):
            for op in ("sum", "max", "min", "prod"):
                rs = vc.prepare_reduce_scatter(d, z, op=op, order=order)
                ar = vc.prepare_all_reduce(d, y, op=op, order=order)
                rs(stream=stream)
                ar(stream=stream)
                torch.cuda.synchronize()
                want = oracle.reduce_points(xs_at, idx, n, M, dtype, op, order)
                chk = Check("sampled")
                check_rs_sampled(chk, torch, z, idx, want, n, M, q, dtype, op)
                check_full_sampled(chk, torch, "AR", y, idx, want, dtype)
                t = timer.alternating([("rs", lambda: rs(stream=stream)),
                                       ("ar", lambda: ar(stream=stream))])
                row = {"dtype": dtype, "order": order, "op": op}
                for key, bk in (("rs", "reduce_scatter"), ("ar", "fused_ar")):
                    st = call_stats(t[key], b[bk], peak)
                    row[key] = {k: st[k] for k in ("median_us", "mean_us", "cv", "frac")}
                row["oracle"] = {"indices": int(idx.size), "mismatches": chk.mismatches}
                combos.append(row)
        del d, z, y, rs, ar
        torch.cuda.empty_cache()
    fr = [r[k]["frac"] for r in rows for k in ("rs", "ar")]
    fo = [r[k]["frac"] for r in combos for k in ("rs", "ar")]
    return {"config": "per-rank 64 MiB and 1 GiB x N in {2,4,8,16,64} (N*bytes <= 64 GiB) x "
                      "int32/int64/fp32/bf16; SUM, ring; RS, AG, fused AR (in place); and at "
                      "8 ranks x 64 MiB, fp32/bf16, every op x order, RS and AR",
            "points": rows,
            "min_frac_rs_ar": round(min(fr), 4),
            "ops_orders_n8_64mib": combos,
            "ops_orders_min_frac_rs_ar": round(min(fo), 4),
            "oracle_mismatches": sum(r["oracle"]["mismatches"] for r in rows + combos)}


def configs_report(torch, vc, args, dev, stream, peak, d, memory):
    """Every configuration the workload list names, each with per-call
    median / P95 / CV (alternating path order), algorithmic bytes, GB/s, the
    fraction of the copy peak and its oracle check.  The full-size fp32 four-
    rank entry reuses the headline's input buffers."""
    out = {}
    jobs = (("C1_worked_example_n4_m20_int64", lambda: config_c1(torch, vc, dev, stream, peak)),
            ("C2_n8_m1000003_f32_uniform", lambda: config_c2(torch, vc, dev, stream, peak)),
            ("C3_n8_bucket25mib_bf16_normal", lambda: config_c3(torch, vc, dev, stream, peak)),
            ("C4_n4_256mib_f32_normal",
             lambda: config_c4(torch, vc, dev, stream, peak, "n4_256mib_f32_normal", args, d,
                               memory)),
            ("C4_n4_m67108864_i64_uniform",
             lambda: config_c4(torch, vc, dev, stream, peak, "n4_m67108864_i64_uniform", args)),
            ("C5_sweep_summary", lambda: config_c5(torch, vc, dev, stream, peak)))
    for name, fn in jobs:
        t0 = time.perf_counter()
        try:
            out[name] = fn()
        except Exception as e:  # recorded in the line, never hidden
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
        out[name]["wall_s"] = round(time.perf_counter() - t0, 1)
        torch.cuda.empty_cache()
    return out


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
    the device; each kernel's time is the mean of 10 single calls after 3
    warm-ups, the fastest and the slowest left out (call_stats: the event
    clock's 2.048 us steps).  Before each call a read of twice the L2 evicts the last
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

    def t_ms(fn, reps=10):
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
        return call_stats(times, 1, 1.0)["mean_us"] / 1e3

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
                    "timing": "mean of 10 single calls less the fastest and slowest, "
                              "each after an L2-evicting read"}
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


def run_one(args):
    """One collective on one synthetic workload, timed back to back: the
    case a single-kernel profile captures.  --one PATH:DTYPE:N:ELEMENTS,
    PATH in {rs, ag, ar, dec}; inputs uniform[-1, 1) (floats) or uniform
    [-100, 100] (integers), seeded; --op / --order as given; W warm-up calls,
    then K calls between two events.  Prints one JSON line."""
    import torch

    import allreduce_reducescatter_allgather_gb300 as vc
    import synthetic_inputs as si
    path, dtype, n, M = args.one.split(":")
    n, M = int(n), int(M)
    if path not in ("rs", "ag", "ar", "dec") or dtype not in ESIZE:
        raise SystemExit(f"--one {args.one}: PATH in rs/ag/ar/dec, DTYPE in {sorted(ESIZE)}")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    dist = "uniform_pm1" if dtype in ("float32", "bfloat16") else "uniform_int"
    kw = {} if dist == "uniform_pm1" else {"lo": -100, "hi": 100}
    d = si.generate_device(torch, dtype, dist, n, M, si.SEED_BASE + 5, dev, **kw)
    q = vc.vc_shard_count(M, n)
    z = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
    y = [torch.empty_like(t) for t in d]
    call = {"rs": lambda: vc.prepare_reduce_scatter(d, z, op=args.op, order=args.order),
            "ag": lambda: vc.prepare_all_gather(z, y),
            "ar": lambda: vc.prepare_all_reduce(d, y, op=args.op, order=args.order),
            "dec": lambda: vc.prepare_all_reduce_decomposed(d, z, y, op=args.op,
                                                            order=args.order)}[path]()
    for _ in range(args.warmup):
        call(stream=stream)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        call(stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    key = {"rs": "reduce_scatter", "ag": "all_gather", "ar": "fused_ar",
           "dec": "decomposed_ar"}[path]
    nbytes = step_bytes(n, M, ESIZE[dtype])[key]
    peak, kind = measured_peak()
    g = nbytes / (ms / 1e3) / 1e9
    print(json.dumps({"one": args.one, "op": args.op, "order": args.order, "q": q,
                      "shard_offset_bytes": (q * ESIZE[dtype]) % 16, "calls": args.steps,
                      "us_per_call": round(ms * 1e3, 2), "bytes": nbytes, "gbs": round(g, 1),
                      "frac": round(g / peak, 4), "peak_kind": kind}), flush=True)
    return 0


def run_bucket_path(args):
    """One gradient-bucket collective over the transformer-shaped set of
    bucket_report (145 bf16 tensors, 351 MiB per rank, 8 ranks), W warm-up
    calls then K timed, one launch per bucket each: the case a single-kernel
    profile of the bucket kernels captures.  --bucket-path PATH, PATH in
    ar_fused, ar_views, rs_fused, rs_views, ag_fused.  Prints one JSON line."""
    import torch

    import allreduce_reducescatter_allgather_gb300 as vc  # noqa: F401 (loads the library)
    from allreduce_reducescatter_allgather_gb300 import bucketing
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n = 8
    shapes = transformer_grad_shapes()
    gb = bucketing.GradientBuckets(shapes, torch.bfloat16, n, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(99)
    grads = [[torch.randn(s, generator=g, device=dev).to(torch.bfloat16) for s in shapes]
             for _ in range(n)]
    gb.bind(grads)
    gb.reduce_scatter(op=args.op, order=args.order)  # the shards the AllGather reads
    fn = {"ar_fused": lambda: gb.all_reduce_tensors(op=args.op, order=args.order, fused=True),
          "ar_views": lambda: gb.all_reduce(op=args.op, order=args.order),
          "rs_fused": lambda: gb.reduce_scatter_tensors(op=args.op, order=args.order, fused=True),
          "rs_views": lambda: gb.reduce_scatter(op=args.op, order=args.order),
          "ag_fused": lambda: gb.all_gather_tensors()}[args.bucket_path]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    print(json.dumps({"bucket_path": args.bucket_path, "buckets": len(gb.buckets),
                      "bucket_counts": [bk.count for bk in gb.buckets], "calls": args.steps,
                      "us_per_call": round(a.elapsed_time(b) / args.steps * 1e3, 1)}), flush=True)
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
                    choices=["ring", "recursive_halving", "pairwise_tree",
                             "double_binary_tree"])
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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration report (every workload, oracle-checked)")
    ap.add_argument("--one", default="",
                    help="time one collective instead: PATH:DTYPE:N:ELEMENTS, e.g. "
                         "rs:bfloat16:12:8388608 (PATH in rs, ag, ar, dec)")
    ap.add_argument("--bucket-path", default="",
                    choices=["", "ar_fused", "ar_views", "rs_fused", "rs_views", "ag_fused"],
                    help="time one gradient-bucket collective over the 145-tensor set instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    workload = dict(si.WORKLOADS[args.workload])
    if args.elements > 0:
        workload["M"] = args.elements
    if args.impl == "reference":
        return run_reference(args, workload)
    if args.sweep or args.one or args.bucket_path:
        import __graft_entry__
        __graft_entry__.build()
        if args.bucket_path:
            return run_bucket_path(args)
        return run_sweep(args) if args.sweep else run_one(args)
    if dist_info()[0] == 1:
        import __graft_entry__
        __graft_entry__.build()  # under torchrun the library must be built beforehand
    return run_ours(args, workload)


if __name__ == "__main__":
    sys.exit(main())
