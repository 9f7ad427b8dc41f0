"""Host-side logic of bench.py on CPU: the byte accounting of a step, the
recorded-traffic lookup and the L2 note, and the max-over-ranks /
sum-over-ranks aggregation, the latter with two gloo ranks."""
from __future__ import annotations

import os
import socket

import pytest

import bench


def test_step_bytes():
    n, M, s = 4, 67_108_864, 4
    b = bench.step_bytes(n, M, s)
    assert b["reduce_scatter"] == n * M * s + M * s
    assert b["all_gather"] == M * s + n * M * s
    assert b["fused_ar"] == 2 * n * M * s
    assert b["step"] == 4 * n * M * s + 2 * M * s


def test_recorded_traffic_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu record only while the
    measured kernels' code still hashes to the digest recorded with it."""
    rec = bench.ROOT / "profiles" / "dram_traffic.txt"
    text = rec.read_text()
    got = bench.recorded_traffic("vc_ar_kernel", "n4_256mib_f32_normal")
    if f"source_sha: {bench.source_digest()}" in text:
        assert got is not None and got > 0
    else:
        assert got is None
    # the same record under a given digest: used while the sources hash to
    # it, ignored otherwise (whatever digest the committed record carries)
    import re
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    (fake / "profiles" / "dram_traffic.txt").write_text(
        re.sub(r"(?m)^source_sha: \S+$", "source_sha: 0000000000000000", text))
    monkeypatch.setattr(bench, "ROOT", fake)
    monkeypatch.setattr(bench, "source_digest", lambda: "0000000000000000")
    assert bench.recorded_traffic("vc_ar_kernel", "n4_256mib_f32_normal") > 0
    assert bench.recorded_traffic("vc_ar_kernel", "another_workload") is None
    monkeypatch.setattr(bench, "source_digest", lambda: "ffffffffffffffff")
    assert bench.recorded_traffic("vc_ar_kernel", "n4_256mib_f32_normal") is None


def test_l2_note_names_small_cases():
    """A step whose inputs fit twice in the 129 MB L2 is called out as a
    small case; the full-size workload is not."""
    assert "far larger" in bench.l2_note(4 * 256 << 20)
    assert "small case" in bench.l2_note(4 * 8 << 20)


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, total = bench.aggregate(torch, 10.0 + 5 * rank, 1000 * (rank + 1), world)
        q.put((rank, ms, total))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, total in got:
        assert ms == 15.0          # the slower rank's time
        assert total == 3000       # every rank's bytes


def _worker_lost_peer(rank, world, port, q):
    import datetime
    import time

    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(0)  # leaves between steps, without joining the collective
    t0 = time.monotonic()
    try:
        bench.aggregate(torch, 10.0, 1000, world)
        q.put(("returned", time.monotonic() - t0))
    except Exception as e:  # noqa: BLE001 - any error is the expected outcome
        q.put(("raised", time.monotonic() - t0, type(e).__name__))


def test_lost_rank_ends_the_collective_with_an_error():
    """A rank that leaves between steps: the other rank's next collective
    fails within the process-group timeout instead of waiting forever."""
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_worker_lost_peer, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = q.get(timeout=120)
    for p in procs:
        p.join(60)
        if p.is_alive():
            p.kill()
    assert out[0] == "raised", out
    assert out[1] < 60, out


def test_call_stats_marks_unstable_figures():
    """Median / P95 / CV of per-call times and the median's rate; a ratio is
    claimable only from figures with CV <= 5 %."""
    st = bench.call_stats([1.0, 1.0, 1.0, 1.0], 2_000_000, 1000.0)
    assert st["median_us"] == 1000.0 and st["cv"] == 0.0 and st["stable"]
    assert st["gbs"] == 2.0 and st["frac"] == 0.002
    st = bench.call_stats([1.0, 2.0, 1.0, 2.0], 1, 1.0)
    assert not st["stable"] and st["cv"] > 0.05
    assert st["p95_us"] == 2000.0


def test_sample_indices_cover_every_chunk_boundary():
    import numpy as np
    M, n = 1_000_003, 8
    q = -(-M // n)
    idx = bench.sample_indices(M, n, q, k=100, seed=3)
    assert np.all(np.diff(idx) > 0) and idx[0] == 0 and idx[-1] == M - 1
    for c in range(1, n):
        assert c * q - 1 in idx and c * q in idx


def test_check_counts_mismatches_bitwise():
    """The comparator works on bits: -0.0 differs from +0.0, NaN equals
    itself when the payload is the same."""
    import numpy as np
    chk = bench.Check("full")
    a = np.array([1.0, 0.0, np.nan], np.float32)
    chk.eq("x", a, a.copy())
    assert chk.mismatches == 0
    chk.eq("x", np.array([1.0, -0.0, np.nan], np.float32), a)
    assert chk.mismatches == 1 and chk.compared == 6
    s = chk.summary(indices=3)
    assert not s["bit_exact"] and s["indices"] == 3 and s["outputs"] == ["x"]


def test_call_stats_rate_survives_a_coarse_event_clock():
    """A 29.5 us call read by an event clock that advances in 2.048 us
    steps: four readings of ten land on 30.72 us, six on 28.672 us.  The
    median sits on the grid; the rate comes from the mean of the middle
    eight, which stays within the step's tenth of the true time, and one
    slow outlier does not move it."""
    ms = [0.028672] * 6 + [0.03072] * 4
    st = bench.call_stats(ms, 1_000_000, 1.0)
    assert st["median_us"] == 28.67
    assert abs(st["mean_us"] - 29.5) < 0.2
    assert abs(st["gbs"] - 1e6 / 29.44e-6 / 1e9) < 0.1
    slow = ms[:-1] + [0.060]
    assert bench.call_stats(slow, 1_000_000, 1.0)["mean_us"] == st["mean_us"]
