"""Gradient buckets: DDP's assignment rule with the pages' caps (CPU), and the
bucketed AllReduce on the GPU against the oracle run on the same bucket
layout."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from conftest import ints, read_golden
from gpu_util import assert_bits_equal, to_host

MiB = 1 << 20


def test_assignment_matches_hand_derivation():
    from allreduce_reducescatter_allgather_gb300.bucketing import (
        BUCKET_BYTES, FIRST_BUCKET_BYTES, assign_buckets)
    assert FIRST_BUCKET_BYTES == 1 * MiB and BUCKET_BYTES == 25 * MiB
    g = read_golden("ddp_buckets.txt")
    sizes = [int(float(s) * MiB) for s in g["sizes_mib"].split()]
    got = assign_buckets(sizes)
    want = [ints(g[f"bucket{k}"]) for k in range(4)]
    assert got == want


def test_assignment_invariants():
    from allreduce_reducescatter_allgather_gb300.bucketing import assign_buckets
    rng = np.random.default_rng(0)
    sizes = [int(x) for x in rng.integers(1, 8 * MiB, 300)]
    buckets = assign_buckets(sizes)
    flat = [t for b in buckets for t in b]
    assert flat == list(reversed(range(len(sizes))))  # every tensor once, backward order
    for k, b in enumerate(buckets):
        cap = 1 * MiB if k == 0 else 25 * MiB
        total = sum(sizes[t] for t in b)
        assert total <= cap or len(b) == 1
        if k + 1 < len(buckets):  # closed because the next tensor did not fit
            assert total + sizes[buckets[k + 1][0]] > cap


# ------------------------------------------------------------------ GPU --

SHAPES = [(3,), (17, 5), (1000,), (256, 256), (4099,), (64, 1024), (7, 7, 7), (300_001,),
          (2,), (1 << 20,), (12345,), (513, 9), (1,)]


@pytest.fixture(scope="module")
def genv():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import allreduce_reducescatter_allgather_gb300 as vc
    from allreduce_reducescatter_allgather_gb300 import bucketing
    dev = torch.device("cuda:0")
    return torch, vc, bucketing, dev


def _oracle_buckets(gb, grads_np, dtype, op, order):
    """The oracle's AllReduce of every bucket, laid out as the library lays
    it out (zero padding included), sliced back into tensors."""
    out = [[None] * len(gb.shapes) for _ in range(gb.nranks)]
    st = oracle.NP_STORAGE[dtype]
    for b in gb.buckets:
        bufs = [np.zeros(b.count, st) for _ in range(gb.nranks)]
        for r in range(gb.nranks):
            for t, off in zip(b.tensors, b.offsets):
                bufs[r][off:off + gb.numels[t]] = grads_np[r][t]
        ys = oracle.all_reduce(bufs, dtype, op, order)
        for r in range(gb.nranks):
            for t, off in zip(b.tensors, b.offsets):
                out[r][t] = ys[r][off:off + gb.numels[t]]
    return out


def _oracle_bucket_shards(gb, grads_np, dtype, op, order):
    """The oracle's ReduceScatter of every bucket as the library lays it out
    (zero padding between tensors): shards[bucket][rank]."""
    st = oracle.NP_STORAGE[dtype]
    out = []
    for b in gb.buckets:
        bufs = [np.zeros(b.count, st) for _ in range(gb.nranks)]
        for r in range(gb.nranks):
            for t, off in zip(b.tensors, b.offsets):
                bufs[r][off:off + gb.numels[t]] = grads_np[r][t]
        out.append(oracle.reduce_scatter(bufs, dtype, op, order))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,op,order", [("float32", "sum", "ring"),
                                            ("bfloat16", "avg", "recursive_halving"),
                                            ("int64", "max", "double_binary_tree")])
def test_bucket_views_and_packing_match_oracle(genv, dtype, op, order):
    torch, vc, bk, dev = genv
    n = 8
    tdt = {"float32": torch.float32, "bfloat16": torch.bfloat16, "int64": torch.int64}[dtype]
    dist = "uniform_int" if dtype == "int64" else "uniform_pm1"
    kw = {"lo": -100, "hi": 100} if dtype == "int64" else {}
    # small caps so that this set spans several buckets
    gb = bk.GradientBuckets(SHAPES, tdt, n, dev, first_cap=64 << 10, cap=2 * MiB)
    assert len(gb.buckets) >= 3
    grads_np = [[si.generate_rank(dtype, dist, 11 + t, r, gb.numels[t], **kw)
                 for t in range(len(SHAPES))] for r in range(n)]
    want = _oracle_buckets(gb, grads_np, dtype, op, order)

    def to_dev(a):
        if dtype == "bfloat16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    # views: write the gradients into the bucket views, reduce in place
    for r in range(n):
        for t, v in enumerate(gb.views(r)):
            v.copy_(to_dev(grads_np[r][t]).view(v.shape))
    gb.all_reduce(op=op, order=order)
    torch.cuda.synchronize()
    for r in range(n):
        for t, v in enumerate(gb.views(r)):
            assert_bits_equal(to_host(v.reshape(-1), dtype), want[r][t], dtype, f"view r{r} t{t}")
    # the buckets' ReduceScatter (ZeRO): from the views' buffers, and from
    # separately allocated tensors (packed, or fused where the order allows)
    want_rs = _oracle_bucket_shards(gb, grads_np, dtype, op, order)
    for r in range(n):  # the AllReduce above overwrote the views
        for t, v in enumerate(gb.views(r)):
            v.copy_(to_dev(grads_np[r][t]).view(v.shape))
    got = gb.reduce_scatter(op=op, order=order)
    torch.cuda.synchronize()
    for i, sh in enumerate(got):
        for r in range(n):
            assert_bits_equal(to_host(sh[r], dtype), want_rs[i][r], dtype, f"RS views b{i} r{r}")
    for fused in (False, True):
        grads = [[to_dev(grads_np[r][t]).view(SHAPES[t]).clone() for t in range(len(SHAPES))]
                 for r in range(n)]
        for b in gb.buckets:
            for buf in b.buffers:
                buf.zero_()
        gb.bind(grads)
        for sh in got:
            for t in sh:
                t.fill_(3)
        got = gb.reduce_scatter_tensors(op=op, order=order, fused=fused)
        torch.cuda.synchronize()
        for i, sh in enumerate(got):
            for r in range(n):
                assert_bits_equal(to_host(sh[r], dtype), want_rs[i][r], dtype,
                                  f"RS fused={fused} b{i} r{r}")
        # gathering the shards back into the tensors completes the
        # decomposed AllReduce of the buckets
        gb.all_gather_tensors()
        torch.cuda.synchronize()
        for r in range(n):
            for t in range(len(SHAPES)):
                assert_bits_equal(to_host(grads[r][t].reshape(-1), dtype), want[r][t], dtype,
                                  f"RS+AG fused={fused} r{r} t{t}")
    # separately allocated tensors: packed, reduced, unpacked; and fused
    # (one launch per bucket) where the order allows it
    for fused in (False, True):
        for b in gb.buckets:
            for buf in b.buffers:
                buf.zero_()
        grads = [[to_dev(grads_np[r][t]).view(SHAPES[t]).clone() for t in range(len(SHAPES))]
                 for r in range(n)]
        gb.bind(grads)
        gb.all_reduce_tensors(op=op, order=order, fused=fused)
        torch.cuda.synchronize()
        for r in range(n):
            for t in range(len(SHAPES)):
                assert_bits_equal(to_host(grads[r][t].reshape(-1), dtype), want[r][t], dtype,
                                  f"fused={fused} r{r} t{t}")


@pytest.mark.gpu
def test_bucketed_equals_per_tensor_for_chunk_free_orders(genv):
    """Recursive halving and the tree fold every element the same way
    wherever it sits, so bucketed and per-tensor AllReduce agree bit for bit
    (the ring's rotation depends on the element's chunk, so it does not)."""
    torch, vc, bk, dev = genv
    n = 4
    gb = bk.GradientBuckets(SHAPES, torch.float32, n, dev)
    src = [[torch.randn(s, device=dev) for s in SHAPES] for _ in range(n)]
    grads = [[g.clone() for g in row] for row in src]
    gb.bind(grads)
    for order in ("recursive_halving", "pairwise_tree"):
        for r in range(n):
            for t in range(len(SHAPES)):
                grads[r][t].copy_(src[r][t])
        gb.all_reduce_tensors(order=order)
        for t in range(len(SHAPES)):
            # the oracle's AllReduce of the tensor on its own, wherever the
            # bucket put it, and the library's per-tensor call
            xs = [to_host(src[r][t].reshape(-1), "float32") for r in range(n)]
            want = oracle.all_reduce(xs, "float32", "sum", order)
            ref = [torch.empty_like(src[0][t]) for _ in range(n)]
            vc.vc_all_reduce([src[r][t] for r in range(n)], ref, order=order)
            for r in range(n):
                assert_bits_equal(to_host(grads[r][t].reshape(-1), "float32"), want[r],
                                  "float32", f"bucketed {order} tensor {t} rank {r}")
                assert torch.equal(grads[r][t], ref[r])


FUSED_SHAPES = [(5,), (16_381,), (0,), (3, 7), (70_001,), (1,), (4096,), (33_333,)]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,op", [("float32", "sum"), ("bfloat16", "avg"),
                                      ("int32", "prod"), ("int64", "min")])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 12, 64])
def test_fused_bucket_matches_oracle(genv, dtype, op, n):
    """vc_all_reduce_bucket against the oracle's ring AllReduce of the packed
    bucket (each tensor at the previous one's end rounded up to 16 bytes,
    zeros between), out of place, with every other tensor a view whose base
    is one element off the 16-byte grid (the element-by-element path); N =
    2, 4, 8 take the compile-time kernels, the others the run-time one.
    Then vc_reduce_scatter_bucket against the oracle's ReduceScatter."""
    torch, vc, bk, dev = genv
    tdt = {"float32": torch.float32, "bfloat16": torch.bfloat16, "int32": torch.int32,
           "int64": torch.int64}[dtype]
    es = torch.empty(0, dtype=tdt).element_size()
    dist = "uniform_pm1" if dtype in ("float32", "bfloat16") else "uniform_int"
    kw = {} if dist == "uniform_pm1" else {"lo": -3, "hi": 3}
    counts = [int(np.prod(s)) for s in FUSED_SHAPES]
    host = [[si.generate_rank(dtype, dist, 50 + k, r, counts[k], **kw) for k in range(len(counts))]
            for r in range(n)]

    def to_dev(a, shift):
        t = torch.from_numpy(a.view(np.int16) if dtype == "bfloat16" else a)
        t = t.view(tdt) if dtype == "bfloat16" else t
        big = torch.empty(a.size + shift, dtype=tdt, device=dev)
        big[shift:].copy_(t.to(dev))
        return big[shift:]

    ins = [[to_dev(host[r][k], k % 2) for k in range(len(counts))] for r in range(n)]
    outs = [[to_dev(np.zeros_like(host[r][k]), (k + 1) % 2) for k in range(len(counts))]
            for r in range(n)]
    plan = vc.BucketPlan(ins, outs)
    plan(op=op)
    torch.cuda.synchronize()
    # the oracle: the packed bucket, its ring AllReduce, sliced back
    align, off, base = 16 // es, 0, []
    for c in counts:
        base.append(off)
        off = -(-(off + c) // align) * align
    assert plan.bucket_count == off
    st = oracle.NP_STORAGE[dtype]
    bufs = [np.zeros(off, st) for _ in range(n)]
    for r in range(n):
        for k, c in enumerate(counts):
            bufs[r][base[k]:base[k] + c] = host[r][k]
    ys = oracle.all_reduce(bufs, dtype, op, "ring")
    for r in range(n):
        for k, c in enumerate(counts):
            assert_bits_equal(to_host(outs[r][k], dtype), ys[r][base[k]:base[k] + c], dtype,
                              f"N={n} rank {r} tensor {k}")
            # inputs untouched (out of place)
            assert_bits_equal(to_host(ins[r][k], dtype), host[r][k], dtype, "input kept")
    # the bucket's ReduceScatter: every shard element, gaps and padding
    # included, against the oracle's ReduceScatter of the packed bucket
    q = plan.shard_count
    shards = [torch.full((q,), 7, dtype=tdt, device=dev) for _ in range(n)]
    plan.reduce_scatter(shards, op=op)
    torch.cuda.synchronize()
    zs = oracle.reduce_scatter(bufs, dtype, op, "ring")
    for r in range(n):
        assert_bits_equal(to_host(shards[r], dtype), zs[r], dtype, f"N={n} shard {r}")
    # the bucket's AllGather: those shards back into the output tensors is
    # the AllReduce again; arbitrary shards give the oracle's AllGather
    for t in (x for row in outs for x in row):
        t.fill_(5)
    plan.all_gather(shards)
    torch.cuda.synchronize()
    for r in range(n):
        for k, c in enumerate(counts):
            assert_bits_equal(to_host(outs[r][k], dtype), ys[r][base[k]:base[k] + c], dtype,
                              f"AG(RS) N={n} rank {r} tensor {k}")
    rnd = [si.generate_rank(dtype, dist, 90, r, q, **kw) for r in range(n)]
    dsh = [to_dev(a, 0) for a in rnd]
    plan.all_gather(dsh)
    torch.cuda.synchronize()
    gs = oracle.all_gather(rnd, off, dtype)
    for r in range(n):
        for k, c in enumerate(counts):
            assert_bits_equal(to_host(outs[r][k], dtype), gs[r][base[k]:base[k] + c], dtype,
                              f"AG N={n} rank {r} tensor {k}")


@pytest.mark.gpu
def test_fused_bucket_in_place_equals_bucket_views(genv):
    """In place on the transformer-shaped gradient set: the fused call gives
    the bits of the bucket views path, bucket by bucket."""
    torch, vc, bk, dev = genv
    n = 8
    shapes = [(1024, 1024), (1024,), (4096, 1024), (1024, 4096), (32000, 1024), (1000, 3)]
    gb = bk.GradientBuckets(shapes, torch.bfloat16, n, dev)
    src = [[torch.randn(s, device=dev).to(torch.bfloat16) for s in shapes] for _ in range(n)]
    for r in range(n):
        for t, v in enumerate(gb.views(r)):
            v.copy_(src[r][t])
    grads = [[g.clone() for g in row] for row in src]
    gb.bind(grads)
    gb.all_reduce(op="sum", order="ring")
    gb.all_reduce_tensors(op="sum", order="ring", fused=True)
    torch.cuda.synchronize()
    host = [[to_host(g.reshape(-1), "bfloat16") for g in row] for row in src]
    want = _oracle_buckets(gb, host, "bfloat16", "sum", "ring")
    for r in range(n):
        for t, v in enumerate(gb.views(r)):
            assert torch.equal(grads[r][t], v)
            assert_bits_equal(to_host(grads[r][t].reshape(-1), "bfloat16"), want[r][t],
                              "bfloat16", f"fused in place tensor {t} rank {r}")


@pytest.mark.gpu
def test_fused_buckets_replay_from_a_cuda_graph(genv):
    """The fused bucket calls only enqueue work on the current stream, so a
    training step can capture them in a CUDA graph once and replay it on new
    gradients written into the same tensors: every replay gives the bits of
    the bucket views path on those gradients."""
    torch, vc, bk, dev = genv
    n = 4
    shapes = [(1000, 3), (4096,), (333, 77), (7,)]
    gb = bk.GradientBuckets(shapes, torch.float32, n, dev, first_cap=64 << 10, cap=1 << 20)
    grads = [[torch.empty(s, device=dev) for s in shapes] for _ in range(n)]
    gb.bind(grads)
    gb.all_reduce_tensors(fused=True)  # first call outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gb.all_reduce_tensors(fused=True)
    for it in range(3):
        src = [[torch.randn(s, device=dev) for s in shapes] for _ in range(n)]
        for r in range(n):
            for t in range(len(shapes)):
                grads[r][t].copy_(src[r][t])
                gb.views(r)[t].copy_(src[r][t])
        g.replay()
        gb.all_reduce(op="sum", order="ring")
        torch.cuda.synchronize()
        host = [[to_host(x.reshape(-1), "float32") for x in row] for row in src]
        want = _oracle_buckets(gb, host, "float32", "sum", "ring")
        for r in range(n):
            for t, v in enumerate(gb.views(r)):
                assert torch.equal(grads[r][t], v), (it, r, t)
                assert_bits_equal(to_host(grads[r][t].reshape(-1), "float32"), want[r][t],
                                  "float32", f"replay {it} tensor {t} rank {r}")
