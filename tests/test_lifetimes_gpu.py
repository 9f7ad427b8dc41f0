"""Buffer lifetimes of the decomposed AllReduce and the ZeRO-style RS-only
flow ("NCCL 专家课程 07", 显存实验: RS-only keeps 64 of 256 MiB; the naive RS+AG
lifetime peaks at 576 MiB, releasing the input first brings it to 320 MiB).
Here the release is stream-ordered (no synchronize) and the results must be
the fused AllReduce's bits."""
from __future__ import annotations

import pytest

import synthetic_inputs as si

pytestmark = pytest.mark.gpu
MiB = 1 << 20


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import allreduce_reducescatter_allgather_gb300 as vc
    from allreduce_reducescatter_allgather_gb300 import lifetimes
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    return torch, vc, lifetimes, dev


@pytest.mark.parametrize("dtype,order", [("float32", "ring"), ("float32", "pairwise_tree"),
                                         ("bfloat16", "recursive_halving"), ("int64", "ring")])
def test_low_peak_decomposed_matches_fused(env, dtype, order):
    torch, vc, lt, dev = env
    n, M = 8, 1_000_003
    dist = "uniform_pm1" if dtype != "int64" else "uniform_int"
    kw = {} if dtype != "int64" else {"lo": -100, "hi": 100}
    base = si.generate_device(torch, dtype, dist, n, M, seed=3, device=dev, **kw)
    ref = [torch.empty_like(t) for t in base]
    vc.vc_all_reduce(base, ref, order=order)
    inputs = [t.clone() for t in base]
    outs = lt.all_reduce_decomposed_low_peak(inputs, order=order)
    torch.cuda.synchronize()
    assert inputs == []  # ownership taken
    for r in range(n):
        assert torch.equal(outs[r], ref[r])


def _peak(torch, dev, fn):
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    kept = fn()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(dev) - base
    steady = torch.cuda.memory_allocated(dev) - base
    del kept
    return peak, steady


def test_peak_and_steady_memory(env):
    """4 ranks x 64 MiB fp32 (the page's 256 MiB tensor, split over four
    virtual ranks): RS-only steady = shards, stream-ordered RS+AG peak =
    inputs + shards, naive RS+AG peak = inputs + shards + outputs."""
    torch, vc, lt, dev = env
    n, M = 4, (64 * MiB) // 4
    src = si.generate_device(torch, "float32", "normal", n, M, seed=1, device=dev)
    inputs_b, shard_b = n * M * 4, M * 4  # 256 MiB of inputs, 64 MiB of shards

    def rs_only():
        return lt.reduce_scatter_keep_shards([t.clone() for t in src])

    def low_peak():
        return lt.all_reduce_decomposed_low_peak([t.clone() for t in src])

    def naive():
        full = [t.clone() for t in src]
        q = vc.vc_shard_count(M, n)
        sh = [torch.empty(q, device=dev) for _ in range(n)]
        out = [torch.empty_like(t) for t in full]
        vc.vc_reduce_scatter(full, sh)
        vc.vc_all_gather(sh, out)
        return out

    peak, steady = _peak(torch, dev, rs_only)
    assert steady == shard_b
    assert peak == inputs_b + shard_b
    peak, steady = _peak(torch, dev, low_peak)
    assert steady == inputs_b
    assert peak == inputs_b + shard_b
    peak, _ = _peak(torch, dev, naive)
    assert peak == 2 * inputs_b + shard_b


def test_inputs_from_another_stream(env):
    """Inputs written on a side stream: the caller orders its stream after
    the producer; the helper records the inputs on the stream that reads
    them, so their memory is not handed out before the ReduceScatter ran."""
    torch, vc, lt, dev = env
    n, M = 4, 1 << 22
    src = si.generate_device(torch, "float32", "uniform_pm1", n, M, seed=2, device=dev)
    ref = [torch.empty_like(t) for t in src]
    vc.vc_all_reduce(src, ref)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        inputs = [t * 1.0 for t in src]
    torch.cuda.current_stream(dev).wait_stream(side)
    outs = lt.all_reduce_decomposed_low_peak(inputs)
    # allocations on the side stream after the release must not clobber
    # anything still in flight
    with torch.cuda.stream(side):
        junk = [torch.full((M,), 7.0, device=dev) for _ in range(n)]
    torch.cuda.synchronize()
    for r in range(n):
        assert torch.equal(outs[r], ref[r])
    del junk
