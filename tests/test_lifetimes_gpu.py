"""Buffer lifetimes of the decomposed AllReduce and the ZeRO-style RS-only
flow ("NCCL 专家课程 07", 显存实验必须区分 steady 与 peak: RS-only keeps 64 of
256 MiB; the naive RS+AG lifetime peaks at 576 MiB, releasing the input first
brings it to 320 MiB; and ZeRO/FSDP 为什么停在 ReduceScatter).  Here the release
is stream-ordered (no synchronize).  The shards and outputs of every flow are
compared bit for bit with the CPU oracle on the same host inputs: the oracle's
ReduceScatter for the kept shards, its AllReduce for the gathered outputs
(same order, so the bits must agree)."""
from __future__ import annotations

import pytest

import oracle
import synthetic_inputs as si
from gpu_util import assert_bits_equal, to_device, to_host

pytestmark = pytest.mark.gpu
MiB = 1 << 20

CASES = [("float32", "ring", "sum"), ("float32", "pairwise_tree", "sum"),
         ("bfloat16", "recursive_halving", "avg"), ("int64", "ring", "prod"),
         ("float32", "double_binary_tree", "max")]


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


def _host_inputs(dtype, n, M, seed):
    if dtype == "int64":
        return si.generate(dtype, "uniform_int", n, M, seed=seed, lo=-100, hi=100)
    return si.generate(dtype, "uniform_pm1", n, M, seed=seed)


@pytest.mark.parametrize("dtype,order,op", CASES)
def test_low_peak_decomposed_matches_oracle(env, dtype, order, op):
    torch, vc, lt, dev = env
    n, M = 8, 1_000_003
    xs = _host_inputs(dtype, n, M, seed=3)
    want = oracle.all_reduce(xs, dtype, op, order)
    inputs = to_device(torch, xs, dtype, dev)
    outs = lt.all_reduce_decomposed_low_peak(inputs, op=op, order=order)
    torch.cuda.synchronize()
    assert inputs == []  # ownership taken
    for r in range(n):
        assert_bits_equal(to_host(outs[r], dtype), want[r], dtype, f"low-peak AR rank {r}")


@pytest.mark.parametrize("dtype,order,op", CASES)
def test_reduce_scatter_keep_shards_matches_oracle(env, dtype, order, op):
    """The ZeRO step: only the shards survive, and each is the oracle's
    ReduceScatter shard (padding tail included)."""
    torch, vc, lt, dev = env
    n, M = 8, 1_000_003
    xs = _host_inputs(dtype, n, M, seed=4)
    want = oracle.reduce_scatter(xs, dtype, op, order)
    inputs = to_device(torch, xs, dtype, dev)
    shards = lt.reduce_scatter_keep_shards(inputs, op=op, order=order)
    torch.cuda.synchronize()
    assert inputs == []
    q = vc.vc_shard_count(M, n)
    assert len(shards) == n and all(s.numel() == q for s in shards)
    for r in range(n):
        assert_bits_equal(to_host(shards[r], dtype), want[r], dtype, f"kept shard {r}")
    # the shards gathered into fresh outputs give the oracle's AllReduce
    outs = lt.all_gather_new(shards, M)
    torch.cuda.synchronize()
    assert shards == []
    want_ar = oracle.all_reduce(xs, dtype, op, order)
    for r in range(n):
        assert_bits_equal(to_host(outs[r], dtype), want_ar[r], dtype, f"gathered rank {r}")


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
    them, so their memory is not handed out before the ReduceScatter ran.
    The outputs are the oracle's AllReduce of the host inputs."""
    torch, vc, lt, dev = env
    n, M = 4, 1 << 22
    xs = _host_inputs("float32", n, M, seed=2)
    want = oracle.all_reduce(xs, "float32", "sum", "ring")
    src = to_device(torch, xs, "float32", dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
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
        assert_bits_equal(to_host(outs[r], "float32"), want[r], "float32", f"rank {r}")
    del junk
