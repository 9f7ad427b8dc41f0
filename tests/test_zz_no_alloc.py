"""vc_all_reduce_decomposed_noalloc: the decomposed AllReduce for callers that
cannot allocate device memory (a framework allocator owns the memory, the path
cannot pay for cudaMalloc, or the caller holds only its input and output
buffers).  Its shards live in a fixed 32 MiB scratch array inside the library.

Checked through the C ABI on two calls in a row with different inputs (the
second call must not see anything the first left in the shared scratch):
against the CPU oracle's decomposed AllReduce of the same host inputs, and
against the existing vc_all_reduce_decomposed with caller-allocated shards.
Both in the same order, so bit for bit.  Kept in a file of its own that
pytest collects last; it passes alone in a fresh process and after the other
tests.
"""
from __future__ import annotations

import ctypes

import pytest

import oracle
import synthetic_inputs as si
from gpu_util import assert_bits_equal, to_device, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import allreduce_reducescatter_allgather_gb300 as vc
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    return torch, vc, dev


CASES = [("float32", 8, 1_000_003, "sum", "ring"),
         ("float32", 8, 1_000_003, "sum", "recursive_halving"),
         ("bfloat16", 8, 2_000_001, "avg", "pairwise_tree"),
         ("int64", 4, 777_777, "prod", "ring"),
         ("int32", 64, 65_537, "max", "ring"),
         ("float32", 3, 17, "min", "ring"),
         ("float32", 12, 300_007, "sum", "double_binary_tree"),
         ("int32", 5, 100_003, "sum", "pairwise_tree")]


def _inputs(dtype, n, M, seed):
    if dtype in ("float32", "bfloat16"):
        return si.generate(dtype, "uniform_pm1", n, M, seed=seed)
    return si.generate(dtype, "uniform_int", n, M, seed=seed, lo=-100, hi=100)


@pytest.mark.parametrize("dtype,n,M,op,order", CASES)
def test_noalloc_matches_oracle_and_decomposed_on_two_calls(env, dtype, n, M, op, order):
    torch, vc, dev = env
    from allreduce_reducescatter_allgather_gb300._binding import (
        DTYPES, OPS, ORDERS, lib, pointer_table)
    L = lib()
    fn = L.vc_all_reduce_decomposed_noalloc
    vpp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream(dev)
    q = vc.vc_shard_count(M, n)
    for call, seed in enumerate((11, 12)):
        xs = _inputs(dtype, n, M, seed + n)
        d = to_device(torch, xs, dtype, dev)
        # the existing entry point, with caller-allocated shards
        shards = [torch.empty(q, dtype=d[0].dtype, device=dev) for _ in range(n)]
        ref = [torch.empty_like(t) for t in d]
        vc.vc_all_reduce_decomposed(d, shards, ref, op=op, order=order)
        # the no-allocation entry point, straight through the C ABI
        got = [torch.full_like(t, 3) for t in d]
        status = fn(pointer_table([t.data_ptr() for t in d]),
                    pointer_table([t.data_ptr() for t in got]), n, M, DTYPES[dtype], OPS[op],
                    ORDERS[order], ctypes.c_void_p(stream.cuda_stream))
        assert status == 0, L.vc_status_string(status)
        torch.cuda.synchronize()
        _, want = oracle.all_reduce_decomposed(xs, dtype, op, order)
        for r in range(n):
            assert_bits_equal(to_host(got[r], dtype), want[r], dtype,
                              f"call {call} rank {r} vs oracle")
            assert_bits_equal(to_host(got[r], dtype), to_host(ref[r], dtype), dtype,
                              f"call {call} rank {r} vs vc_all_reduce_decomposed")


def test_noalloc_in_place_through_binding(env):
    torch, vc, dev = env
    n, M = 8, 100_003
    xs = _inputs("float32", n, M, 5)
    d = to_device(torch, xs, "float32", dev)
    q = vc.vc_shard_count(M, n)
    ref = [torch.empty_like(t) for t in d]
    vc.vc_all_reduce_decomposed(d, [torch.empty(q, device=dev) for _ in range(n)], ref)
    vc.vc_all_reduce_decomposed_noalloc(d)  # in place
    torch.cuda.synchronize()
    _, want = oracle.all_reduce_decomposed(xs, "float32", "sum", "ring")
    for r in range(n):
        assert_bits_equal(to_host(d[r], "float32"), want[r], "float32", f"rank {r} vs oracle")
        assert torch.equal(d[r], ref[r])


def test_noalloc_rejects_shards_beyond_the_scratch(env):
    torch, vc, dev = env
    from allreduce_reducescatter_allgather_gb300._binding import (
        NOALLOC_SCRATCH_BYTES, DTYPES, OPS, ORDERS, lib, noalloc_scratch_needed, pointer_table)
    n = 4
    M = NOALLOC_SCRATCH_BYTES // 4 + 1  # fp32: one element more than fits
    assert noalloc_scratch_needed(M, n, "float32") > NOALLOC_SCRATCH_BYTES
    d = [torch.zeros(M, device=dev) for _ in range(n)]
    out = [torch.full((M,), 9.0, device=dev) for _ in range(n)]
    with pytest.raises(ValueError, match="scratch"):
        vc.vc_all_reduce_decomposed_noalloc(d, out)
    status = lib().vc_all_reduce_decomposed_noalloc(
        pointer_table([t.data_ptr() for t in d]), pointer_table([t.data_ptr() for t in out]),
        n, M, DTYPES["float32"], OPS["sum"], ORDERS["ring"], None)
    assert status == 1  # VC_ERR_INVALID_ARGUMENT, nothing launched
    torch.cuda.synchronize()
    assert all(torch.all(t == 9.0).item() for t in out)
    # exactly at the limit it runs
    M = NOALLOC_SCRATCH_BYTES // 4
    d = [torch.ones(M, device=dev) for _ in range(n)]
    out = [torch.empty(M, device=dev) for _ in range(n)]
    vc.vc_all_reduce_decomposed_noalloc(d, out)
    torch.cuda.synchronize()
    assert all(torch.all(t == float(n)).item() for t in out)

