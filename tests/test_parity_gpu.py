"""Parity of the CUDA collectives with the CPU oracle, through the C ABI.

Integers, and floats in the same order as the oracle, must match bit for bit;
a float result in a different order must lie within the bound the tests name.
Small and medium cases compare every element of every output; the full-size
four-rank 256 MiB workload compares a million sampled indices (plus every
chunk boundary) one by one, and checks properties that hold at any size on
the device.  Output buffers carry guard elements after their end (and, when
they start inside their allocation, before it) that must come back
untouched.
"""
from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from conftest import ints, read_golden
from gpu_util import assert_bits_equal, to_device, to_host, torch_dtype

pytestmark = pytest.mark.gpu

ORDERS = ["ring", "recursive_halving", "pairwise_tree", "double_binary_tree"]
OPS = ["sum", "prod", "max", "min", "avg"]
GUARD = 32  # guard elements after every output buffer


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
    return SimpleNamespace(torch=torch, vc=vc, dev=dev)


def orders_for(n):
    """Every order is defined for any N but recursive halving (N = 2^k)."""
    return [o for o in ORDERS if n & (n - 1) == 0 or o != "recursive_halving"]


def sentinel(dtype):
    return {"int32": -77, "int64": -77, "float32": 12345.0, "bfloat16": 77.0}[dtype]


class Guarded:
    """N device buffers of `numel` elements, each followed by GUARD sentinel
    elements inside the same allocation, optionally starting `offset`
    elements into it (a misaligned base)."""

    def __init__(self, env, n, numel, dtype, offset=0):
        torch = env.torch
        self.dtype = dtype
        self.bigs = []
        self.views = []
        for _ in range(n):
            big = torch.full((offset + numel + GUARD,), sentinel(dtype),
                             dtype=torch_dtype(torch, dtype), device=env.dev)
            self.bigs.append(big)
            self.views.append(big[offset:offset + numel])
        self.offset, self.numel = offset, numel

    def check_guards(self, env):
        for big in self.bigs:
            tail = big[self.offset + self.numel:]
            assert env.torch.all(tail == sentinel(self.dtype)).item(), "guard overwritten"
            head = big[:self.offset]
            assert env.torch.all(head == sentinel(self.dtype)).item(), "head guard overwritten"

    def host(self):
        return [to_host(v, self.dtype) for v in self.views]


def run_all_paths(env, xs, dtype, op, order, offset=0):
    """RS, AG (of the GPU's own shards), fused AR and decomposed AR."""
    vc = env.vc
    n, M = len(xs), xs[0].size
    q = vc.vc_shard_count(M, n)
    d = to_device(env.torch, xs, dtype, env.dev, offset=offset)
    z = Guarded(env, n, q, dtype, offset)
    g = Guarded(env, n, M, dtype, offset)
    y = Guarded(env, n, M, dtype, offset)
    s2 = Guarded(env, n, q, dtype, offset)
    y2 = Guarded(env, n, M, dtype, offset)
    vc.vc_reduce_scatter(d, z.views, op=op, order=order)
    vc.vc_all_gather(z.views, g.views)
    vc.vc_all_reduce(d, y.views, op=op, order=order)
    vc.vc_all_reduce_decomposed(d, s2.views, y2.views, op=op, order=order)
    env.torch.cuda.synchronize()
    for b in (z, g, y, s2, y2):
        b.check_guards(env)
    return SimpleNamespace(rs=z.host(), ag=g.host(), ar=y.host(), dec_shards=s2.host(),
                           dec=y2.host())


def check_all_paths(res, xs, dtype, op, order, tag=""):
    n = len(xs)
    oz = oracle.reduce_scatter(xs, dtype, op, order)
    oy = oracle.all_reduce(xs, dtype, op, order)
    og = oracle.all_gather(res.rs, xs[0].size, dtype)  # AG on its own, from the GPU's shards
    for r in range(n):
        t = f"{tag} {dtype} {op} {order} rank {r}"
        assert_bits_equal(res.rs[r], oz[r], dtype, "RS " + t)
        assert_bits_equal(res.dec_shards[r], oz[r], dtype, "decomposed shards " + t)
        assert_bits_equal(res.ar[r], oy[r], dtype, "AR " + t)
        assert_bits_equal(res.dec[r], oy[r], dtype, "decomposed AR " + t)
        assert_bits_equal(res.ag[r], og[r], dtype, "AG " + t)


def gen(dtype, n, M, seed):
    if dtype in ("float32", "bfloat16"):
        return si.generate(dtype, "uniform_pm1", n, M, seed=seed)
    return si.generate(dtype, "uniform_int", n, M, seed=seed, lo=-100, hi=100)


# ------------------------------------------------- the pages' contracts --

@pytest.mark.parametrize("order", ORDERS)
def test_worked_example(env, order):
    """Four ranks, twenty int64, 100r + i: 600 + 4i, shards of five, every
    path and op ("NCCL 专家课程 07", 一个四 rank 手算例子)."""
    g = read_golden("worked_example_n4_m20_int64.txt")
    xs = si.generate("int64", "rank_linear", 4, 20, seed=0)
    res = run_all_paths(env, xs, "int64", "sum", order)
    expect = np.array(ints(g["allreduce"]), np.int64)
    for r in range(4):
        np.testing.assert_array_equal(res.ar[r], expect)
        np.testing.assert_array_equal(res.dec[r], expect)
        np.testing.assert_array_equal(res.rs[r], np.array(ints(g[f"shard{r}"]), np.int64))
    for op in OPS:
        check_all_paths(run_all_paths(env, xs, "int64", op, order), xs, "int64", op, order)


def test_negative_contracts(env):
    """A rolled gather and RS(MAX)+AG both differ from AR(SUM) on the GPU's
    own results (条件一, 条件二)."""
    vc, torch = env.vc, env.torch
    xs = si.generate("int64", "rank_linear", 4, 20, seed=0)
    d = to_device(torch, xs, "int64", env.dev)
    direct = [torch.empty_like(t) for t in d]
    vc.vc_all_reduce(d, direct, op="sum")
    zmax = [torch.empty(5, dtype=torch.int64, device=env.dev) for _ in range(4)]
    gmax = [torch.empty_like(t) for t in d]
    vc.vc_reduce_scatter(d, zmax, op="max")
    vc.vc_all_gather(zmax, gmax)
    zsum = [torch.empty(5, dtype=torch.int64, device=env.dev) for _ in range(4)]
    gsum = [torch.empty_like(t) for t in d]
    vc.vc_reduce_scatter(d, zsum, op="sum")
    vc.vc_all_gather(zsum, gsum)
    torch.cuda.synchronize()
    assert torch.equal(direct[0], gsum[0])
    rolled = gsum[0].reshape(4, -1).roll(1, dims=0).reshape(-1)
    assert not torch.equal(direct[0], rolled)
    assert not torch.equal(direct[0], gmax[0])


def test_padding_contract(env):
    """M = 1003 on four ranks: shards of 251, RS + AG trimmed equals the direct
    AR; an unpadded 250-element output is rejected before any kernel runs and
    stays untouched (Contract 实验四)."""
    vc, torch = env.vc, env.torch
    g = read_golden("padding_m1003_n4.txt")
    n, M = int(g["n"]), int(g["M"])
    xs = si.generate("int64", "rank_linear", n, M, seed=0)
    res = run_all_paths(env, xs, "int64", "sum", "ring")
    assert all(z.size == int(g["q"]) for z in res.rs)
    for r in range(n):
        np.testing.assert_array_equal(res.dec[r], res.ar[r])
    check_all_paths(res, xs, "int64", "sum", "ring")
    d = to_device(torch, xs, "int64", env.dev)
    bad = [torch.full((int(g["unpadded_output"]),), 7, dtype=torch.int64, device=env.dev)
           for _ in range(n)]
    with pytest.raises(ValueError, match="ceil"):
        vc.vc_reduce_scatter(d, bad)
    torch.cuda.synchronize()
    assert all(torch.all(b == 7).item() for b in bad)


def test_max_is_not_zero_padded(env):
    """MAX over all-negative int64 with M % N != 0: the shard tail holds the
    dtype minimum and matches the identity-padded oracle, not a zero pad."""
    vc, torch = env.vc, env.torch
    n, M = 4, 19
    xs = [-(100 * r + np.arange(M, dtype=np.int64)) - 1 for r in range(n)]
    res = run_all_paths(env, xs, "int64", "max", "ring")
    check_all_paths(res, xs, "int64", "max", "ring")
    q = oracle.shard_count(M, n)
    zero_padded = [np.concatenate([x, np.zeros(n * q - M, np.int64)]) for x in xs]
    bad = oracle.reduce_scatter(zero_padded, "int64", "max", "ring")
    assert not np.array_equal(res.rs[-1], bad[-1])
    assert res.rs[-1][-1] == np.iinfo(np.int64).min
    del vc, torch


# ------------------------------------------------------ workload configs --

@pytest.mark.parametrize("order", ORDERS)
@pytest.mark.parametrize("op", OPS)
def test_n8_m1000003_fp32(env, op, order):
    """Eight ranks, 1,000,003 fp32 uniform[-1,1) (q = 125,001, five padding
    slots, misaligned shard starts): every path bit for bit."""
    w = si.WORKLOADS["n8_m1000003_f32_uniform"]
    xs = si.generate(w["dtype"], w["dist"], w["n"], w["M"], seed=w["seed"])
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.125) for x in xs]
    res = run_all_paths(env, xs, "float32", op, order)
    check_all_paths(res, xs, "float32", op, order)


@pytest.fixture(scope="module")
def bucket_bf16():
    w = si.WORKLOADS["n8_bucket25mib_bf16_normal"]
    return si.generate(w["dtype"], w["dist"], w["n"], w["M"], seed=w["seed"], sigma=w["sigma"])


@pytest.mark.parametrize("order", ORDERS)
def test_gradient_bucket_bf16(env, bucket_bf16, order):
    """Eight ranks, one 25 MiB bucket of bf16 normal(0, 1e-3): SUM then AVG
    with fp32 accumulation; RS (ZeRO-style shards) and fused AR bit for bit."""
    vc, torch = env.vc, env.torch
    xs = bucket_bf16
    n, M = len(xs), xs[0].size
    q = vc.vc_shard_count(M, n)
    d = to_device(torch, xs, "bfloat16", env.dev)
    for op in ("sum", "avg"):
        z = Guarded(env, n, q, "bfloat16")
        y = Guarded(env, n, M, "bfloat16")
        vc.vc_reduce_scatter(d, z.views, op=op, order=order)
        vc.vc_all_reduce(d, y.views, op=op, order=order)
        torch.cuda.synchronize()
        z.check_guards(env)
        y.check_guards(env)
        oz = oracle.reduce_scatter(xs, "bfloat16", op, order)
        oy = oracle.all_reduce(xs, "bfloat16", op, order)
        zh, yh = z.host(), y.host()
        for r in range(n):
            assert_bits_equal(zh[r], oz[r], "bfloat16", f"RS {op} {order}")
        assert_bits_equal(yh[0], oy[0], "bfloat16", f"AR {op} {order}")
        for r in range(1, n):
            assert torch.equal(y.views[r], y.views[0])


def test_bf16_other_order_within_one_ulp(env, bucket_bf16):
    """Against an oracle in a different order, bf16 results lie within one
    bf16 ulp of the fp32-accumulated oracle rounded to bf16."""
    vc, torch = env.vc, env.torch
    xs = [x[:2_000_000] for x in bucket_bf16]
    d = to_device(torch, xs, "bfloat16", env.dev)
    y = [torch.empty_like(t) for t in d]
    vc.vc_all_reduce(d, y, op="sum", order="ring")
    torch.cuda.synchronize()
    got = to_host(y[0], "bfloat16").astype(np.int32)
    for order in ("recursive_halving", "pairwise_tree"):
        ref = oracle.all_reduce(xs, "bfloat16", "sum", order)[0].astype(np.int32)
        # adjacent bf16 values of one sign differ by 1 in their bit pattern
        same_sign = (got & 0x8000) == (ref & 0x8000)
        diff = np.abs(got - ref)
        ok = (same_sign & (diff <= 1)) | ((got & 0x7FFF) == 0) & ((ref & 0x7FFF) <= 1) \
            | ((ref & 0x7FFF) == 0) & ((got & 0x7FFF) <= 1)
        assert np.all(ok), order


def _sample_indices(rng, limit, q, n, K):
    idx = rng.integers(0, limit, size=K, dtype=np.int64)
    edges = []
    for c in range(n + 1):
        for off in (-2, -1, 0, 1, 2):
            edges.append(c * q + off)
    edges += [limit - 1, limit - 2]
    edges = np.array([e for e in edges if 0 <= e < limit], np.int64)
    return np.unique(np.concatenate([idx, edges]))


def _check_sampled(env, d, y0, z, dtype, op, order, K=1 << 20, seed=0):
    """Compare sampled AR outputs (y0) and RS shards (z) with the oracle
    reducing those indices one by one from the device's own input bytes."""
    torch = env.torch
    n, M = len(d), d[0].numel()
    q = env.vc.vc_shard_count(M, n)
    rng = np.random.default_rng(seed)
    # AllReduce indices
    idx = _sample_indices(rng, M, q, n, K)
    ti = torch.from_numpy(idx).to(env.dev)
    xs_at = [to_host(t[ti], dtype) for t in d]
    want = oracle.reduce_points(xs_at, idx, n, M, dtype, op, order)
    assert_bits_equal(to_host(y0[ti], dtype), want, dtype, f"sampled AR {dtype} {op} {order}")
    # ReduceScatter indices over the padded range [0, N*q)
    idx = _sample_indices(rng, n * q, q, n, K // 4)
    safe = torch.from_numpy(np.minimum(idx, M - 1)).to(env.dev)
    xs_at = [to_host(t[safe], dtype) for t in d]
    want = oracle.reduce_points(xs_at, idx, n, M, dtype, op, order)
    flat = torch.cat([zz for zz in z])
    got = to_host(flat[torch.from_numpy(idx).to(env.dev)], dtype)
    assert_bits_equal(got, want, dtype, f"sampled RS {dtype} {op} {order}")


@pytest.mark.parametrize("name", ["n4_256mib_f32_normal", "n4_m67108864_i64_uniform"])
def test_full_size_four_ranks(env, name):
    """Four ranks of 67,108,864 elements (fp32 normal, int64 uniform): fused
    AR, RS and decomposed AR at full size in the bench's launch configuration;
    a million sampled indices against the oracle, and on the device: all AR
    outputs identical, AR == decomposed AR, RS shard r == AR[rq : rq+q]."""
    vc, torch = env.vc, env.torch
    w = dict(si.WORKLOADS[name])
    dtype = w.pop("dtype")
    d = si.generate_device(torch, dtype, w.pop("dist"), w.pop("n"), w.pop("M"),
                           w.pop("seed"), env.dev, **w)
    n, M = len(d), d[0].numel()
    q = vc.vc_shard_count(M, n)
    for order in ORDERS:
        y = [torch.empty_like(t) for t in d]
        z = [torch.empty(q, dtype=d[0].dtype, device=env.dev) for _ in range(n)]
        s2 = [torch.empty(q, dtype=d[0].dtype, device=env.dev) for _ in range(n)]
        y2 = [torch.empty_like(t) for t in d]
        vc.vc_all_reduce(d, y, op="sum", order=order)
        vc.vc_reduce_scatter(d, z, op="sum", order=order)
        vc.vc_all_reduce_decomposed(d, s2, y2, op="sum", order=order)
        torch.cuda.synchronize()
        for r in range(n):
            assert torch.equal(y[r], y[0])
            assert torch.equal(y2[r], y[0])
            assert torch.equal(s2[r], z[r])
            assert torch.equal(z[r], y[0][r * q:(r + 1) * q])
        _check_sampled(env, d, y[0], z, dtype, "sum", order, seed=ORDERS.index(order))
        del y, z, s2, y2
    torch.cuda.empty_cache()


# ------------------------------------------------------------- the sweep --

SWEEP_DTYPES = ["int32", "int64", "float32", "bfloat16"]
SWEEP_OPS = ["sum", "max", "min", "prod"]


def _sweep_cases(max_bytes):
    cases = []
    k = 0
    for dtype in SWEEP_DTYPES:
        es = {"int32": 4, "int64": 8, "float32": 4, "bfloat16": 2}[dtype]
        for n in (2, 4, 8, 16, 64):
            for nbytes in [8192 * 4 ** j for j in range(9)] + [1 << 30]:
                if nbytes > max_bytes or n * nbytes > (64 << 30):
                    continue
                op = SWEEP_OPS[k % 4]
                order = ORDERS[(k // 4) % 4]
                k += 1
                cases.append((dtype, n, nbytes // es, op, order))
    return cases


@pytest.mark.parametrize("dtype,n,M,op,order", _sweep_cases(512 << 10))
def test_sweep_full_compare(env, dtype, n, M, op, order):
    """Per-rank sizes 8 KiB .. 512 KiB, N in {2, 4, 8, 16, 64}, four dtypes,
    ops and orders cycled: every path, every element."""
    xs = gen(dtype, n, M, seed=1000 + n + M)
    if op == "prod" and dtype in ("float32", "bfloat16"):
        xs = gen_prod_floats(dtype, n, M)
    res = run_all_paths(env, xs, dtype, op, order)
    check_all_paths(res, xs, dtype, op, order, tag=f"N={n} M={M}")


def gen_prod_floats(dtype, n, M):
    # factors near 1 keep long products finite
    xs = si.generate("float32", "uniform_pm1", n, M, seed=n * 7 + M)
    xs = [np.float32(1.0) + x * np.float32(1.0 / 64) for x in xs]
    if dtype == "bfloat16":
        import torch
        return [torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                for x in xs]
    return xs


LARGE = [("float32", 2, 1 << 28), ("bfloat16", 16, 1 << 28), ("int32", 64, 1 << 25),
         ("int64", 8, 1 << 26), ("float32", 64, 1 << 28)]


@pytest.mark.parametrize("dtype,n,M", LARGE)
def test_sweep_large_sampled(env, dtype, n, M):
    """Large sweep points (up to 1 GiB per rank, and 64 ranks x 1 GiB): RS and
    in-place AR, sampled indices against the oracle, outputs identical."""
    vc, torch = env.vc, env.torch
    dist = "uniform_pm1" if dtype in ("float32", "bfloat16") else "uniform_int"
    kw = {} if dist == "uniform_pm1" else {"lo": -100, "hi": 100}
    d = si.generate_device(torch, dtype, dist, n, M, seed=7 + n, device=env.dev, **kw)
    q = vc.vc_shard_count(M, n)
    order = "pairwise_tree" if dtype == "bfloat16" else "ring"
    z = [torch.empty(q, dtype=d[0].dtype, device=env.dev) for _ in range(n)]
    vc.vc_reduce_scatter(d, z, op="sum", order=order)
    torch.cuda.synchronize()
    rng = np.random.default_rng(n)
    idx = _sample_indices(rng, n * q, q, n, 1 << 16)
    safe = torch.from_numpy(np.minimum(idx, M - 1)).to(env.dev)
    xs_at = [to_host(t[safe], dtype) for t in d]
    want = oracle.reduce_points(xs_at, idx, n, M, dtype, "sum", order)
    got = to_host(torch.cat(z)[torch.from_numpy(idx).to(env.dev)], dtype)
    assert_bits_equal(got, want, dtype, "sampled RS")
    del z
    # the in-place AR overwrites the inputs: keep the operands of the probes
    probe = _sample_indices(rng, M, q, n, 1 << 16)
    tp = torch.from_numpy(probe).to(env.dev)
    xs_probe = [to_host(t[tp], dtype) for t in d]
    vc.vc_all_reduce(d, None, op="sum", order=order)
    torch.cuda.synchronize()
    want = oracle.reduce_points(xs_probe, probe, n, M, dtype, "sum", order)
    for r in (0, n // 2, n - 1):
        assert_bits_equal(to_host(d[r][tp], dtype), want, dtype, f"in-place AR rank {r}")
    for r in range(1, n):
        assert torch.equal(d[r], d[0])
    del d
    torch.cuda.empty_cache()


# ------------------------------------------------------------ edge cases --

EDGE_NM = [(1, 1), (1, 37), (2, 1), (2, 3), (3, 2), (3, 7), (4, 3), (4, 5), (5, 1), (7, 6),
           (7, 15), (8, 7), (8, 9), (8, 33), (13, 12), (13, 200), (16, 17), (32, 31),
           (63, 1000), (64, 63), (64, 65), (64, 1031)]


@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
@pytest.mark.parametrize("offset", [0, 1])
def test_edge_shapes(env, dtype, offset):
    """Tiny and ragged shapes (M < N, M = N +- 1, odd q, every residue of M
    and q modulo the vector width), N = 1 and N = 64, and bases one element
    off 16-byte alignment: every path, every element."""
    k = 0
    for n, M in EDGE_NM:
        for order in orders_for(n):
            op = OPS[k % len(OPS)]
            k += 1
            xs = gen(dtype, n, M, seed=n * 1000 + M)
            res = run_all_paths(env, xs, dtype, op, order, offset=offset)
            check_all_paths(res, xs, dtype, op, order, tag=f"N={n} M={M} off={offset}")


EVERY_N = list(range(1, 18)) + [31, 32, 33, 48, 63, 64]


@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
def test_every_rank_count(env, dtype):
    """Every rank count from 1 to 17 and around 32 and 64, in every order it
    takes: each compile-time instance (ring 1..8, 16, 32, 64; trees 3, 5, 6,
    7 and the powers of two) and the run-time ones, on the vector path (the
    length spans many vectors per thread and ends in a ragged tail), every
    path, every element."""
    k = 0
    for n in EVERY_N:
        M = 3 * 4096 + 17 * n + 5
        for order in orders_for(n):
            op = OPS[k % len(OPS)]
            k += 1
            xs = gen(dtype, n, M, seed=9000 + 31 * n + k)
            if op == "prod" and dtype in ("float32", "bfloat16"):
                xs = gen_prod_floats(dtype, n, M)
            res = run_all_paths(env, xs, dtype, op, order)
            check_all_paths(res, xs, dtype, op, order, tag=f"N={n} M={M}")


TREE_N = [3, 5, 6, 7, 9, 12, 17, 24, 33, 48, 63]


@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
@pytest.mark.parametrize("order", ["pairwise_tree", "double_binary_tree"])
def test_trees_any_rank_count(env, dtype, order):
    """Tree orders at rank counts that are not powers of two (compile-time
    and run-time N, both envelopes): every path, every element, four ops, a
    size that spans many blocks and ends in a ragged tail."""
    k = 0
    for n in TREE_N:
        M = 40_000 + 13 * n + 1
        op = SWEEP_OPS[k % 4]
        k += 1
        xs = gen(dtype, n, M, seed=5000 + n)
        if op == "prod" and dtype in ("float32", "bfloat16"):
            xs = gen_prod_floats(dtype, n, M)
        res = run_all_paths(env, xs, dtype, op, order)
        check_all_paths(res, xs, dtype, op, order, tag=f"N={n} M={M}")


@pytest.mark.parametrize("n", [6, 12, 48])
def test_trees_any_rank_count_large_sampled(env, n):
    """64 MiB per rank, N not a power of two: fused AR and RS in both tree
    orders, sampled indices against the oracle; all AR outputs identical and
    RS shard r == AR[rq : rq+q] on the device."""
    vc, torch = env.vc, env.torch
    M = 1 << 24
    d = si.generate_device(torch, "float32", "normal", n, M, seed=90 + n, device=env.dev)
    q = vc.vc_shard_count(M, n)
    for order in ("pairwise_tree", "double_binary_tree"):
        y = [torch.empty_like(t) for t in d]
        z = [torch.empty(q, dtype=d[0].dtype, device=env.dev) for _ in range(n)]
        vc.vc_all_reduce(d, y, op="sum", order=order)
        vc.vc_reduce_scatter(d, z, op="sum", order=order)
        torch.cuda.synchronize()
        for r in range(n):
            assert torch.equal(y[r], y[0])
            lo, hi = r * q, min((r + 1) * q, M)
            if lo < M:
                assert torch.equal(z[r][:hi - lo], y[0][lo:hi])
        _check_sampled(env, d, y[0], z, "float32", "sum", order, seed=n, K=1 << 16)
        del y, z
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
def test_residues(env, dtype):
    """M and q in every residue class modulo the vector width, N = 4 and 8."""
    V = {"int32": 4, "int64": 2, "float32": 4, "bfloat16": 8}[dtype]
    for n in (4, 8):
        for M in range(n * 64, n * 64 + n * V + 1):
            xs = gen(dtype, n, M, seed=M)
            res = run_all_paths(env, xs, dtype, "sum", "ring")
            check_all_paths(res, xs, dtype, "sum", "ring", tag=f"N={n} M={M}")


@pytest.mark.parametrize("dtype", ["float32", "int64", "bfloat16"])
def test_in_place(env, dtype):
    """In-place AR and in-place decomposed AR (recvbufs = sendbufs)."""
    vc, torch = env.vc, env.torch
    n, M = 8, 100_003
    xs = gen(dtype, n, M, seed=3)
    for order in ORDERS:
        oy = oracle.all_reduce(xs, dtype, "sum", order)
        d = to_device(torch, xs, dtype, env.dev)
        vc.vc_all_reduce(d, None, op="sum", order=order)
        d2 = to_device(torch, xs, dtype, env.dev)
        q = vc.vc_shard_count(M, n)
        sh = [torch.empty(q, dtype=d2[0].dtype, device=env.dev) for _ in range(n)]
        vc.vc_all_reduce_decomposed(d2, sh, None, op="sum", order=order)
        torch.cuda.synchronize()
        for r in range(n):
            assert_bits_equal(to_host(d[r], dtype), oy[r], dtype, f"in-place AR {order}")
            assert_bits_equal(to_host(d2[r], dtype), oy[r], dtype, f"in-place dec {order}")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int32"])
def test_in_place_straddling_vectors(env, dtype):
    """In-place AllReduce where vectors straddle chunk boundaries (and the
    double tree's halfway point): the straddling path folds the vector once
    per chunk and stores each fold's lanes element by element, so the second
    fold re-reads a vector whose other lanes the first fold already
    overwrote.  Run-time N (12, 33) and compile-time N (6, 8), every order,
    SUM and AVG, against the oracle."""
    vc, torch = env.vc, env.torch
    for n in (6, 8, 12, 33):
        M = 7 * n * 1024 + 5 * n + 3  # q = 7174: not a whole number of vectors
        for order in orders_for(n):
            for op in ("sum", "avg") if dtype != "int32" else ("sum", "max"):
                xs = gen(dtype, n, M, seed=n * 131 + len(order))
                oy = oracle.all_reduce(xs, dtype, op, order)
                d = to_device(torch, xs, dtype, env.dev)
                vc.vc_all_reduce(d, None, op=op, order=order)
                torch.cuda.synchronize()
                for r in range(n):
                    assert_bits_equal(to_host(d[r], dtype), oy[r], dtype,
                                      f"in-place N={n} {order} {op} rank {r}")


ESIZE = {"int32": 4, "int64": 8, "float32": 4, "bfloat16": 2}


@pytest.mark.parametrize("dtype", ["float32", "bfloat16", "int64"])
def test_partial_last_span(env, dtype):
    """The reduction kernels with the operands preloaded (N <= 8) give a
    thread U vectors (four up to four ranks, two up to eight) in each span of
    256 x U vectors, and take the last span of the index space first; there
    a thread may own only its first k < U vectors.  Shapes whose vector count
    is a whole number of spans, one vector short of it, one past it, and one
    element short, on 3 and 8 ranks, every order, SUM and MAX, all paths
    against the oracle."""
    V = 16 // ESIZE[dtype]
    for n, U in ((3, 4), (8, 2)):
        span = 256 * U
        for nv, extra in ((3 * span, 0), (3 * span - 1, 0), (3 * span + 1, 0), (3 * span, -1)):
            M = nv * V + extra
            for order in orders_for(n):
                for op in ("sum", "max"):
                    xs = gen(dtype, n, M, seed=M + n)
                    res = run_all_paths(env, xs, dtype, op, order)
                    check_all_paths(res, xs, dtype, op, order, tag=f"N={n} M={M}")


@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
def test_shards_off_the_vector_grid(env, dtype):
    """When q elements are not a whole number of 16-byte vectors, shard c
    holds the indices from cq on, so its vectors sit off the 16-byte grid by
    a different amount for each c; a shard buffer may also start off the
    grid itself.  ReduceScatter stores and AllGather loads then realign
    across the warp.  Every offset a shard can take (q = 1 and q = -1 modulo
    the vector width, eight ranks, shard bases moved by 0 .. V-1 elements,
    inputs and outputs aligned), and q a whole number of vectors with only
    the bases moved; several warps per shard, a padded last shard; guards
    before and after every shard and output.  Also at three ranks (the
    compile-time kernels with four vectors per thread) and twelve (the
    kernel with a run-time N)."""
    vc, torch = env.vc, env.torch
    V = 16 // ESIZE[dtype]
    k = 0
    # eight ranks: the compile-time kernels that preload their operands;
    # three: the same with four vectors per thread; twelve: the kernel with
    # a run-time N (one vector per thread, element-aligned pieces)
    for n, q, shift in [(8, q, sh) for q in (V * 301 + 1, V * 97 + V - 1, V * 160)
                        for sh in range(V)] + \
                       [(n, q, sh) for n in (3, 12) for q in (V * 211 + 1, V * 53 + V - 1)
                        for sh in range(V)]:
        M = n * q - min(3, n - 1)  # ceil(M / n) = q
        op = SWEEP_OPS[k % len(SWEEP_OPS)]
        orders = orders_for(n)
        order = orders[k % len(orders)] if dtype in ("float32", "bfloat16") else "ring"
        k += 1
        xs = gen(dtype, n, M, seed=7100 + 13 * q + shift)
        if op == "prod" and dtype in ("float32", "bfloat16"):
            xs = gen_prod_floats(dtype, n, M)
        d = to_device(torch, xs, dtype, env.dev)
        z = Guarded(env, n, q, dtype, shift)
        g = Guarded(env, n, M, dtype)
        vc.vc_reduce_scatter(d, z.views, op=op, order=order)
        vc.vc_all_gather(z.views, g.views)
        torch.cuda.synchronize()
        z.check_guards(env)
        g.check_guards(env)
        oz = oracle.reduce_scatter(xs, dtype, op, order)
        zh = z.host()
        og = oracle.all_gather(zh, M, dtype)
        gh = g.host()
        for r in range(n):
            t = f"{dtype} {op} {order} N={n} q={q} shift={shift} rank {r}"
            assert_bits_equal(zh[r], oz[r], dtype, "RS " + t)
            assert_bits_equal(gh[r], og[r], dtype, "AG " + t)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_avg_subnormal_quotients(env, dtype):
    """AVG divides the ordered sum by N once.  For N a power of two the
    kernels multiply by the exact reciprocal 2^-k instead; the correctly
    rounded product and quotient are the same bits, including where the
    result is subnormal.  Operands near the smallest normal fp32 (biased
    exponents 1..9, both signs), so many quotients fall below it; every
    path against the oracle's division, at power-of-two N and at N = 3, 12."""
    vc, torch = env.vc, env.torch
    rng = np.random.default_rng(17)
    for n in (2, 3, 4, 8, 12, 16, 64):
        M = 4099
        xs = []
        for _ in range(n):
            bits = (rng.integers(1, 10, M, dtype=np.uint32) << 23) \
                | rng.integers(0, 1 << 23, M, dtype=np.uint32) \
                | (rng.integers(0, 2, M, dtype=np.uint32) << 31)
            f = bits.view(np.float32)
            xs.append(f if dtype == "float32" else oracle.bf16_round(f))
        for order in orders_for(n):
            res = run_all_paths(env, xs, dtype, "avg", order)
            check_all_paths(res, xs, dtype, "avg", order, tag=f"subnormal N={n}")
        oy = oracle.all_reduce(xs, dtype, "avg", "ring")
        as_f = oy[0].view(np.float32) if dtype == "float32" else \
            (oy[0].astype(np.uint32) << 16).view(np.float32)
        assert np.count_nonzero((as_f != 0) & (np.abs(as_f) < np.finfo(np.float32).tiny)) > 20


def test_all_gather_from_arbitrary_shards(env):
    """AG alone, from shards that are not RS outputs, with misaligned shard
    bases and q not a multiple of the vector width."""
    vc, torch = env.vc, env.torch
    for dtype in SWEEP_DTYPES:
        for n, M in ((3, 1000), (8, 1_000_003), (64, 4099)):
            q = vc.vc_shard_count(M, n)
            zs = gen(dtype, n, q, seed=q)
            for off in (0, 1):
                dz = to_device(torch, zs, dtype, env.dev, offset=off)
                y = Guarded(env, n, M, dtype)
                vc.vc_all_gather(dz, y.views)
                torch.cuda.synchronize()
                y.check_guards(env)
                want = oracle.all_gather(zs, M, dtype)
                yh = y.host()
                for r in range(n):
                    assert_bits_equal(yh[r], want[r], dtype, f"AG {dtype} N={n} off={off}")


@pytest.mark.parametrize("n", [8, 64])
def test_fp32_other_order_within_bound(env, n):
    """Against the oracle in another order, fp32 sums satisfy
    |gpu - oracle| <= 2 N 2^-24 sum_s |x^(s)_i|."""
    vc, torch = env.vc, env.torch
    M = 200_003
    xs = si.generate("float32", "uniform_pm1", n, M, seed=n)
    d = to_device(torch, xs, "float32", env.dev)
    absum = sum(np.abs(x.astype(np.float64)) for x in xs)
    for order in ORDERS:
        y = [torch.empty_like(t) for t in d]
        vc.vc_all_reduce(d, y, op="sum", order=order)
        torch.cuda.synchronize()
        got = to_host(y[0], "float32").astype(np.float64)
        for other in ORDERS + ["sequential"]:
            ref = oracle.all_reduce(xs, "float32", "sum", other)[0].astype(np.float64)
            assert np.all(np.abs(got - ref) <= 2 * n * 2.0 ** -24 * absum), (order, other)


def test_user_stream(env):
    """Calls enqueue on the stream they are given."""
    vc, torch = env.vc, env.torch
    n, M = 4, 1 << 20
    xs = gen("float32", n, M, seed=5)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = to_device(torch, xs, "float32", env.dev)
        y = [torch.empty_like(t) for t in d]
        vc.vc_all_reduce(d, y, op="sum", order="ring", stream=s)
    s.synchronize()
    oy = oracle.all_reduce(xs, "float32", "sum", "ring")
    assert_bits_equal(to_host(y[0], "float32"), oy[0], "float32", "stream")


# -------------------------------------------------------- reduce / broadcast --

@pytest.mark.parametrize("dtype", SWEEP_DTYPES)
def test_reduce_and_broadcast(env, dtype):
    """Reduce = the oracle's reduce (the AllReduce value at the root), bit for
    bit; Broadcast copies the root's buffer to every output; Reduce then
    Broadcast equals the fused AllReduce ("通信与互联（01）" 二.2)."""
    vc, torch = env.vc, env.torch
    for n, M, op, order in ((4, 20, "sum", "ring"), (8, 1_000_003, "max", "recursive_halving"),
                            (3, 4099, "prod", "ring"), (64, 5003, "sum", "pairwise_tree"),
                            (16, 65_537, "avg", "ring"), (1, 333, "min", "ring")):
        if op == "prod" and dtype in ("float32", "bfloat16"):
            xs = gen_prod_floats(dtype, n, M)
        else:
            xs = gen(dtype, n, M, seed=n + M)
        for off in (0, 1):
            d = to_device(torch, xs, dtype, env.dev, offset=off)
            root = Guarded(env, 1, M, dtype, off)
            vc.vc_reduce(d, root.views[0], op=op, order=order)
            outs = Guarded(env, n, M, dtype, off)
            vc.vc_broadcast(root.views[0], outs.views)
            ar = [torch.empty_like(t) for t in d]
            vc.vc_all_reduce(d, ar, op=op, order=order)
            torch.cuda.synchronize()
            root.check_guards(env)
            outs.check_guards(env)
            want = oracle.reduce(xs, dtype, op, order)
            got = to_host(root.views[0], dtype)
            assert_bits_equal(got, want, dtype, f"reduce N={n} M={M} {op} {order} off={off}")
            for r in range(n):
                assert_bits_equal(to_host(outs.views[r], dtype), want, dtype, "broadcast")
                assert torch.equal(ar[r], outs.views[r])


def test_reduce_in_place_at_root_and_broadcast_including_root(env):
    vc, torch = env.vc, env.torch
    n, M = 8, 100_003
    xs = gen("float32", n, M, seed=9)
    d = to_device(torch, xs, "float32", env.dev)
    want = oracle.reduce(xs, "float32", "sum", "ring")
    vc.vc_reduce(d, d[3])  # root 3 reduces into its own input
    vc.vc_broadcast(d[3], d)  # every rank, the root's own buffer included
    torch.cuda.synchronize()
    for r in range(n):
        assert_bits_equal(to_host(d[r], "float32"), want, "float32", f"rank {r}")


def test_prepared_calls_match_direct_calls(env):
    """Prepared handles (checked once, one C call per use) give the same bits
    as the direct calls, on the current stream and on another one."""
    vc, torch = env.vc, env.torch
    n, M = 8, 300_007
    xs = gen("float32", n, M, seed=21)
    d = to_device(torch, xs, "float32", env.dev)
    q = vc.vc_shard_count(M, n)
    y, y2 = [torch.empty_like(t) for t in d], [torch.empty_like(t) for t in d]
    z = [torch.empty(q, device=env.dev) for _ in range(n)]
    g = [torch.empty_like(t) for t in d]
    for order in ORDERS:
        vc.prepare_all_reduce(d, y, order=order)()
        vc.prepare_reduce_scatter(d, z, order=order)()
        vc.prepare_all_gather(z, g)()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        vc.prepare_all_reduce_decomposed(d, [torch.empty_like(t) for t in z], y2,
                                         order=order)(stream=s)
        torch.cuda.synchronize()
        oy = oracle.all_reduce(xs, "float32", "sum", order)
        oz = oracle.reduce_scatter(xs, "float32", "sum", order)
        for r in range(n):
            assert_bits_equal(to_host(y[r], "float32"), oy[r], "float32", "prepared AR")
            assert_bits_equal(to_host(y2[r], "float32"), oy[r], "float32", "prepared dec")
            assert_bits_equal(to_host(g[r], "float32"), oy[r], "float32", "prepared AG")
            assert_bits_equal(to_host(z[r], "float32"), oz[r], "float32", "prepared RS")


def test_prepared_calls_replay_from_a_cuda_graph(env):
    """The collectives only enqueue work on the stream they are given (no
    synchronisation, no allocation), so prepared calls can be captured in a
    CUDA graph and replayed on new inputs written into the same buffers."""
    vc, torch = env.vc, env.torch
    n, M = 8, 200_003
    q = vc.vc_shard_count(M, n)
    d = [torch.empty(M, device=env.dev) for _ in range(n)]
    y = [torch.empty(M, device=env.dev) for _ in range(n)]
    y2 = [torch.empty(M, device=env.dev) for _ in range(n)]
    z = [torch.empty(q, device=env.dev) for _ in range(n)]
    sh = [torch.empty(q, device=env.dev) for _ in range(n)]
    calls = [vc.prepare_all_reduce(d, y, order="ring"),
             vc.prepare_reduce_scatter(d, z, order="recursive_halving"),
             vc.prepare_all_reduce_decomposed(d, sh, y2, order="pairwise_tree")]
    for c in calls:  # first calls outside capture (per-device queries are cached)
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    for seed in (31, 32):
        xs = gen("float32", n, M, seed=seed)
        for t, x in zip(d, xs):
            t.copy_(torch.from_numpy(x))
        g.replay()
        torch.cuda.synchronize()
        oy = oracle.all_reduce(xs, "float32", "sum", "ring")
        oz = oracle.reduce_scatter(xs, "float32", "sum", "recursive_halving")
        ot = oracle.all_reduce(xs, "float32", "sum", "pairwise_tree")
        for r in range(n):
            assert_bits_equal(to_host(y[r], "float32"), oy[r], "float32", "graph AR")
            assert_bits_equal(to_host(z[r], "float32"), oz[r], "float32", "graph RS")
            assert_bits_equal(to_host(y2[r], "float32"), ot[r], "float32", "graph dec")


# ------------------------------------------- the gather's early launch --

@pytest.mark.parametrize("n,M", [(4, 4099), (8, 262_147), (4, 1 << 22), (12, 1_000_003)])
def test_decomposed_back_to_back_matches_fused(env, n, M):
    """The AllGather of a decomposed AllReduce may be scheduled while the
    ReduceScatter before it drains; it must still see every shard element
    that ReduceScatter wrote.  Many decomposed calls back to back on fresh
    inputs (each input written by a torch kernel right before), each
    compared on the device with the fused AllReduce of the same inputs."""
    vc, torch = env.vc, env.torch
    q = vc.vc_shard_count(M, n)
    base = [torch.randn(M, device=env.dev) for _ in range(n)]
    d = [torch.empty_like(t) for t in base]
    y = [torch.empty_like(t) for t in base]
    y2 = [torch.empty_like(t) for t in base]
    sh = [torch.empty(q, device=env.dev) for _ in range(n)]
    ar = vc.prepare_all_reduce(d, y, order="ring")
    dec = vc.prepare_all_reduce_decomposed(d, sh, y2, order="ring")
    bad = torch.zeros((), dtype=torch.int64, device=env.dev)
    for it in range(40):
        for t, b in zip(d, base):
            torch.mul(b, float(it + 1), out=t)
        dec()
        ar()
        for r in range(n):
            bad += (y2[r] != y[0]).sum()
        bad += (y[n - 1] != y[0]).sum()
    torch.cuda.synchronize()
    assert int(bad) == 0
    # and the last call against the oracle
    xs = [to_host(t, "float32") for t in d]
    oy = oracle.all_reduce(xs, "float32", "sum", "ring")
    assert_bits_equal(to_host(y2[0], "float32"), oy[0], "float32", "last decomposed")


def test_all_gather_right_after_a_kernel_that_writes_the_shards(env):
    """AllGather launched directly after a torch kernel that produces the
    shards (a kernel that never signals an early start): it must wait for
    that kernel's writes."""
    vc, torch = env.vc, env.torch
    n, M = 8, 1 << 21
    q = vc.vc_shard_count(M, n)
    src = [torch.randn(q, device=env.dev) for _ in range(n)]
    z = [torch.empty(q, device=env.dev) for _ in range(n)]
    out = [torch.empty(M, device=env.dev) for _ in range(n)]
    ag = vc.prepare_all_gather(z, out)
    bad = torch.zeros((), dtype=torch.int64, device=env.dev)
    for it in range(40):
        for t, s in zip(z, src):
            torch.add(s, float(it), out=t)
        ag()
        want = torch.cat(z)[:M]
        for r in range(n):
            bad += (out[r] != want).sum()
    torch.cuda.synchronize()
    assert int(bad) == 0


# -------------------------------------------------------- maximum sizes --

@pytest.mark.parametrize("n", [3, 9])
def test_more_than_2_31_elements_per_rank(env, n):
    """Element indices past 2^31 (bf16, 2^31 + 13 elements = 4 GiB per rank;
    three ranks take a compile-time ring, nine the run-time-N ring; shards
    off the 16-byte grid): fused AR and RS, sampled indices against the
    oracle (every chunk boundary and the last elements included), all AR
    outputs identical, and RS shard r == AR[rq : rq+q]."""
    vc, torch = env.vc, env.torch
    M = (1 << 31) + 13
    d = []
    for r in range(n):
        g = torch.Generator(device=env.dev)
        g.manual_seed(700 + r)
        d.append(torch.empty(M, dtype=torch.bfloat16, device=env.dev))
        # in 2^28-element slices, to keep the fp32 temporary small
        for lo in range(0, M, 1 << 28):
            hi = min(M, lo + (1 << 28))
            d[r][lo:hi] = torch.randn(hi - lo, generator=g, device=env.dev)
    q = vc.vc_shard_count(M, n)
    y = [torch.empty_like(t) for t in d]
    z = [torch.empty(q, dtype=torch.bfloat16, device=env.dev) for _ in range(n)]
    vc.vc_all_reduce(d, y, op="sum", order="ring")
    vc.vc_reduce_scatter(d, z, op="sum", order="ring")
    torch.cuda.synchronize()
    for r in range(n):
        assert torch.equal(y[r], y[0])
        lo, hi = r * q, min((r + 1) * q, M)
        assert torch.equal(z[r][:hi - lo], y[0][lo:hi])
    _check_sampled(env, d, y[0], z, "bfloat16", "sum", "ring", K=1 << 16, seed=31)
    del d, y, z
    torch.cuda.empty_cache()


def test_concurrent_host_threads(env):
    """Every entry point is thread-safe: four host threads, each on its own
    stream with its own buffers (different N, dtype and order), issue
    collectives at once; every result matches the oracle."""
    import threading
    vc, torch = env.vc, env.torch
    cases = [(4, "float32", "ring"), (6, "bfloat16", "pairwise_tree"),
             (8, "int64", "double_binary_tree"), (12, "float32", "ring")]
    inputs = {k: gen(dt, n, 50_003, seed=600 + k) for k, (n, dt, _) in enumerate(cases)}
    results, errors = {}, []

    def work(k):
        try:
            n, dt, order = cases[k]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                d = to_device(torch, inputs[k], dt, env.dev)
                y = [torch.empty_like(t) for t in d]
                q = vc.vc_shard_count(50_003, n)
                z = [torch.empty(q, dtype=d[0].dtype, device=env.dev) for _ in range(n)]
                for _ in range(20):
                    vc.vc_all_reduce(d, y, op="sum", order=order, stream=s)
                    vc.vc_reduce_scatter(d, z, op="sum", order=order, stream=s)
            s.synchronize()
            results[k] = ([to_host(t, dt) for t in y], [to_host(t, dt) for t in z])
        except Exception as e:  # reported below, on the main thread
            errors.append((k, e))

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k, (n, dt, order) in enumerate(cases):
        oy = oracle.all_reduce(inputs[k], dt, "sum", order)
        oz = oracle.reduce_scatter(inputs[k], dt, "sum", order)
        ys, zs = results[k]
        for r in range(n):
            assert_bits_equal(ys[r], oy[r], dt, f"thread {k} AR rank {r}")
            assert_bits_equal(zs[r], oz[r], dt, f"thread {k} RS rank {r}")
