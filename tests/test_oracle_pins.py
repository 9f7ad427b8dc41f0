"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here needs a GPU.  Each test ties a part of the oracle to something
other than the oracle's own code: values printed on the pages (golden files),
closed forms, hand-derived roundings, literal schedule replays, exact integer
arithmetic, library routines, or invariants.  Several also plant a mistake (a
wrong order, a rolled gather, a zero pad) and check that the comparison used
elsewhere catches it.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from oracle import simulators as sim
import synthetic_inputs as si
from conftest import ints, read_golden

ORDERS = ["ring", "recursive_halving", "pairwise_tree", "double_binary_tree"]
ALL_ORDERS = ORDERS + ["sequential"]
OPS = ["sum", "prod", "max", "min", "avg"]


def _orders_for(n, orders):
    """The orders defined for N ranks: all but recursive halving unless N is a
    power of two."""
    return [o for o in orders if n & (n - 1) == 0 or o != "recursive_halving"]


def lin(n, M, dtype="int64"):
    return si.generate(dtype, "rank_linear", n, M, seed=0)


# ------------------------------------------------------------------ layout --

@pytest.mark.parametrize("order", ALL_ORDERS)
def test_worked_example_sum(order):
    """Four ranks, twenty int64, x = 100r + i: AllReduce = 600 + 4i and the
    printed shards of five ("NCCL 专家课程 07", 一个四 rank 手算例子)."""
    g = read_golden("worked_example_n4_m20_int64.txt")
    n, M = int(g["n"]), int(g["M"])
    xs = lin(n, M)
    expect = np.array(ints(g["allreduce"]), np.int64)
    ys = oracle.all_reduce(xs, "int64", "sum", order)
    for y in ys:
        np.testing.assert_array_equal(y, expect)
    zs = oracle.reduce_scatter(xs, "int64", "sum", order)
    for r in range(n):
        np.testing.assert_array_equal(zs[r], np.array(ints(g[f"shard{r}"]), np.int64))
    # the independent formula the page checks both paths against
    np.testing.assert_array_equal(expect, 600 + 4 * np.arange(M))
    _, ys2 = oracle.all_reduce_decomposed(xs, "int64", "sum", order)
    for y in ys2:
        np.testing.assert_array_equal(y, expect)


@pytest.mark.parametrize("order", ALL_ORDERS)
def test_worked_example_other_ops_closed_forms(order):
    """The same inputs under the other ops: MAX 300 + i, MIN i, PROD the
    product of (100r + i), AVG 150 + i (integer division of 600 + 4i by 4)."""
    n, M = 4, 20
    xs = lin(n, M)
    i = np.arange(M, dtype=np.int64)
    closed = {
        "max": 300 + i,
        "min": i,
        "prod": i * (100 + i) * (200 + i) * (300 + i),
        "avg": 150 + i,
        "sum": 600 + 4 * i,
    }
    for op, expect in closed.items():
        for y in oracle.all_reduce(xs, "int64", op, order):
            np.testing.assert_array_equal(y, expect, err_msg=op)


def test_padding_contract_1003():
    """M = 1003 on four ranks: q = 251, padded to 1004, RS + AG trimmed back
    equals the direct AllReduce ("NCCL 专家课程 07", Contract 实验四)."""
    g = read_golden("padding_m1003_n4.txt")
    n, M = int(g["n"]), int(g["M"])
    assert oracle.shard_count(M, n) == int(g["q"])
    assert oracle.shard_count(M, n) * n == int(g["padded"])
    assert M // n == int(g["unpadded_output"])
    xs = lin(n, M)
    for order in ALL_ORDERS:
        direct = oracle.all_reduce(xs, "int64", "sum", order)
        zs, ys = oracle.all_reduce_decomposed(xs, "int64", "sum", order)
        assert all(z.size == int(g["reducescatter_recvcount"]) for z in zs)
        for y, d in zip(ys, direct):
            assert y.size == int(g["allreduce_count"])
            np.testing.assert_array_equal(y, d)
        # the single padding slot of the last shard holds the identity
        assert zs[-1][-1] == 0


@pytest.mark.parametrize("dtype", ["int32", "int64", "float32", "bfloat16"])
@pytest.mark.parametrize("op", OPS)
def test_padding_tail_is_identity(dtype, op):
    """RS shard positions past M reduce the padding and hold e(op): 0 for SUM
    and AVG, 1 for PROD, the dtype minimum (-inf) for MAX, maximum (+inf) for
    MIN (条件三; MAX is never padded with 0)."""
    n, M = 4, 13  # q = 4, last shard has 3 padding slots
    xs = si.generate(dtype, "uniform_int", n, M, seed=5, lo=-9, hi=9)
    zs = oracle.reduce_scatter(xs, dtype, op, "ring")
    tail = zs[-1][1:]
    e = oracle.identity(dtype, op)
    if dtype in ("float32",):
        want = {"sum": 0.0, "avg": 0.0, "prod": 1.0, "max": -np.inf, "min": np.inf}[op]
        assert e == np.float32(want)
    elif dtype == "bfloat16":
        want = {"sum": 0x0000, "avg": 0x0000, "prod": 0x3F80, "max": 0xFF80, "min": 0x7F80}[op]
        assert int(e) == want
    else:
        info = np.iinfo(np.int32 if dtype == "int32" else np.int64)
        want = {"sum": 0, "avg": 0, "prod": 1, "max": info.min, "min": info.max}[op]
        assert int(e) == want
    np.testing.assert_array_equal(tail, np.full(tail.size, e))


# -------------------------------------------------------- negative checks --

def test_rolled_gather_is_rejected():
    """A gather rolled by one shard differs from the direct AllReduce even
    though every shard is right ("NCCL 专家课程 07", 条件一, Contract 实验二)."""
    n, M = 4, 20
    xs = lin(n, M)
    direct = oracle.all_reduce(xs, "int64", "sum", "ring")[0]
    _, ys = oracle.all_reduce_decomposed(xs, "int64", "sum", "ring")
    wrong = np.roll(ys[0].reshape(n, -1), 1, axis=0).reshape(-1)
    assert not np.array_equal(direct, wrong)
    np.testing.assert_array_equal(direct, ys[0])


def test_wrong_reduction_op_is_rejected():
    """RS(MAX) followed by AG differs from AR(SUM) (条件二, Contract 实验三)."""
    n, M = 4, 20
    xs = lin(n, M)
    direct = oracle.all_reduce(xs, "int64", "sum", "ring")[0]
    zs = oracle.reduce_scatter(xs, "int64", "max", "ring")
    wrong = oracle.all_gather(zs, M, "int64")[0]
    assert not np.array_equal(direct, wrong)


def test_max_with_zero_padding_is_rejected():
    """MAX over all-negative inputs with M % N != 0: padding with 0 instead of
    the identity changes the shard tail and the shard's maximum (条件三)."""
    n, M = 4, 19
    xs = [-(100 * r + np.arange(M, dtype=np.int64)) - 1 for r in range(n)]
    q = oracle.shard_count(M, n)
    good = oracle.reduce_scatter(xs, "int64", "max", "ring")
    # the planted mistake: pad each rank with zeros to N*q and reduce that
    zero_padded = [np.concatenate([x, np.zeros(n * q - M, np.int64)]) for x in xs]
    bad = oracle.reduce_scatter(zero_padded, "int64", "max", "ring")
    assert not np.array_equal(good[-1], bad[-1])
    assert good[-1][-1] == np.iinfo(np.int64).min and bad[-1][-1] == 0
    true_max = max(int(x[(n - 1) * q:].max()) for x in xs)
    assert int(good[-1][: M - (n - 1) * q].max()) == true_max
    assert int(bad[-1].max()) != true_max


# --------------------------------------------------------------- orders ----

def _bits(v):
    return int(np.asarray(v, np.float32).view(np.uint32))


def test_hand_derived_fp32_orders():
    """Each order's fp32 value for operands (1, u, u, u), u = 2^-24, derived by
    hand (golden file): the four orders give three different roundings."""
    g = read_golden("hand_fp32_orders_n4.txt")
    ops = np.array(ints(g["operands"]), np.uint32).view(np.float32)
    n = 4
    # element i of rank s is ops[s]; put the element in every chunk c (q = 1)
    xs = [np.full(n, ops[s], np.float32) for s in range(n)]
    ring = oracle.all_reduce(xs, "float32", "sum", "ring")[0]
    for c in range(n):
        assert _bits(ring[c]) == int(g[f"ring_c{c}"], 0), c
    for order in ("recursive_halving", "pairwise_tree", "sequential"):
        y = oracle.all_reduce(xs, "float32", "sum", order)[0]
        assert all(_bits(v) == int(g[order], 0) for v in y), order
    # double binary tree: elements 0, 1 (first half) tree A, 2, 3 tree B
    y = oracle.all_reduce(xs, "float32", "sum", "double_binary_tree")[0]
    assert [_bits(v) for v in y] == [int(g["pairwise_tree"], 0)] * 2 + \
        [int(g["double_tree_b"], 0)] * 2


def test_ring_schedule_tables_n4():
    """The ring replay reproduces the pages' N=4 tables: chunks sent per step,
    final owners (rank n holds (n+1) mod N), the full-state staircase and
    the AllGather grid."""
    g = read_golden("ring_n4_schedule.txt")
    n = 4
    bufs = [np.arange(n, dtype=np.int64) * 10 + r for r in range(n)]
    chunks, log, contrib = sim.ring_reduce_scatter(bufs, "sum")
    for s in range(n - 1):
        assert log[s] == ints(g[f"rs_step{s + 1}"])
    owners = ints(g["rs_owner"])
    for r in range(n):
        assert owners[r] == (r + 1) % n
        assert contrib[r][owners[r]] == sorted(contrib[r][owners[r]], key=lambda t: (t - owners[r]) % n)
        assert len(contrib[r][owners[r]]) == n
        expect = [[int(t) for t in cell.split(",")] for cell in g[f"state_r{r}"].split("|")]
        assert contrib[r] == expect
    _, aglog, grids = sim.ring_all_gather(chunks)
    for s in range(n - 1):
        assert aglog[s] == ints(g[f"ag_step{s + 1}"])
    for k, step in enumerate((3, 4, 5, 6)):
        rows = g[f"grid_after{step}"].split()
        assert [["#" if h else "." for h in row] for row in grids[k]] == [list(x) for x in rows]


@pytest.mark.parametrize("n", [2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_ring_replay_equals_oracle_fold(n, op):
    """The literal ring replay leaves, at rank (c-1) mod N, a chunk c equal bit
    for bit to the oracle's ring fold (fp32), and AllGather of the replay
    equals the oracle AllReduce."""
    C = 257
    xs = si.generate("float32", "uniform_pm1", n, n * C, seed=11 + n)
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.25) for x in xs]
    chunks, _, _ = sim.ring_reduce_scatter(xs, op)
    fin, _, _ = sim.ring_all_gather(chunks)
    y = oracle.all_reduce(xs, "float32", op, "ring")[0]
    for c in range(n):
        got = chunks[(c - 1) % n][c]
        np.testing.assert_array_equal(got.view(np.uint32), y[c * C:(c + 1) * C].view(np.uint32))
    for r in range(n):
        np.testing.assert_array_equal(np.concatenate(fin[r]).view(np.uint32), y.view(np.uint32))


def test_ring_pin_has_teeth():
    """The planted mistake 'ring = rank-order fold' is caught: for fp32 sums
    the ring and sequential orders differ somewhere at N=8."""
    n, C = 8, 4096
    xs = si.generate("float32", "uniform_pm1", n, n * C, seed=3)
    ring = oracle.all_reduce(xs, "float32", "sum", "ring")[0]
    seq = oracle.all_reduce(xs, "float32", "sum", "sequential")[0]
    assert not np.array_equal(ring.view(np.uint32), seq.view(np.uint32))
    # ...but chunk 0 of the ring starts at rank 0, so there it is the same fold
    np.testing.assert_array_equal(ring[:C].view(np.uint32), seq[:C].view(np.uint32))


def test_ring_primitive_sequence():
    """The NCCL-style primitive replay runs send, (k-2) recvReduceSend,
    recvReduceCopySend, (k-2) recvCopySend, recv = 2k-1 steps, and its
    result equals the oracle's ring AllReduce bit for bit."""
    g = read_golden("ring_primitives_k4.txt")
    k = int(g["k"])
    xs = si.generate("float32", "uniform_pm1", k, k * 64, seed=4)
    outs, names = sim.ring_all_reduce_primitives(xs, "sum")
    assert names == g["sequence"].split()
    y = oracle.all_reduce(xs, "float32", "sum", "ring")[0]
    for o in outs:
        np.testing.assert_array_equal(o.view(np.uint32), y.view(np.uint32))
    for kk in range(2, 9):
        xs = si.generate("float32", "uniform_pm1", kk, kk * 8, seed=kk)
        outs, names = sim.ring_all_reduce_primitives(xs, "sum")
        assert len(names) == 2 * kk - 1
        y = oracle.all_reduce(xs, "float32", "sum", "ring")[0]
        np.testing.assert_array_equal(outs[0].view(np.uint32), y.view(np.uint32))


def test_recursive_halving_pairs_n8():
    """Pairs (0,4)(1,5)(2,6)(3,7), (0,2)(1,3)(4,6)(5,7), (0,1)(2,3)(4,5)(6,7)
    and exchanged sizes M/2, M/4, M/8 ("ReduceScatter" page, N=8 table)."""
    g = read_golden("recursive_halving_n8.txt")
    n, C = 8, 16
    M = n * C
    xs = si.generate("float32", "uniform_pm1", n, M, seed=8)
    chunks, pairs, sizes = sim.recursive_halving_reduce_scatter(xs, "sum")
    for j in range(3):
        expect = [tuple(int(t) for t in p.split("-")) for p in g[f"step{j + 1}"].split()]
        assert pairs[j] == expect
    assert [M // s for s in sizes] == ints(g["size_denominators"])


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_recursive_halving_replay_equals_oracle_fold(n, op):
    """The replay leaves finished chunk r at rank r, equal bit for bit to the
    oracle's recursive-halving fold."""
    C = 33
    xs = si.generate("float32", "uniform_pm1", n, n * C, seed=21 + n)
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.25) for x in xs]
    chunks, pairs, _ = sim.recursive_halving_reduce_scatter(xs, op)
    assert len(pairs) == int(math.log2(n))
    zs = oracle.reduce_scatter(xs, "float32", op, "recursive_halving")
    for r in range(n):
        np.testing.assert_array_equal(chunks[r].view(np.uint32), zs[r].view(np.uint32))


def test_tree_shape_n8():
    """The tree's parent table matches the figure: r0 <- r4 <- {r2, r6},
    r2 <- {r1, r3}, r6 <- {r5, r7}; odd ranks are leaves."""
    g = read_golden("tree_n8_parents.txt")
    expect = ints(g["parents"])
    assert list(oracle.tree_parents(8)) == expect
    assert [sim.tree_parent(r, 8) for r in range(8)] == expect
    leaves = [r for r in range(8) if r not in expect]
    assert leaves == ints(g["leaves"])


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 33, 64])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_tree_replay_equals_oracle_fold(n, op):
    """Reduce-then-broadcast over the tree gives every rank the oracle's
    pairwise_tree value; reduce plus broadcast take 2*log2(N) steps."""
    M = 3 * n + 5
    xs = si.generate("float32", "uniform_pm1", n, M, seed=31 + n)
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.25) for x in xs]
    outs, parents, steps = sim.tree_reduce_broadcast(xs, op)
    assert steps == 2 * math.ceil(math.log2(n)) if n > 1 else steps == 0
    y = oracle.all_reduce(xs, "float32", op, "pairwise_tree")
    for o, yy in zip(outs, y):
        np.testing.assert_array_equal(o.view(np.uint32), yy.view(np.uint32))


@pytest.mark.parametrize("n", [3, 5, 6, 12])
def test_recursive_halving_needs_power_of_two(n):
    """Recursive halving needs N = 2^k ("ReduceScatter" page, algorithm table:
    hypercube).  The ring and both tree orders take any N."""
    xs = si.generate("float32", "uniform_pm1", n, 10, seed=n)
    with pytest.raises(oracle.OracleError):
        oracle.all_reduce(xs, "float32", "sum", "recursive_halving")
    for order in ("ring", "pairwise_tree", "double_binary_tree"):
        oracle.all_reduce(xs, "float32", "sum", order)


# ------------------------------------------------- trees for any rank count --

def _children(parents):
    kids = {r: [] for r in range(len(parents))}
    for r, p in enumerate(parents):
        if p >= 0:
            kids[p].append(r)
    return kids


def _depth(parents, r):
    d = 0
    while parents[r] >= 0:
        r = parents[r]
        d += 1
        assert d <= len(parents), "cycle"
    return d


@pytest.mark.parametrize("n", range(1, 65))
def test_tree_shape_any_n_keeps_the_figures_properties(n):
    """For every N the tree keeps what "通信与互联（01）" 六.1 states of it:
    rank 0 is the root and has a single child, the tree is binary, odd ranks
    are exactly the leaves, a rank's level (lowest set bit) grows towards the
    root, and the depth is ceil(log2 N), so reduce + broadcast take
    2*ceil(log2 N) steps.  A fallback that hung orphans on the root would
    give it several children (N = 6: ranks 4 and 5)."""
    parents = [int(p) for p in oracle.tree_parents(n)]
    assert parents == [sim.tree_parent(r, n) for r in range(n)]
    assert parents[0] == -1
    kids = _children(parents)
    if n == 1:
        return
    assert len(kids[0]) == 1
    assert all(len(k) <= 2 for k in kids.values())
    assert [r for r in range(n) if not kids[r]] == [r for r in range(n) if r % 2 == 1]
    for r in range(1, n):
        p = parents[r]
        assert p == 0 or (p & -p) > (r & -r)
        # in-order labels, as in the figure: a lower child on the left, a
        # higher one on the right
        assert len([c for c in kids[r] if c < r]) <= 1 and len([c for c in kids[r] if c > r]) <= 1
    assert max(_depth(parents, r) for r in range(n)) == math.ceil(math.log2(n))


def test_tree_non_power_of_two_hand_tables():
    g = read_golden("tree_non_pow2.txt")
    for n in (5, 6, 12):
        assert [int(p) for p in oracle.tree_parents(n)] == ints(g[f"parents_{n}"])
    for n in (5, 6):
        assert [sim.tree_b_parent(r, n) for r in range(n)] == ints(g[f"parents_b_{n}"])


def test_tree_non_power_of_two_hand_values():
    """Hand-rounded fp32 sums that tell the tree from the ring, the parent
    fallback r - L from a fallback to the root, and the odd-N mirror tree B
    from a shifted one."""
    g = read_golden("tree_non_pow2.txt")
    for n, keys in ((6, ("tree", "tree_b")), (5, ("tree", "tree_b"))):
        a = [np.float32(v) for v in ints(g[f"n{n}_operands"])]
        xs = [np.array([v, v], np.float32) for v in a]  # M = 2: one element per tree
        y = oracle.all_reduce(xs, "float32", "sum", "pairwise_tree")[0]
        assert _bits(y[0]) == int(g[f"n{n}_tree"], 0)
        d = oracle.all_reduce(xs, "float32", "sum", "double_binary_tree")[0]
        assert [_bits(v) for v in d] == [int(g[f"n{n}_tree"], 0), int(g[f"n{n}_tree_b"], 0)]
    a = [np.float32(v) for v in ints(g["n6_operands"])]
    xs = [np.array([v], np.float32) for v in a]
    assert _bits(oracle.all_reduce(xs, "float32", "sum", "ring")[0][0]) == int(g["n6_ring"], 0)


_PAD = {"sum": 0.0, "prod": 1.0, "max": -np.inf, "min": np.inf}


@pytest.mark.parametrize("n", [3, 5, 6, 7, 9, 12, 17, 24, 33, 63])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_tree_non_power_of_two_is_the_padded_power_of_two_tree(n, op):
    """The tree over N ranks equals, bit for bit, the tree over the next
    power of two P (pinned by the figure) with ranks N..P-1 holding the op's
    identity: a missing rank only passes its one subtree through, and
    x (+) e = x exactly for every finite x other than -0."""
    P = 1 << (n - 1).bit_length()
    M = 37
    xs = si.generate("float32", "uniform_pm1", n, M, seed=400 + n)
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.25) for x in xs]
    pad = [np.full(M, _PAD[op], np.float32) for _ in range(P - n)]
    y = oracle.all_reduce(xs, "float32", op, "pairwise_tree")[0]
    yp = oracle.all_reduce(xs + pad, "float32", op, "pairwise_tree")[0]
    np.testing.assert_array_equal(y.view(np.uint32), yp.view(np.uint32))


@pytest.mark.parametrize("n", [2, 4, 6, 10, 12, 14, 30, 62])
def test_double_tree_even_n_swaps_leaves_and_inner_nodes(n):
    """For even N the shifted second tree makes A's leaves B's inner nodes and
    the reverse ("通信与互联（01）" 六.3), at every even N, not only N = 8."""
    pa = [int(p) for p in oracle.tree_parents(n)]
    pb = [sim.tree_b_parent(r, n) for r in range(n)]
    inner_a = set(p for p in pa if p >= 0)
    leaves_b = set(range(n)) - set(p for p in pb if p >= 0)
    assert inner_a == leaves_b
    assert pb.count(-1) == 1 and pb.index(-1) == 1


def test_step_counts():
    """Ring RS and AG take N-1 steps each and AR 2(N-1) ("NCCL 专家课程 07",
    源码二); recursive halving takes log2 N steps ("ReduceScatter" page)."""
    for n in (2, 3, 4, 8, 16):
        xs = [np.zeros(n, np.int64) for _ in range(n)]
        chunks, log, _ = sim.ring_reduce_scatter(xs)
        _, aglog, _ = sim.ring_all_gather(chunks)
        assert len(log) == n - 1 and len(aglog) == n - 1
        assert len(log) + len(aglog) == 2 * (n - 1)
    for n in (2, 4, 8, 16, 64):
        xs = [np.zeros(n, np.int64) for _ in range(n)]
        _, pairs, _ = sim.recursive_halving_reduce_scatter(xs)
        assert len(pairs) == int(math.log2(n))


# ---------------------------------------------------------- float bounds ----

def _gamma(k):
    u = 2.0 ** -24
    return k * u / (1 - k * u)


@pytest.mark.parametrize("n", [2, 3, 5, 8, 16, 64])
def test_float_sums_within_rounding_bound_of_exact(n):
    """Inputs k*2^-23 - 1 have exact sums computable in int64; every order's
    fp32 result lies within gamma_{N-1} * sum|x| of the exact sum (recursive
    summation bound), and two orders within twice that of each other."""
    M = 4099
    xs = si.generate("float32", "uniform_pm1", n, M, seed=40 + n)
    exact_scaled = sum((x.astype(np.float64) * 2.0 ** 23).astype(np.int64) for x in xs)
    exact = exact_scaled.astype(np.float64) * 2.0 ** -23
    absum = sum(np.abs(x.astype(np.float64)) for x in xs)
    bound = _gamma(n - 1) * absum
    results = {}
    orders = _orders_for(n, ALL_ORDERS)
    for order in orders:
        y = oracle.all_reduce(xs, "float32", "sum", order)[0].astype(np.float64)
        assert np.all(np.abs(y - exact) <= bound), order
        results[order] = y
    for a in results.values():
        for b in results.values():
            assert np.all(np.abs(a - b) <= 2 * bound)


@pytest.mark.parametrize("n", [3, 5, 7, 8, 12])
def test_avg_is_sum_divided_once(n):
    """AVG = the ordered SUM divided by N in one fp32 division (numpy's
    float32 division is the correctly rounded IEEE one); N not a power of two
    separates this from multiplying by a rounded 1/N."""
    M = 4000
    xs = si.generate("float32", "uniform_pm1", n, M, seed=9)
    orders = _orders_for(n, ORDERS)
    for order in orders:
        s = oracle.all_reduce(xs, "float32", "sum", order)[0]
        a = oracle.all_reduce(xs, "float32", "avg", order)[0]
        np.testing.assert_array_equal(a, (s / np.float32(n)).astype(np.float32))


# ---------------------------------------------------------- special cases --

@pytest.mark.parametrize("dtype", ["int32", "int64", "float32", "bfloat16"])
def test_single_rank_is_copy(dtype):
    """N = 1: every op and order returns the input (AVG divides by 1)."""
    x = si.generate(dtype, "uniform_int", 1, 37, seed=1, lo=-50, hi=50)
    for op in OPS:
        for order in ALL_ORDERS:
            y = oracle.all_reduce(x, dtype, op, order)[0]
            np.testing.assert_array_equal(y, x[0])
            z = oracle.reduce_scatter(x, dtype, op, order)[0]
            np.testing.assert_array_equal(z, x[0])


def test_two_ranks_all_orders_equal():
    """N = 2: every order is a single combine, so all agree bitwise."""
    xs = si.generate("float32", "uniform_pm1", 2, 5001, seed=2)
    ref = oracle.all_reduce(xs, "float32", "sum", "sequential")[0]
    for order in ORDERS:
        y = oracle.all_reduce(xs, "float32", "sum", order)[0]
        np.testing.assert_array_equal(y.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n", [4, 8, 64])
def test_small_integer_floats_exact_in_every_order(n):
    """Small-integer-valued floats (|sum| < 2^24) are summed exactly whatever
    the order: every order equals the int64 sum."""
    M = 3001
    xs_i = si.generate("int64", "uniform_int", n, M, seed=n, lo=-1000, hi=1000)
    xs_f = [x.astype(np.float32) for x in xs_i]
    exact = sum(xs_i).astype(np.float32)
    for order in ALL_ORDERS:
        y = oracle.all_reduce(xs_f, "float32", "sum", order)[0]
        np.testing.assert_array_equal(y, exact)


@pytest.mark.parametrize("dtype", ["int32", "int64"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 64])
def test_integer_ops_wraparound_and_order_free(dtype, n):
    """Integer results are the same in every order and equal numpy's
    wrapping reductions; PROD overflows and wraps modulo 2^w."""
    M = 513
    xs = si.generate(dtype, "uniform_int", n, M, seed=60 + n, lo=-100, hi=100)
    wide = np.stack([x.astype(np.int64) for x in xs])
    with np.errstate(over="ignore"):
        expect = {
            "sum": wide.sum(axis=0),
            "prod": wide.prod(axis=0),
            "max": wide.max(axis=0),
            "min": wide.min(axis=0),
            # C division truncates toward zero (no overflow at these sizes)
            "avg": np.trunc(wide.sum(axis=0) / n).astype(np.int64),
        }
    orders = _orders_for(n, ALL_ORDERS)
    for op in OPS:
        outs = [oracle.all_reduce(xs, dtype, op, order)[0] for order in orders]
        for o in outs[1:]:
            np.testing.assert_array_equal(o, outs[0])
        np.testing.assert_array_equal(outs[0], expect[op].astype(outs[0].dtype))


def test_int64_prod_wraps_like_python_modular_arithmetic():
    """PROD of large int64 values wraps modulo 2^64 (checked with Python's
    unbounded integers)."""
    n, M = 16, 64
    xs = si.generate("int64", "uniform_int", n, M, seed=77, lo=-(1 << 40), hi=1 << 40)
    y = oracle.all_reduce(xs, "int64", "prod", "ring")[0]
    for i in range(M):
        p = 1
        for s in range(n):
            p = p * int(xs[s][i])
        p %= 1 << 64
        if p >= 1 << 63:
            p -= 1 << 64
        assert int(y[i]) == p


# -------------------------------------------------------------- invariants --

@pytest.mark.parametrize("dtype", ["int32", "int64", "float32", "bfloat16"])
@pytest.mark.parametrize("order", ORDERS)
def test_allreduce_equals_rs_then_ag(dtype, order):
    """AR == AG(RS(x)) bit for bit in the same order; every rank's AR output
    is identical; RS shard r is AR[rq : rq+q] with identity past M
    ("NCCL 专家课程 07", 数学证明)."""
    n, M = 8, 1001
    if dtype in ("float32", "bfloat16"):
        xs = si.generate(dtype, "uniform_pm1", n, M, seed=5)
    else:
        xs = si.generate(dtype, "uniform_int", n, M, seed=5, lo=-100, hi=100)
    for op in OPS:
        ar = oracle.all_reduce(xs, dtype, op, order)
        zs, dec = oracle.all_reduce_decomposed(xs, dtype, op, order)
        for y in ar[1:]:
            np.testing.assert_array_equal(y, ar[0])
        for y in dec:
            np.testing.assert_array_equal(y, ar[0])
        q = oracle.shard_count(M, n)
        e = oracle.identity(dtype, op) if op != "avg" else np.zeros(1, zs[0].dtype)[0]
        for r in range(n):
            lo, hi = r * q, min(M, (r + 1) * q)
            np.testing.assert_array_equal(zs[r][: hi - lo], ar[0][lo:hi])
            np.testing.assert_array_equal(zs[r][hi - lo:], np.full(q - (hi - lo), e))


def test_reduce_points_matches_full_result():
    """Reducing sampled indices one by one gives the same values as the full
    AllReduce / ReduceScatter (the mode used at full size)."""
    n, M = 8, 10007
    xs = si.generate("float32", "uniform_pm1", n, M, seed=12)
    q = oracle.shard_count(M, n)
    idx = np.array([0, 1, q - 1, q, 2 * q + 3, M - 1, M, n * q - 1], np.int64)
    xs_at = [np.where(idx < M, x[np.minimum(idx, M - 1)], 0).astype(np.float32) for x in xs]
    for order in ORDERS:
        zs = oracle.reduce_scatter(xs, "float32", "sum", order)
        padded = np.concatenate(zs)
        got = oracle.reduce_points(xs_at, idx, n, M, "float32", "sum", order)
        np.testing.assert_array_equal(got.view(np.uint32), padded[idx].view(np.uint32))


# --------------------------------------------------------------- bfloat16 --

def test_bf16_rounding_matches_torch_cpu_rne():
    """The oracle's fp32 -> bf16 rounding equals torch's CPU conversion (a
    round-to-nearest-even library routine) on all 2^32 fp32 bit patterns
    that are not NaN; a NaN stays a NaN."""
    torch = pytest.importorskip("torch")
    step = 1 << 26
    low = np.arange(step, dtype=np.uint32)
    for k in range((1 << 32) // step):
        f = (low + np.uint32(k * step)).view(np.float32)
        ours = oracle.bf16_round(f)
        ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        differ = ours != ref
        if differ.any():  # only NaN payloads may differ
            assert not np.isfinite(f[differ]).any() and not np.isinf(f[differ]).any(), k
            nan_out = ours[differ]
            assert np.all(((nan_out & 0x7F80) == 0x7F80) & ((nan_out & 0x7F) != 0)), k
    nan_in = np.array([0x7FC00000, 0x7F800001, 0xFFFFFFFF, 0x7F80FFFF], np.uint32).view(np.float32)
    nan_out = oracle.bf16_round(nan_in)
    assert np.all(((nan_out & 0x7F80) == 0x7F80) & ((nan_out & 0x7F) != 0))


@pytest.mark.parametrize("order", ORDERS)
def test_bf16_accumulates_in_fp32_and_rounds_once(order):
    """bf16 results equal the fp32 result over the exactly widened operands,
    rounded once to bf16 (torch CPU rounding as the independent rounder)."""
    torch = pytest.importorskip("torch")
    n, M = 8, 20000
    xs = si.generate("bfloat16", "normal", n, M, seed=13, sigma=1e-3)
    wide = [(x.astype(np.uint32) << 16).view(np.float32) for x in xs]
    for op in ("sum", "avg", "max", "min"):
        y16 = oracle.all_reduce(xs, "bfloat16", op, order)[0]
        y32 = oracle.all_reduce(wide, "float32", op, order)[0]
        ref = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy()
        np.testing.assert_array_equal(y16.view(np.int16), ref)


# --------------------------------------------------------- reduce / broadcast --

@pytest.mark.parametrize("order", ALL_ORDERS)
def test_reduce_broadcast_compose_to_allreduce(order):
    """all_reduce = reduce + broadcast ("通信与互联（01）" 二.2), bit for bit in
    the same order; the worked example reduces to 600 + 4i at the root."""
    xs = lin(4, 20)
    y = oracle.reduce(xs, "int64", "sum", order)
    np.testing.assert_array_equal(y, 600 + 4 * np.arange(20))
    for ys in oracle.broadcast(y, 4, "int64"):
        np.testing.assert_array_equal(ys, y)
    n, M = 8, 3001
    xf = si.generate("float32", "uniform_pm1", n, M, seed=17)
    for op in OPS:
        ar = oracle.all_reduce(xf, "float32", op, order)
        out = oracle.broadcast(oracle.reduce(xf, "float32", op, order), n, "float32")
        for a, b in zip(ar, out):
            np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_broadcast_is_a_copy():
    """Every rank receives the root's buffer unchanged (bf16 bits included)."""
    x = si.generate("bfloat16", "normal", 1, 777, seed=4, sigma=3.0)[0]
    for y in oracle.broadcast(x, 5, "bfloat16"):
        np.testing.assert_array_equal(y, x)


# ------------------------------------------------------- double binary tree --

def test_double_tree_shape_n8():
    """Tree B of the figure: root r1 -> r5 -> {r3, r7}, r3 -> {r2, r4},
    r7 -> {r6, r0}; A's inner nodes are B's leaves and the reverse."""
    g = read_golden("double_tree_n8.txt")
    pb = [sim.tree_b_parent(r, 8) for r in range(8)]
    assert pb == ints(g["parents_b"])
    leaves_b = [r for r in range(8) if r not in pb]
    inner_b = sorted(set(p for p in pb if p >= 0) | {pb.index(-1)})
    assert leaves_b == ints(g["leaves_b"]) and inner_b == ints(g["inner_b"])
    pa = list(oracle.tree_parents(8))
    inner_a = sorted(set(p for p in pa if p >= 0))
    assert inner_a == leaves_b


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 33, 64])
@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_double_tree_replay_equals_oracle(n, op):
    """Halves reduced over the tree and the shifted tree, replayed, equal the
    oracle's double_binary_tree fold bit for bit (odd M: the first half is
    the larger)."""
    M = 4 * n + 3
    xs = si.generate("float32", "uniform_pm1", n, M, seed=70 + n)
    if op == "prod":
        xs = [np.float32(1.0) + x * np.float32(0.25) for x in xs]
    outs, _ = sim.double_tree_reduce_broadcast(xs, op)
    y = oracle.all_reduce(xs, "float32", op, "double_binary_tree")
    for o, yy in zip(outs, y):
        np.testing.assert_array_equal(o.view(np.uint32), yy.view(np.uint32))
    h = (M + 1) // 2
    tree = oracle.all_reduce(xs, "float32", op, "pairwise_tree")[0]
    np.testing.assert_array_equal(y[0][:h].view(np.uint32), tree[:h].view(np.uint32))
