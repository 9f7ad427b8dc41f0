"""The C ABI without a GPU: the library loads, exports what the header
declares, and rejects bad arguments before launching anything.

No call here reaches a kernel launch: either validation fails first, or the
launch hook (VC_TEST_FAIL_LAUNCH) turns the launch into VC_ERR_CUDA.  The
fake device pointers below are never dereferenced.
"""
from __future__ import annotations

import re
import subprocess

import pytest

from conftest import ROOT

SUCCESS, INVALID, UNSUPPORTED, ALIAS, CUDA = 0, 1, 2, 3, 4
I32, I64, F32, BF16 = 0, 1, 2, 3
SUM, PROD, MAX, MIN, AVG = 0, 1, 2, 3, 4
RING, RH, TREE, DTREE = 0, 1, 2, 3
MiB = 1 << 20


@pytest.fixture(scope="module")
def vc():
    import __graft_entry__
    __graft_entry__.build()
    import allreduce_reducescatter_allgather_gb300 as pkg
    return pkg


@pytest.fixture(autouse=True)
def no_launch(monkeypatch):
    # any call that passes validation reports a launch failure instead of
    # launching: the pointers here are not real device memory
    monkeypatch.setenv("VC_TEST_FAIL_LAUNCH", "1")


def fake(n, base, stride=16 * MiB):
    return [base + r * stride for r in range(n)]


def table(vc, ptrs):
    from allreduce_reducescatter_allgather_gb300._binding import pointer_table
    return pointer_table(ptrs)


def header_functions():
    text = (ROOT / "include" / "vc.h").read_text()
    return sorted(set(re.findall(r"^\S.*?\b(vc_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = header_functions()
    assert names == sorted(["vc_shard_count", "vc_reduce_scatter", "vc_all_gather",
                            "vc_all_reduce", "vc_all_reduce_decomposed", "vc_reduce",
                            "vc_broadcast", "vc_copy_tiles",
                            "vc_all_reduce_decomposed_noalloc", "vc_bucket_plan",
                            "vc_all_reduce_bucket", "vc_reduce_scatter_bucket",
                            "vc_all_gather_bucket", "vc_status_string"])


def test_library_exports_every_declared_symbol(vc):
    from allreduce_reducescatter_allgather_gb300._binding import EXPORTS, LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", str(LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (vc_\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(vc.lib(), name)
    assert set(EXPORTS) == set(header_functions())


def test_shard_count(vc):
    L = vc.lib()
    assert L.vc_shard_count(20, 4) == 5
    assert L.vc_shard_count(1003, 4) == 251
    assert L.vc_shard_count(1_000_003, 8) == 125_001
    assert L.vc_shard_count(0, 4) == 0
    assert L.vc_shard_count(3, 8) == 1
    assert L.vc_shard_count(10, 0) == 0


def test_status_strings(vc):
    L = vc.lib()
    for code in range(5):
        assert L.vc_status_string(code)
    assert b"unknown" in L.vc_status_string(99)


def rs(vc, send, recv, n, M, dt=F32, op=SUM, order=RING):
    return vc.lib().vc_reduce_scatter(table(vc, send) if send is not None else None,
                                      table(vc, recv) if recv is not None else None,
                                      n, M, dt, op, order, None)


def ar(vc, send, recv, n, M, dt=F32, op=SUM, order=RING):
    return vc.lib().vc_all_reduce(table(vc, send), table(vc, recv), n, M, dt, op, order, None)


def ag(vc, send, recv, n, M, dt=F32):
    return vc.lib().vc_all_gather(table(vc, send), table(vc, recv), n, M, dt, None)


def dec(vc, send, shard, recv, n, M, dt=F32, op=SUM, order=RING):
    return vc.lib().vc_all_reduce_decomposed(table(vc, send), table(vc, shard), table(vc, recv),
                                             n, M, dt, op, order, None)


def test_rank_count_limits(vc):
    for n in (0, -1, 65):
        k = max(n, 1)
        assert rs(vc, fake(k, 1 << 40), fake(k, 2 << 40), n, 1000) == INVALID
        assert ar(vc, fake(k, 1 << 40), fake(k, 2 << 40), n, 1000) == INVALID
    assert ar(vc, fake(64, 1 << 40), fake(64, 2 << 40), 64, 1000) == CUDA  # valid: hook fires


def test_unknown_enums(vc):
    s, r = fake(4, 1 << 40), fake(4, 2 << 40)
    assert rs(vc, s, r, 4, 100, dt=9) == INVALID
    assert rs(vc, s, r, 4, 100, op=5) == INVALID
    assert rs(vc, s, r, 4, 100, order=4) == INVALID
    assert ar(vc, s, r, 4, 100, dt=-1) == INVALID
    assert ag(vc, s, r, 4, 100, dt=7) == INVALID


def test_null_pointers(vc):
    assert rs(vc, None, fake(4, 2 << 40), 4, 100) == INVALID
    assert rs(vc, fake(4, 1 << 40), None, 4, 100) == INVALID
    s = fake(4, 1 << 40)
    s[2] = 0
    assert ar(vc, s, fake(4, 2 << 40), 4, 100) == INVALID
    assert ag(vc, fake(4, 1 << 40), s, 4, 100) == INVALID


def test_count_zero_launches_nothing(vc):
    # succeeds without launching (the launch hook would report CUDA otherwise)
    assert rs(vc, None, None, 4, 0) == SUCCESS
    assert ar(vc, fake(4, 1 << 40), fake(4, 2 << 40), 4, 0) == SUCCESS
    assert ag(vc, fake(4, 1 << 40), fake(4, 2 << 40), 4, 0) == SUCCESS


def test_power_of_two_orders(vc):
    """Recursive halving needs N = 2^k (the hypercube condition on the
    "ReduceScatter" page); the ring and both tree orders take any N."""
    for n in (3, 5, 6, 12, 63):
        s, r = fake(n, 1 << 40), fake(n, 2 << 40)
        assert rs(vc, s, r, n, 1000, order=RH) == UNSUPPORTED
        assert ar(vc, s, r, n, 1000, order=TREE) == CUDA
        assert rs(vc, s, r, n, 1000, order=DTREE) == CUDA
        assert ar(vc, s, r, n, 1000, order=RING) == CUDA
    for n in (1, 2, 4, 8, 16, 32, 64):
        s, r = fake(n, 1 << 40), fake(n, 2 << 40)
        assert ar(vc, s, r, n, 1000, order=RH) == CUDA
        assert rs(vc, s, r, n, 1000, order=TREE) == CUDA
        assert rs(vc, s, r, n, 1000, order=DTREE) == CUDA


def test_alias_rules(vc):
    n, M = 4, 1000
    bytes_m = M * 4
    s = fake(n, 1 << 40)
    # in-place AllReduce per rank is allowed
    assert ar(vc, s, list(s), n, M) == CUDA
    # an output that is another rank's input is not
    r = list(s)
    r[0], r[1] = s[1], s[0]
    assert ar(vc, s, r, n, M) == ALIAS
    # partial overlap with its own input is not
    r = list(s)
    r[2] = s[2] + 4
    assert ar(vc, s, r, n, M) == ALIAS
    # two outputs overlapping each other
    r = fake(n, 2 << 40)
    r[3] = r[2] + bytes_m - 4
    assert ar(vc, s, r, n, M) == ALIAS
    # ReduceScatter output inside an input
    r = fake(n, 2 << 40)
    r[1] = s[0] + 128
    assert rs(vc, s, r, n, M) == ALIAS
    # ReduceScatter output exactly at its own input is not in-place-safe
    assert rs(vc, s, list(s), n, M) == ALIAS
    # AllGather output over a shard
    shards = fake(n, 3 << 40)
    r = fake(n, 2 << 40)
    r[0] = shards[3] - 64
    assert ag(vc, shards, r, n, M) == ALIAS
    # inputs may overlap each other (read only)
    s2 = [s[0]] * n
    assert ar(vc, s2, fake(n, 2 << 40), n, M) == CUDA
    # adjacent but disjoint ranges are fine
    r = [(2 << 40) + k * bytes_m for k in range(n)]
    assert ar(vc, s, r, n, M) == CUDA


def test_decomposed_alias_rules(vc):
    n, M = 4, 1000
    s, z, r = fake(n, 1 << 40), fake(n, 3 << 40), fake(n, 2 << 40)
    assert dec(vc, s, z, r, n, M) == CUDA
    assert dec(vc, s, z, list(s), n, M) == CUDA  # in place
    z2 = list(z)
    z2[1] = r[2] + 16
    assert dec(vc, s, z2, r, n, M) == ALIAS
    z2 = list(z)
    z2[0] = s[0]
    assert dec(vc, s, z2, r, n, M) == ALIAS
    z2 = list(z)
    z2[3] = z2[2]
    assert dec(vc, s, z2, r, n, M) == ALIAS


def test_oversized_count_rejected(vc):
    s, r = fake(2, 1 << 40), fake(2, 2 << 40)
    assert ar(vc, s, r, 2, 1 << 62, dt=I64) == INVALID


def test_launch_failure_surfaces_as_cuda_error(vc):
    s, z, r = fake(4, 1 << 40), fake(4, 3 << 40), fake(4, 2 << 40)
    assert rs(vc, s, z, 4, 100) == CUDA
    assert ag(vc, z, r, 4, 100) == CUDA
    assert ar(vc, s, r, 4, 100) == CUDA
    assert dec(vc, s, z, r, 4, 100) == CUDA


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from allreduce_reducescatter_allgather_gb300 import _binding
    monkeypatch.setattr(_binding, "LIB_PATH", tmp_path / "missing" / "libvc.so")
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="CUDA library missing"):
        _binding.lib()


def test_binding_refuses_host_tensors():
    """Every entry point of the binding refuses tensors in host memory with
    an error before anything runs: there is no CPU path to fall back on."""
    torch = pytest.importorskip("torch")
    import allreduce_reducescatter_allgather_gb300 as vc
    n, M = 4, 10
    q = -(-M // n)
    xs = [torch.zeros(M) for _ in range(n)]
    ys = [torch.zeros(M) for _ in range(n)]
    zs = [torch.zeros(q) for _ in range(n)]
    calls = [
        lambda: vc.vc_all_reduce(xs, ys),
        lambda: vc.vc_all_reduce(xs),
        lambda: vc.vc_reduce_scatter(xs, zs),
        lambda: vc.vc_all_gather(zs, ys),
        lambda: vc.vc_all_reduce_decomposed(xs, zs, ys),
        lambda: vc.vc_all_reduce_decomposed_noalloc(xs, ys),
        lambda: vc.vc_reduce(xs, ys[0]),
        lambda: vc.vc_broadcast(xs[0], ys),
        lambda: vc.prepare_all_reduce(xs, ys),
        lambda: vc.prepare_all_reduce_decomposed(xs, zs, ys),
        lambda: vc.prepare_reduce_scatter(xs, zs),
        lambda: vc.prepare_all_gather(zs, ys),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="not a CUDA tensor"):
            call()
    assert all(torch.count_nonzero(y) == 0 for y in ys)


def test_element_misaligned_pointer_rejected(vc):
    """A buffer not aligned to its element size is rejected on the host (the
    element-wise kernel paths would otherwise access it misaligned)."""
    s, r = fake(4, 1 << 40), fake(4, 2 << 40)
    s[1] += 2
    assert ar(vc, s, r, 4, 100, dt=F32) == INVALID
    assert ar(vc, s, r, 4, 100, dt=BF16) == CUDA  # 2-byte aligned is enough for bf16
    r[0] += 4
    assert rs(vc, fake(4, 1 << 40), r, 4, 100, dt=I64) == INVALID
    assert ag(vc, fake(4, 1 << 40), r, 4, 100, dt=I32) == CUDA


def test_noalloc_checks(vc):
    """The no-allocation AllReduce validates like the others and rejects
    shards that do not fit its static scratch, before touching the GPU."""
    from allreduce_reducescatter_allgather_gb300._binding import NOALLOC_SCRATCH_BYTES
    L = vc.lib()

    def na(send, recv, n, M, dt=F32, op=SUM, order=RING):
        return L.vc_all_reduce_decomposed_noalloc(table(vc, send), table(vc, recv), n, M, dt,
                                                  op, order, None)
    s, r = fake(4, 1 << 40), fake(4, 2 << 40)
    assert na(s, r, 4, NOALLOC_SCRATCH_BYTES // 4 + 1) == INVALID
    assert na(s, r, 4, 0) == SUCCESS
    assert na(s, r, 0, 100) == INVALID
    assert na(s, r, 3, 100, order=RH) == UNSUPPORTED
    r2 = list(r)
    r2[1] = s[2]
    assert na(s, r2, 4, 100) == ALIAS
    assert na(s, list(s), 4, 100) == CUDA  # valid, in place: the launch hook fires


def test_reduce_and_broadcast_checks(vc):
    """Reduce writes one output that may be exactly one input (in place at
    the root); Broadcast's outputs may include the source itself."""
    import ctypes
    L = vc.lib()
    s, r = fake(4, 1 << 40), fake(4, 2 << 40)

    def red(send, out, n=4, M=100, order=RING):
        return L.vc_reduce(table(vc, send), ctypes.c_void_p(out), n, M, F32, SUM, order, None)

    def bc(src, outs, n=4, M=100):
        return L.vc_broadcast(ctypes.c_void_p(src), table(vc, outs), n, M, F32, None)

    assert red(s, r[0]) == CUDA          # valid: the launch hook fires
    assert red(s, s[2]) == CUDA          # in place at the root
    assert red(s, s[2] + 8) == ALIAS     # partial overlap
    assert red(s, 0) == INVALID
    assert red(s, r[0], order=RH, n=3) == UNSUPPORTED
    assert red(s, r[0], M=0) == SUCCESS
    assert bc(s[0], r) == CUDA
    assert bc(s[0], [s[0]] + r[1:]) == CUDA   # root's own buffer included
    r2 = list(r)
    r2[3] = r2[1] + 4
    assert bc(s[0], r2) == ALIAS
    r2 = list(r)
    r2[1] = s[0] + 4
    assert bc(s[0], r2) == ALIAS
    assert bc(0, r) == INVALID


def test_copy_tiles_checks(vc):
    import ctypes
    L = vc.lib()
    assert L.vc_copy_tiles(None, 0, None) == SUCCESS
    assert L.vc_copy_tiles(None, 3, None) == INVALID
    assert L.vc_copy_tiles(ctypes.c_void_p(1 << 40), -1, None) == INVALID
    assert L.vc_copy_tiles(ctypes.c_void_p((1 << 40) + 4), 3, None) == INVALID
    assert L.vc_copy_tiles(ctypes.c_void_p(1 << 40), 3, None) == CUDA  # launch hook


def test_alias_check_agrees_with_pairwise_rule(vc):
    """The O(N log N) overlap check gives the same answer as the plain
    pairwise rule on random layouts (many overlapping, many disjoint)."""
    import random
    rnd = random.Random(7)
    M, es = 100, 4
    nb = M * es

    def pairwise(ins, outs, in_place):
        for r in range(len(outs)):
            for s in range(len(outs)):
                o0, o1 = outs[r], outs[r] + nb
                if s != r and o0 < outs[s] + nb and outs[s] < o1:
                    return ALIAS
                if ins[s] < o1 and o0 < ins[s] + nb:
                    if not (in_place and s == r and ins[s] == outs[r]):
                        return ALIAS
        return CUDA  # valid: the launch hook fires

    seen = {ALIAS: 0, CUDA: 0}
    for trial in range(600):
        n = rnd.choice([1, 2, 3, 4, 8, 17, 64])
        base = 1 << 40
        spread = rnd.choice([2, 40, 400])  # dense layouts collide, sparse ones do not
        slots = [base + 16 * rnd.randrange(0, spread * n) for _ in range(2 * n)]
        if spread == 400 and rnd.random() < 0.5:  # disjoint by construction
            slots = [base + k * (nb + 16 * rnd.randrange(0, 4)) * 2 for k in range(2 * n)]
        ins, outs = slots[:n], slots[n:]
        if rnd.random() < 0.3:  # in place for some ranks
            for r in range(n):
                if rnd.random() < 0.5:
                    outs[r] = ins[r]
        want = pairwise(ins, outs, True)
        seen[want] += 1
        assert ar(vc, ins, outs, n, M) == want, (trial, n)
    assert seen[ALIAS] > 100 and seen[CUDA] > 100, seen
    # ReduceScatter: outputs of q elements against inputs of M, never in place
    for trial in range(200):
        n = rnd.choice([2, 4, 8])
        q = -(-M // n)
        ins = [base + k * nb * 3 for k in range(n)]
        outs = [base + (1 << 30) + k * q * es for k in range(n)]
        if trial % 2:
            r = rnd.randrange(n)
            outs[r] = ins[rnd.randrange(n)] + 16 * rnd.randrange(0, nb // 16)
        want = ALIAS if trial % 2 else CUDA
        assert rs(vc, ins, outs, n, M) == want, trial


# ------------------------------------------------------- fused bucket plan --

def _plan(vc, ins, outs, counts, n, dtype=F32, order=RING, max_tiles=None):
    """vc_bucket_plan on host pointer tables ins[k][r] / outs[k][r]; returns
    (status, tiles, ntiles, bucket_count)."""
    import ctypes
    from allreduce_reducescatter_allgather_gb300._binding import BucketTile
    L = vc.lib()
    flat_in = [ins[k][r] for k in range(len(counts)) for r in range(n)]
    flat_out = [outs[k][r] for k in range(len(counts)) for r in range(n)]
    vpp = ctypes.POINTER(ctypes.c_void_p)
    ti = (ctypes.c_void_p * max(1, len(flat_in)))(*flat_in)
    to = (ctypes.c_void_p * max(1, len(flat_out)))(*flat_out)
    cnt = (ctypes.c_size_t * max(1, len(counts)))(*counts)
    nt, bc = ctypes.c_int(-1), ctypes.c_size_t(0)
    args = (ctypes.cast(ti, vpp), ctypes.cast(to, vpp), cnt, len(counts), n, dtype, order)
    st = L.vc_bucket_plan(*args, None, 0, ctypes.byref(nt), ctypes.byref(bc))
    if st != SUCCESS:
        return st, None, nt.value, bc.value
    cap = nt.value if max_tiles is None else max_tiles
    tiles = (BucketTile * max(1, cap))()
    st = L.vc_bucket_plan(*args, tiles, cap, ctypes.byref(nt), ctypes.byref(bc))
    return st, [tiles[i] for i in range(nt.value)] if st == SUCCESS else None, nt.value, bc.value


def _layout(counts, es):
    """Bucket offsets as the header defines them: each tensor at the end of
    the previous one rounded up to 16 bytes."""
    align, off, base = 16 // es, 0, []
    for c in counts:
        base.append(off)
        off = -(-(off + c) // align) * align
    return base, off


@pytest.mark.parametrize("seed", range(6))
def test_bucket_plan_tiles_partition_the_tensors(vc, seed):
    """Tiles cover every element of every tensor exactly once, in order;
    each sits at the tensor's bucket offset plus its tensor offset; none
    crosses a ring chunk (a multiple of ceil(bucket_count / N)); none is
    larger than 8 KiB; flags bit 0 is set exactly when every rank's input
    and output address of the tile start is 16-byte aligned."""
    import random
    rng = random.Random(seed)
    es = [4, 8, 4, 2][seed % 4]
    dt = {4: F32, 8: I64, 2: BF16}[es] if seed % 4 != 2 else I32
    n = rng.choice([1, 2, 3, 4, 8, 12])
    counts = [rng.choice([0, 1, 3, 7, 100, 4096, 20000, 70001]) for _ in range(rng.randint(1, 9))]
    # one allocation per (tensor, rank): 1 MiB apart; some bases off 16 bytes
    ins = [[(1 << 40) + ((k * n + r) << 22) + es * rng.choice([0, 0, 1]) for r in range(n)]
           for k in range(len(counts))]
    outs = [[(1 << 41) + ((k * n + r) << 22) + es * rng.choice([0, 0, 3]) for r in range(n)]
            for k in range(len(counts))]
    st, tiles, ntiles, bc = _plan(vc, ins, outs, counts, n, dtype=dt)
    assert st == SUCCESS
    base, total = _layout(counts, es)
    assert bc == total
    q = -(-total // n) if total else 1
    seen = {k: 0 for k in range(len(counts))}
    for t in tiles:
        assert t.count > 0 and t.count * es <= 8 << 10   # VC_BUCKET_TILE_MAX_BYTES
        assert t.tensor_offset == seen[t.tensor], "tiles of a tensor follow each other"
        seen[t.tensor] += t.count
        assert t.bucket_offset == base[t.tensor] + t.tensor_offset
        assert t.bucket_offset // q == (t.bucket_offset + t.count - 1) // q, "crosses a chunk"
        aligned = all((ins[t.tensor][r] + t.tensor_offset * es) % 16 == 0 and
                      (outs[t.tensor][r] + t.tensor_offset * es) % 16 == 0 for r in range(n))
        assert bool(t.flags & 1) == aligned
    assert seen == {k: c for k, c in enumerate(counts)}
    assert ntiles == len(tiles)


def test_bucket_plan_realigns_after_a_chunk_split(vc):
    """A tile that starts off the vector grid (after a chunk boundary) is cut
    where the grid resumes, so an aligned tensor's later tiles stay aligned."""
    n, counts = 3, [100, 50_004]   # fp32: total 50_104, q = 16_702 (not a multiple of 4)
    ins = [[(1 << 40) + ((k * n + r) << 22) for r in range(n)] for k in range(2)]
    st, tiles, _, bc = _plan(vc, ins, ins, counts, n)
    assert st == SUCCESS and bc == 50_104
    unaligned = [t for t in tiles if not t.flags & 1]
    # chunk 1 starts at bucket 16_702 = tensor offset 16_602 (2 past the grid):
    # one 2-element tile, then aligned again; chunk 2 starts on the grid
    assert [(t.tensor_offset, t.count) for t in unaligned] == [(16_602, 2)]


def test_bucket_plan_rules(vc):
    n = 4
    ins = [fake(n, (1 << 40) + k * (1 << 30)) for k in range(2)]
    outs = [fake(n, (1 << 42) + k * (1 << 30)) for k in range(2)]
    counts = [1000, 333]
    assert _plan(vc, ins, outs, counts, n)[0] == SUCCESS
    assert _plan(vc, ins, ins, counts, n)[0] == SUCCESS                 # in place
    # floats: ring only; integers: every order (RH needs a power of two)
    assert _plan(vc, ins, outs, counts, n, order=TREE)[0] == UNSUPPORTED
    assert _plan(vc, ins, outs, counts, n, dtype=I64, order=DTREE)[0] == SUCCESS
    assert _plan(vc, [i[:3] for i in ins], [o[:3] for o in outs], counts, 3, dtype=I32,
                 order=RH)[0] == UNSUPPORTED
    # aliasing: two outputs overlap; an input overlaps another tensor's
    # output; an input overlaps its own output but not exactly
    bad = [list(o) for o in outs]
    bad[1][2] = outs[0][2] + 400
    assert _plan(vc, ins, bad, counts, n)[0] == ALIAS
    bad = [list(o) for o in outs]
    bad[1][0] = ins[0][0] + 64
    assert _plan(vc, ins, bad, counts, n)[0] == ALIAS
    bad = [list(i) for i in ins]
    bad[0][1] = ins[0][1] + 16
    assert _plan(vc, ins, bad, counts, n)[0] == ALIAS
    # null or misaligned pointers of non-empty tensors; empty ones are ignored
    bad = [list(i) for i in ins]
    bad[1][3] = 0
    assert _plan(vc, bad, outs, counts, n)[0] == INVALID
    assert _plan(vc, bad, outs, [1000, 0], n)[0] == SUCCESS
    bad[1][3] = ins[1][3] + 2
    assert _plan(vc, bad, outs, counts, n)[0] == INVALID
    # too few tiles: error, with the needed count reported
    st, _, ntiles, _ = _plan(vc, ins, outs, counts, n, max_tiles=1)
    assert st == INVALID and ntiles >= 2


def test_all_reduce_bucket_checks(vc):
    L = vc.lib()
    assert L.vc_all_reduce_bucket(None, 0, None, None, 4, 100, F32, SUM, None) == SUCCESS
    assert L.vc_all_reduce_bucket(1 << 40, 5, 1 << 41, 1 << 42, 4, 100, F32, 9, None) == INVALID
    assert L.vc_all_reduce_bucket(1 << 40, 5, 1 << 41, 1 << 42, 0, 100, F32, SUM, None) == INVALID
    assert L.vc_all_reduce_bucket((1 << 40) + 4, 5, 1 << 41, 1 << 42, 4, 100, F32, SUM,
                                  None) == INVALID
    assert L.vc_all_reduce_bucket(1 << 40, 5, 1 << 41, 1 << 42, 4, 100, F32, SUM, None) == CUDA


def test_reduce_scatter_bucket_checks(vc):
    L = vc.lib()
    shards = fake(4, 1 << 43)
    t = table(vc, shards)
    assert L.vc_reduce_scatter_bucket(None, 0, None, None, 4, 100, F32, SUM, None) == SUCCESS
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, t, 4, 100, F32, 9, None) == INVALID
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, None, 4, 100, F32, SUM, None) == INVALID
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, t, 4, 0, F32, SUM, None) == INVALID
    bad = list(shards)
    bad[2] = 0
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, table(vc, bad), 4, 100, F32, SUM,
                                      None) == INVALID
    bad[2] = shards[1] + 40   # q = 25 fp32 = 100 bytes: overlaps shard 1
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, table(vc, bad), 4, 100, F32, SUM,
                                      None) == ALIAS
    assert L.vc_reduce_scatter_bucket(1 << 40, 5, 1 << 41, t, 4, 100, F32, SUM, None) == CUDA


def test_all_gather_bucket_checks(vc):
    L = vc.lib()
    t = table(vc, fake(4, 1 << 43))
    assert L.vc_all_gather_bucket(None, 0, None, None, 4, 100, F32, None) == SUCCESS
    assert L.vc_all_gather_bucket(1 << 40, 5, t, 1 << 42, 4, 100, 7, None) == INVALID
    assert L.vc_all_gather_bucket(1 << 40, 5, None, 1 << 42, 4, 100, F32, None) == INVALID
    assert L.vc_all_gather_bucket(1 << 40, 5, t, 1 << 42, 65, 100, F32, None) == INVALID
    assert L.vc_all_gather_bucket(1 << 40, 5, table(vc, [1 << 43, 0, 1 << 44, 1 << 45]),
                                  1 << 42, 4, 100, F32, None) == INVALID
    assert L.vc_all_gather_bucket(1 << 40, 5, t, 1 << 42, 4, 100, F32, None) == CUDA
