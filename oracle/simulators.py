"""Step-by-step replays of the schedules the pages describe, on host arrays.

TEST INFRASTRUCTURE (part of the oracle; same import rule as the package).

Each simulator keeps N per-rank buffers and moves chunks between them exactly
as the schedule says, one step at a time, recording who sends what to whom.
They exist to pin the reduction orders of ``vc_oracle.c``: the value each
simulator leaves in a rank's buffer must equal, bit for bit, the closed-form
fold the oracle computes for that order, and the recorded schedule must match
the tables printed on the pages.

Sources (page title, section):
 - ring ReduceScatter / AllGather: "Ring AllReduce 核心流程" (N=4 step table and
   the ring pseudocode: at ReduceScatter step s a rank sends chunk
   (rank - s) mod N to its right neighbour and adds the chunk
   (rank - 1 - s) mod N it receives into its own copy; at AllGather step s it
   forwards chunk (rank + 1 - s) mod N and overwrites chunk (rank - s) mod N),
   "通信与互联（01）" 五.2 / 五.3 (full-state staircase and the AllGather grid);
 - NCCL ring AllReduce primitives: "NCCL 专家课程 07" 源码三 and "为什么说
   AllReduce = ReduceScatter + AllGather" sections 8-10 (send, k-2 x
   recvReduceSend, recvReduceCopySend, k-2 x recvCopySend, recv);
 - recursive halving: "ReduceScatter" page, Recursive Halving table (N=8);
 - binary tree reduce + broadcast: "通信与互联（01）" 六.1 figure.

Arithmetic is numpy elementwise on float32 or int64 arrays, so every float
operation is one IEEE single operation and integers wrap modulo 2^64.
"""
from __future__ import annotations

import numpy as np

_UFUNC = {
    "sum": np.add,
    "avg": np.add,
    "prod": np.multiply,
}


def combine(op: str, own, received):
    """own (+) received, elementwise.  MAX/MIN keep ``own`` on ties."""
    if op in _UFUNC:
        with np.errstate(over="ignore", invalid="ignore"):
            return _UFUNC[op](own, received)
    if op == "max":
        return np.where(received > own, received, own)
    if op == "min":
        return np.where(received < own, received, own)
    raise ValueError(op)


def _split(buf, n):
    assert buf.size % n == 0, "simulators take buffers already padded to N*q"
    return [c.copy() for c in np.split(buf, n)]


# ---------------------------------------------------------------- ring ----

def ring_reduce_scatter(bufs, op: str = "sum"):
    """Ring ReduceScatter over N buffers of N*C elements.

    Returns (chunks, log, contrib): chunks[r][c] is rank r's copy of chunk c
    after N-1 steps; log[s][r] is the chunk rank r sent at step s (0-based)
    to rank (r+1) mod N; contrib[r][c] lists, in the order they were added,
    the ranks whose operands rank r's copy of chunk c contains.
    """
    n = len(bufs)
    chunks = [_split(np.asarray(b), n) for b in bufs]
    contrib = [[[r] for _c in range(n)] for r in range(n)]
    log = []
    for step in range(n - 1):
        # every rank sends at once: snapshot the messages first
        sent = [(r - step) % n for r in range(n)]
        msgs = [(chunks[r][sent[r]].copy(), list(contrib[r][sent[r]])) for r in range(n)]
        log.append(sent)
        for r in range(n):
            src = (r - 1) % n
            recv = (r - 1 - step) % n
            assert recv == sent[src]
            part, who = msgs[src]
            chunks[r][recv] = combine(op, chunks[r][recv], part)
            contrib[r][recv] = who + [r]
    return chunks, log, contrib


def ring_all_gather(chunks):
    """Ring AllGather continuing from the ReduceScatter state, in which rank r
    holds the finished chunk (r+1) mod N.  Returns (chunks, log, grids):
    grids[s][r][c] is True once rank r holds the finished chunk c, starting
    with the state before the first AllGather step."""
    n = len(chunks)
    chunks = [[c.copy() for c in row] for row in chunks]
    have = [[c == (r + 1) % n for c in range(n)] for r in range(n)]
    grids = [[row[:] for row in have]]
    log = []
    for step in range(n - 1):
        sent = [(r + 1 - step) % n for r in range(n)]
        msgs = [chunks[r][sent[r]].copy() for r in range(n)]
        log.append(sent)
        for r in range(n):
            src = (r - 1) % n
            recv = (r - step) % n
            assert recv == sent[src] and have[src][recv]
            chunks[r][recv] = msgs[src]
            have[r][recv] = True
        grids.append([row[:] for row in have])
    return chunks, log, grids


def ring_all_reduce_primitives(bufs, op: str = "sum"):
    """Ring AllReduce as the per-chunk primitive sequence of a NCCL-style ring
    (k ranks): send; k-2 x recvReduceSend; recvReduceCopySend (the last
    reduction, written to the output and forwarded in one primitive); k-2 x
    recvCopySend; recv.  Returns (outputs, primitive names of rank 0)."""
    n = len(bufs)
    chunks = [_split(np.asarray(b), n) for b in bufs]
    out = [[None] * n for _ in range(n)]
    names = []
    # The chunk rank r starts with at primitive step t is (r - t) mod n; what
    # travels is the partial sum, then the finished chunk.
    inflight = [None] * n
    for t in range(2 * n - 1):
        new = [None] * n
        for r in range(n):
            c = (r - t) % n
            src = (r - 1) % n
            if t == 0:
                prim = "send"
                new[r] = chunks[r][c].copy()
            elif t < n - 1:
                prim = "recvReduceSend"
                new[r] = combine(op, chunks[r][c], inflight[src])
            elif t == n - 1:
                prim = "recvReduceCopySend"
                fin = combine(op, chunks[r][c], inflight[src])
                out[r][c] = fin
                new[r] = fin
            elif t < 2 * n - 2:
                prim = "recvCopySend"
                out[r][c] = inflight[src].copy()
                new[r] = inflight[src].copy()
            else:
                prim = "recv"
                out[r][c] = inflight[src].copy()
            if r == 0:
                names.append(prim)
        inflight = new
    return [np.concatenate(row) for row in out], names


# --------------------------------------------------- recursive halving ----

def recursive_halving_reduce_scatter(bufs, op: str = "sum"):
    """Recursive-halving ReduceScatter over N = 2^k buffers of N*C elements.

    At step j (1-based) rank s pairs with s XOR N/2^j; the lower rank of the
    pair keeps the lower half of the chunk range both currently hold and sends
    the upper half, the upper rank the reverse; each adds what it receives
    into the half it keeps.  Returns (chunks, pairs, sizes): chunks[s] is the
    finished chunk s left at rank s; pairs[j] the sorted pairs of step j;
    sizes[j] the elements each rank sent at step j.
    """
    n = len(bufs)
    assert n & (n - 1) == 0, "recursive halving needs N = 2^k"
    total = np.asarray(bufs[0]).size
    data = [np.asarray(b).copy() for b in bufs]
    lo = [0] * n
    hi = [total] * n
    pairs, sizes = [], []
    d = n // 2
    while d >= 1:
        step_pairs = sorted({(min(s, s ^ d), max(s, s ^ d)) for s in range(n)})
        pairs.append(step_pairs)
        new = [x.copy() for x in data]
        sent = None
        for s in range(n):
            p = s ^ d
            assert (lo[s], hi[s]) == (lo[p], hi[p])
            mid = (lo[s] + hi[s]) // 2
            keep = (lo[s], mid) if s < p else (mid, hi[s])
            a, b = keep
            new[s][a:b] = combine(op, data[s][a:b], data[p][a:b])
            sent = (hi[s] - lo[s]) - (b - a)
        for s in range(n):
            mid = (lo[s] + hi[s]) // 2
            if s < (s ^ d):
                hi[s] = mid
            else:
                lo[s] = mid
        data = new
        sizes.append(sent)
        d //= 2
    chunks = [data[s][lo[s]:hi[s]].copy() for s in range(n)]
    return chunks, pairs, sizes


# ---------------------------------------------------------------- tree ----

def tree_parent(r: int, n: int) -> int:
    """Parent of rank r in the tree of the figure: rank r's level is its lowest
    set bit L; its parent is (r - L) | 2L.  When that label is not a rank
    (>= N) the parent is r - L: for N = 2^k only rank N/2 is in that case,
    and it hangs under rank 0, the root with a single child."""
    if r == 0:
        return -1
    low = r & -r
    p = (r - low) | (low << 1)
    return p if p < n else r - low


def tree_reduce_broadcast(bufs, op: str = "sum"):
    """Reduce up the tree, then broadcast down.  In each round every node whose
    children have all reported combines them (lower rank first), adds its own
    operand and sends the result to its parent; the root's result then flows
    back down one level per round.  Returns (outputs, parents, rounds)."""
    n = len(bufs)
    data = [np.asarray(b).copy() for b in bufs]
    parents = [tree_parent(r, n) for r in range(n)]
    children = {p: [r for r in range(n) if parents[r] == p] for p in range(n)}
    done = {}
    rounds = 0
    while 0 not in done:
        ready = [p for p in range(n) if p not in done and all(c in done for c in children[p])]
        for p in ready:
            kids = children[p]
            if kids:
                acc = done[kids[0]]
                for c in kids[1:]:
                    acc = combine(op, acc, done[c])
                done[p] = combine(op, acc, data[p])
            else:
                done[p] = data[p]
        rounds += 1
    # the leaves "send" in round 1; the root finishes in the last round
    reduce_rounds = rounds - 1
    result = done[0]
    have = {0}
    bcast_rounds = 0
    while len(have) < n:
        have |= {r for r in range(n) if parents[r] in have}
        bcast_rounds += 1
    return [result.copy() for _ in range(n)], parents, reduce_rounds + bcast_rounds


def tree_b_node(k: int, n: int) -> int:
    """The rank that plays node k of the first tree in the second one: k + 1
    mod n for even n (the rank numbers shifted by one), n - 1 - k for odd n
    (the mirror image)."""
    return (k + 1) % n if n % 2 == 0 else n - 1 - k


def tree_b_parent(r: int, n: int) -> int:
    """Parent of rank r in the second tree of a double binary tree."""
    k = next(k for k in range(n) if tree_b_node(k, n) == r)
    p = tree_parent(k, n)
    return -1 if p == -1 else tree_b_node(p, n)


def double_tree_reduce_broadcast(bufs, op: str = "sum"):
    """Each rank's buffer is cut in two halves (the first ceil(M/2)
    elements, the rest); the first half is reduced and broadcast over the
    tree, the second over tree B.  Returns (outputs, parents of tree B)."""
    n = len(bufs)
    M = np.asarray(bufs[0]).size
    h = (M + 1) // 2
    first = [np.asarray(b)[:h] for b in bufs]
    # tree B: node k of the plain tree is played by rank tree_b_node(k)
    second = [np.asarray(bufs[tree_b_node(k, n)])[h:] for k in range(n)]
    out_a, _, _ = tree_reduce_broadcast(first, op)
    out_b, _, _ = tree_reduce_broadcast(second, op)
    outs = [np.concatenate([out_a[r], out_b[r]]) for r in range(n)]
    return outs, [tree_b_parent(r, n) for r in range(n)]
