"""Plain CPU oracle for AllReduce / ReduceScatter / AllGather over N virtual ranks.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (its ``cpu_baseline`` and ``--impl reference``) may import
this package.  The CUDA library never imports, links or calls it, and this
package imports nothing of the CUDA library: the two share no code.

The arithmetic lives in ``vc_oracle.c`` (plain C, one element at a time, see
its header for the passages it follows).  This module only loads the compiled
library with ctypes and moves numpy arrays in and out.  ``simulators.py`` holds
literal step-by-step replays of the pages' ring, recursive-halving and tree
schedules, used to pin the orders the C code folds in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "vc_oracle.c"
_LIB = _HERE / "liboracle.so"

# Enumerations of the oracle (its own numbering; mapped from names below).
DTYPES = {"int32": 0, "int64": 1, "float32": 2, "bfloat16": 3}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3, "avg": 4}
ORDERS = {"ring": 0, "recursive_halving": 1, "pairwise_tree": 2, "sequential": 3,
          "double_binary_tree": 4}

# numpy storage type of each dtype (bfloat16 is carried as its raw uint16 bits)
NP_STORAGE = {"int32": np.int32, "int64": np.int64, "float32": np.float32,
              "bfloat16": np.uint16}

_ERRORS = {-1: "bad argument", -2: "unsupported (recursive halving needs N = 2^k)",
           -3: "no memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> Path:
    """Compile vc_oracle.c into liboracle.so with gcc (no fast-math, no FMA
    contraction, so every float operation is one IEEE single operation)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    tmp = _LIB.with_suffix(f".so.tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(_LIB))
        vpp = ctypes.POINTER(ctypes.c_void_p)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.oracle_shard_count.argtypes = [i64, i32]
        L.oracle_shard_count.restype = i64
        L.oracle_identity.argtypes = [i32, i32, ctypes.c_void_p]
        L.oracle_reduce_scatter.argtypes = [vpp, vpp, i32, i64, i32, i32, i32]
        L.oracle_all_gather.argtypes = [vpp, vpp, i32, i64, i32]
        L.oracle_all_reduce.argtypes = [vpp, vpp, i32, i64, i32, i32, i32]
        L.oracle_all_reduce_decomposed.argtypes = [vpp, vpp, vpp, i32, i64, i32, i32, i32]
        L.oracle_reduce_points.argtypes = [vpp, ctypes.c_void_p, i64, i32, i64, i32, i32, i32,
                                           ctypes.c_void_p]
        L.oracle_reduce.argtypes = [vpp, ctypes.c_void_p, i32, i64, i32, i32, i32]
        L.oracle_broadcast.argtypes = [ctypes.c_void_p, vpp, i32, i64, i32]
        L.oracle_bf16_round.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64]
        L.oracle_bf16_round.restype = None
        L.oracle_tree_parents.argtypes = [i32, ctypes.c_void_p]
        for f in ("oracle_identity", "oracle_reduce_scatter", "oracle_all_gather",
                  "oracle_all_reduce", "oracle_all_reduce_decomposed",
                  "oracle_reduce_points", "oracle_tree_parents", "oracle_reduce",
                  "oracle_broadcast"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"error {rc}"))


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))


def _as_inputs(xs, dtype):
    st = NP_STORAGE[dtype]
    out = []
    for x in xs:
        a = np.ascontiguousarray(x)
        if a.dtype != st:
            raise TypeError(f"expected {np.dtype(st)} storage for {dtype}, got {a.dtype}")
        out.append(a)
    return out


def shard_count(M: int, n: int) -> int:
    """q = ceil(M / N)."""
    return int(lib().oracle_shard_count(M, n))


def identity(dtype: str, op: str):
    """The padding value e(op, dtype) as a 0-d numpy value of the storage type."""
    out = np.zeros(1, NP_STORAGE[dtype])
    _check(lib().oracle_identity(DTYPES[dtype], OPS[op], out.ctypes.data))
    return out[0]


def reduce_scatter(xs, dtype: str, op: str, order: str):
    """z[r][j] = reduction over s of x[s][r*q + j], j < q (identity padding)."""
    xs = _as_inputs(xs, dtype)
    n, M = len(xs), (xs[0].size if xs else 0)
    q = shard_count(M, n)
    zs = [np.empty(q, NP_STORAGE[dtype]) for _ in range(n)]
    _check(lib().oracle_reduce_scatter(_ptrs(xs), _ptrs(zs), n, M, DTYPES[dtype], OPS[op],
                                       ORDERS[order]))
    return zs


def all_gather(zs, M: int, dtype: str):
    """y[r][s*q + j] = z[s][j] for every r, trimmed to M."""
    zs = _as_inputs(zs, dtype)
    n = len(zs)
    ys = [np.empty(M, NP_STORAGE[dtype]) for _ in range(n)]
    _check(lib().oracle_all_gather(_ptrs(zs), _ptrs(ys), n, M, DTYPES[dtype]))
    return ys


def _outputs(out, n, count, dtype):
    """Caller-supplied output arrays (checked), or new ones."""
    if out is None:
        return [np.empty(count, NP_STORAGE[dtype]) for _ in range(n)]
    if len(out) != n or any(o.dtype != NP_STORAGE[dtype] or o.size != count
                            or not o.flags.c_contiguous for o in out):
        raise TypeError("output arrays do not match")
    return out


def all_reduce(xs, dtype: str, op: str, order: str, out=None):
    """y[r][i] = reduction over s of x[s][i], identical for every r.  `out`:
    optional preallocated outputs (N arrays of M)."""
    xs = _as_inputs(xs, dtype)
    n, M = len(xs), xs[0].size
    ys = _outputs(out, n, M, dtype)
    _check(lib().oracle_all_reduce(_ptrs(xs), _ptrs(ys), n, M, DTYPES[dtype], OPS[op],
                                   ORDERS[order]))
    return ys


def all_reduce_decomposed(xs, dtype: str, op: str, order: str, shards=None, out=None):
    """ReduceScatter into N shards of q, then AllGather; returns (shards,
    outputs).  `shards`, `out`: optional preallocated arrays."""
    xs = _as_inputs(xs, dtype)
    n, M = len(xs), xs[0].size
    q = shard_count(M, n)
    zs = _outputs(shards, n, q, dtype)
    ys = _outputs(out, n, M, dtype)
    _check(lib().oracle_all_reduce_decomposed(_ptrs(xs), _ptrs(zs), _ptrs(ys), n, M,
                                              DTYPES[dtype], OPS[op], ORDERS[order]))
    return zs, ys


def reduce(xs, dtype: str, op: str, order: str):
    """The AllReduce value, written once (the root's buffer)."""
    xs = _as_inputs(xs, dtype)
    n, M = len(xs), xs[0].size
    y = np.empty(M, NP_STORAGE[dtype])
    _check(lib().oracle_reduce(_ptrs(xs), y.ctypes.data, n, M, DTYPES[dtype], OPS[op],
                               ORDERS[order]))
    return y


def broadcast(x, n: int, dtype: str):
    """N copies of the root's buffer."""
    x = _as_inputs([x], dtype)[0]
    ys = [np.empty(x.size, NP_STORAGE[dtype]) for _ in range(n)]
    _check(lib().oracle_broadcast(x.ctypes.data, _ptrs(ys), n, x.size, DTYPES[dtype]))
    return ys


def reduce_points(xs_at, idx, n: int, M: int, dtype: str, op: str, order: str):
    """Reduce only the global indices idx; xs_at[s][k] is rank s's operand at
    idx[k] (ignored, and replaced by the identity, where idx[k] >= M)."""
    xs_at = _as_inputs(xs_at, dtype)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    K = idx.size
    out = np.empty(K, NP_STORAGE[dtype])
    _check(lib().oracle_reduce_points(_ptrs(xs_at), idx.ctypes.data, K, n, M, DTYPES[dtype],
                                      OPS[op], ORDERS[order], out.ctypes.data))
    return out


def bf16_round(f32):
    """fp32 -> bf16 bits, round to nearest even (the oracle's own rounding)."""
    a = np.ascontiguousarray(f32, dtype=np.float32)
    out = np.empty(a.size, np.uint16)
    lib().oracle_bf16_round(a.ctypes.data, out.ctypes.data, a.size)
    return out.reshape(a.shape)


def tree_parents(n: int):
    """parent[r] of the tree order for ranks 0..N-1 (-1 for the root)."""
    out = np.empty(n, np.int32)
    _check(lib().oracle_tree_parents(n, out.ctypes.data))
    return out
