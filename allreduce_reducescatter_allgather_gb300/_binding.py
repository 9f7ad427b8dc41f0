"""ctypes binding of the C ABI in include/vc.h.

Argument marshalling only: torch tensors in, device pointers and the current
CUDA stream out to libvc.so.  Every step of the collectives runs in the CUDA
kernels; if the library is missing, importing this module succeeds but every
call raises (there is no CPU fallback).

The tensor-level checks mirror PyTorch's capacity check before a collective
("NCCL 专家课程 07", 源码五: the input must hold world_size times the output
for ReduceScatter) and raise ValueError before anything reaches the library;
the library repeats its own pointer-level checks.
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Sequence

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_lib" / "libvc.so"

DTYPES = {"int32": 0, "int64": 1, "float32": 2, "bfloat16": 3}
OPS = {"sum": 0, "prod": 1, "max": 2, "min": 3, "avg": 4}
ORDERS = {"ring": 0, "recursive_halving": 1, "pairwise_tree": 2, "double_binary_tree": 3}
STATUS = {0: "VC_SUCCESS", 1: "VC_ERR_INVALID_ARGUMENT", 2: "VC_ERR_UNSUPPORTED",
          3: "VC_ERR_ALIAS", 4: "VC_ERR_CUDA"}
MAX_RANKS = 64

# Every function the header declares (checked by the tests against vc.h).
EXPORTS = ("vc_shard_count", "vc_reduce_scatter", "vc_all_gather", "vc_all_reduce",
           "vc_all_reduce_decomposed", "vc_reduce", "vc_broadcast", "vc_copy_tiles",
           "vc_all_reduce_decomposed_noalloc", "vc_bucket_plan", "vc_all_reduce_bucket",
           "vc_reduce_scatter_bucket", "vc_all_gather_bucket", "vc_status_string")


class BucketTile(ctypes.Structure):
    """vc_bucket_tile_t."""
    _fields_ = [("bucket_offset", ctypes.c_longlong), ("tensor_offset", ctypes.c_longlong),
                ("count", ctypes.c_longlong), ("tensor", ctypes.c_int), ("flags", ctypes.c_int)]


class VcError(RuntimeError):
    """A non-zero vc_status_t from the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libvc.so with its prototypes set; raises if it was not built."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(
                f"CUDA library missing ({LIB_PATH}); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(str(LIB_PATH))
        vpp = ctypes.POINTER(ctypes.c_void_p)
        i32, sz, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        L.vc_shard_count.argtypes = [sz, i32]
        L.vc_shard_count.restype = sz
        L.vc_reduce_scatter.argtypes = [vpp, vpp, i32, sz, i32, i32, i32, vp]
        L.vc_all_gather.argtypes = [vpp, vpp, i32, sz, i32, vp]
        L.vc_all_reduce.argtypes = [vpp, vpp, i32, sz, i32, i32, i32, vp]
        L.vc_all_reduce_decomposed.argtypes = [vpp, vpp, vpp, i32, sz, i32, i32, i32, vp]
        L.vc_reduce.argtypes = [vpp, vp, i32, sz, i32, i32, i32, vp]
        L.vc_broadcast.argtypes = [vp, vpp, i32, sz, i32, vp]
        L.vc_copy_tiles.argtypes = [vp, i32, vp]
        L.vc_bucket_plan.argtypes = [vpp, vpp, ctypes.POINTER(sz), i32, i32, i32, i32,
                                     ctypes.POINTER(BucketTile), i32, ctypes.POINTER(i32),
                                     ctypes.POINTER(sz)]
        L.vc_all_reduce_bucket.argtypes = [vp, i32, vp, vp, i32, sz, i32, i32, vp]
        L.vc_reduce_scatter_bucket.argtypes = [vp, i32, vp, vpp, i32, sz, i32, i32, vp]
        L.vc_all_gather_bucket.argtypes = [vp, i32, vpp, vp, i32, sz, i32, vp]
        L.vc_all_gather_bucket.restype = i32
        L.vc_bucket_plan.restype = i32
        L.vc_all_reduce_bucket.restype = i32
        L.vc_reduce_scatter_bucket.restype = i32
        for f in ("vc_reduce_scatter", "vc_all_gather", "vc_all_reduce",
                  "vc_all_reduce_decomposed", "vc_reduce", "vc_broadcast", "vc_copy_tiles"):
            getattr(L, f).restype = i32
        L.vc_status_string.argtypes = [i32]
        L.vc_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def pointer_table(ptrs: Sequence[int]):
    """A C array of device pointers (ints) as void**."""
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))


def check_status(status: int):
    if status != 0:
        msg = lib().vc_status_string(status).decode()
        raise VcError(status, msg)


# ------------------------------------------------------------ tensor layer --

def _torch():
    import torch
    return torch


_DTYPE_NAMES = None


def _dtype_name(t) -> str:
    global _DTYPE_NAMES
    if _DTYPE_NAMES is None:
        torch = _torch()
        _DTYPE_NAMES = {torch.int32: "int32", torch.int64: "int64", torch.float32: "float32",
                        torch.bfloat16: "bfloat16"}
    name = _DTYPE_NAMES.get(t.dtype)
    if name is None:
        raise TypeError(f"unsupported dtype {t.dtype}; use int32, int64, float32 or bfloat16")
    return name


def _check_tensors(name: str, ts, dtype: str, numel: int, device):
    if not 1 <= len(ts) <= MAX_RANKS:
        raise ValueError(f"{name}: between 1 and {MAX_RANKS} rank buffers, got {len(ts)}")
    for r, t in enumerate(ts):
        if not t.is_cuda:
            raise ValueError(f"{name}[{r}] is not a CUDA tensor")
        if t.device != device:
            raise ValueError(f"{name}[{r}] is on {t.device}, expected {device}")
        if _dtype_name(t) != dtype:
            raise TypeError(f"{name}[{r}] has dtype {t.dtype}, expected {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name}[{r}] is not contiguous")
        if t.numel() != numel:
            raise ValueError(f"{name}[{r}] holds {t.numel()} elements, expected {numel}")


class _OnDevice:
    """Makes `device` the current CUDA device for one library call, and
    restores the caller's afterwards (the library launches on the current
    device).  Costs one query when it is already current."""
    __slots__ = ("index", "prev")

    def __init__(self, device):
        self.index = device.index

    def __enter__(self):
        cuda = _torch().cuda
        self.prev = cuda.current_device()
        if self.index is not None and self.prev != self.index:
            cuda.set_device(self.index)

    def __exit__(self, *exc):
        if self.index is not None and self.prev != self.index:
            _torch().cuda.set_device(self.prev)
        return False


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptrs(ts):
    return pointer_table([t.data_ptr() for t in ts])


def vc_shard_count(count: int, nranks: int) -> int:
    """q = ceil(count / nranks), the per-rank shard length."""
    return int(lib().vc_shard_count(count, nranks))


def vc_reduce_scatter(sendbufs, recvbufs, op: str = "sum", order: str = "ring", stream=None):
    """recvbufs[r] (q elements) <- reduction of every sendbufs[s] (M elements)
    over the indices of shard r; tail positions past M get the identity."""
    n = len(sendbufs)
    if len(recvbufs) != n:
        raise ValueError("one output shard per rank")
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    q = vc_shard_count(M, n)
    if any(t.numel() != q for t in recvbufs):
        raise ValueError(
            f"output shard must hold ceil(M/N) = {q} elements (M = {M}, N = {n}); "
            f"input must be N times the (padded) output size")
    _check_tensors("recvbufs", recvbufs, dt, q, dev)
    with _OnDevice(dev):
        check_status(lib().vc_reduce_scatter(_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt],
                                             OPS[op], ORDERS[order], _stream(stream, dev)))


def vc_all_gather(sendbufs, recvbufs, count: int | None = None, stream=None):
    """recvbufs[r][s*q + j] <- sendbufs[s][j] for every r, trimmed to count
    (default: recvbufs[0].numel())."""
    n = len(sendbufs)
    if len(recvbufs) != n:
        raise ValueError("one output buffer per rank")
    dt = _dtype_name(recvbufs[0])
    M = recvbufs[0].numel() if count is None else int(count)
    dev = recvbufs[0].device
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    q = vc_shard_count(M, n)
    if any(t.numel() != q for t in sendbufs):
        raise ValueError(f"input shard must hold ceil(M/N) = {q} elements (M = {M}, N = {n})")
    _check_tensors("sendbufs", sendbufs, dt, q, dev)
    with _OnDevice(dev):
        check_status(lib().vc_all_gather(_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt],
                                         _stream(stream, dev)))


def vc_all_reduce(sendbufs, recvbufs=None, op: str = "sum", order: str = "ring", stream=None):
    """recvbufs[r] <- elementwise reduction of all sendbufs, for every r.
    recvbufs=None reduces in place."""
    n = len(sendbufs)
    recvbufs = list(sendbufs) if recvbufs is None else recvbufs
    if len(recvbufs) != n:
        raise ValueError("one output buffer per rank")
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    with _OnDevice(dev):
        check_status(lib().vc_all_reduce(_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt],
                                         OPS[op], ORDERS[order], _stream(stream, dev)))


def vc_all_reduce_decomposed(sendbufs, shardbufs, recvbufs=None, op: str = "sum",
                             order: str = "ring", stream=None):
    """ReduceScatter into shardbufs (q elements each), then AllGather into
    recvbufs (in place if None)."""
    n = len(sendbufs)
    recvbufs = list(sendbufs) if recvbufs is None else recvbufs
    if len(recvbufs) != n or len(shardbufs) != n:
        raise ValueError("one shard and one output buffer per rank")
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    q = vc_shard_count(M, n)
    if any(t.numel() != q for t in shardbufs):
        raise ValueError(f"shard buffers must hold ceil(M/N) = {q} elements")
    _check_tensors("shardbufs", shardbufs, dt, q, dev)
    with _OnDevice(dev):
        check_status(lib().vc_all_reduce_decomposed(_ptrs(sendbufs), _ptrs(shardbufs),
                                                    _ptrs(recvbufs), n, M, DTYPES[dt], OPS[op],
                                                    ORDERS[order], _stream(stream, dev)))


def vc_reduce(sendbufs, recvbuf, op: str = "sum", order: str = "ring", stream=None):
    """recvbuf <- elementwise reduction of all sendbufs (the AllReduce value,
    written once, to the root's buffer; recvbuf may be one of sendbufs)."""
    n = len(sendbufs)
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbuf", [recvbuf], dt, M, dev)
    with _OnDevice(dev):
        check_status(lib().vc_reduce(_ptrs(sendbufs), ctypes.c_void_p(recvbuf.data_ptr()), n, M,
                                     DTYPES[dt], OPS[op], ORDERS[order], _stream(stream, dev)))


def vc_broadcast(sendbuf, recvbufs, stream=None):
    """recvbufs[r] <- sendbuf for every r (one of recvbufs may be sendbuf)."""
    n = len(recvbufs)
    dt = _dtype_name(sendbuf)
    M = sendbuf.numel()
    dev = sendbuf.device
    _check_tensors("sendbuf", [sendbuf], dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    with _OnDevice(dev):
        check_status(lib().vc_broadcast(ctypes.c_void_p(sendbuf.data_ptr()), _ptrs(recvbufs), n, M,
                                        DTYPES[dt], _stream(stream, dev)))


# ------------------------------------------------------ prepared calls --

class Prepared:
    """A collective on fixed buffers, checked once: every call is then one
    C call (the library still repeats its own pointer checks).  Holds
    references to its tensors, so they stay alive as long as the handle.

        ar = prepare_all_reduce(sendbufs, recvbufs, op="sum", order="ring")
        ar()                 # on the current stream
        ar(stream=s)         # on another torch stream
    """

    def __init__(self, fn, args, tensors, device):
        self._fn = fn
        self._args = args
        self._tensors = tensors
        self._device = device

    def __call__(self, stream=None):
        with _OnDevice(self._device):
            check_status(self._fn(*self._args, _stream(stream, self._device)))


def prepare_all_reduce(sendbufs, recvbufs=None, op: str = "sum", order: str = "ring"):
    """vc_all_reduce on these buffers (recvbufs=None: in place)."""
    n = len(sendbufs)
    recvbufs = list(sendbufs) if recvbufs is None else list(recvbufs)
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    args = (_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt], OPS[op], ORDERS[order])
    return Prepared(lib().vc_all_reduce, args, (list(sendbufs), recvbufs), dev)


def prepare_all_reduce_decomposed(sendbufs, shardbufs, recvbufs=None, op: str = "sum",
                                  order: str = "ring"):
    """vc_all_reduce_decomposed on these buffers (recvbufs=None: in place)."""
    n = len(sendbufs)
    recvbufs = list(sendbufs) if recvbufs is None else list(recvbufs)
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    _check_tensors("shardbufs", shardbufs, dt, vc_shard_count(M, n), dev)
    args = (_ptrs(sendbufs), _ptrs(shardbufs), _ptrs(recvbufs), n, M, DTYPES[dt], OPS[op],
            ORDERS[order])
    return Prepared(lib().vc_all_reduce_decomposed, args,
                    (list(sendbufs), list(shardbufs), recvbufs), dev)


def prepare_reduce_scatter(sendbufs, recvbufs, op: str = "sum", order: str = "ring"):
    """vc_reduce_scatter on these buffers."""
    n = len(sendbufs)
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, vc_shard_count(M, n), dev)
    args = (_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt], OPS[op], ORDERS[order])
    return Prepared(lib().vc_reduce_scatter, args, (list(sendbufs), list(recvbufs)), dev)


def prepare_all_gather(sendbufs, recvbufs):
    """vc_all_gather on these buffers."""
    n = len(sendbufs)
    dt = _dtype_name(recvbufs[0])
    M = recvbufs[0].numel()
    dev = recvbufs[0].device
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    _check_tensors("sendbufs", sendbufs, dt, vc_shard_count(M, n), dev)
    args = (_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt])
    return Prepared(lib().vc_all_gather, args, (list(sendbufs), list(recvbufs)), dev)


# ------------------------------------------------ no-allocation variant --

# Size of the library's static shard scratch (VC_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 << 20
_ESIZE = {"int32": 4, "int64": 8, "float32": 4, "bfloat16": 2}


def noalloc_scratch_needed(count: int, nranks: int, dtype: str) -> int:
    """Bytes of shard scratch a call needs: N shards of ceil(count/N)
    elements, each rounded up to 256 bytes."""
    q = -(-count // nranks)
    return nranks * (-(-q * _ESIZE[dtype] // 256) * 256)


def vc_all_reduce_decomposed_noalloc(sendbufs, recvbufs=None, op: str = "sum",
                                     order: str = "ring", stream=None):
    """The decomposed AllReduce (ReduceScatter, then AllGather) for callers
    that cannot allocate device memory where they call it -- code whose
    memory a framework's allocator owns and budgets, latency-critical paths
    that cannot pay for cudaMalloc, plugins handed only their buffers.  The
    N intermediate shards live in a 32 MiB scratch array inside the library
    instead of caller buffers; the call allocates nothing.  Same bits as
    vc_all_reduce_decomposed.  recvbufs=None reduces in place.

    The first call on a device looks up the scratch array's address; make it
    before any stream capture.  Calls share the array: calls that overlap on
    the GPU race.  Raises ValueError when the shards do not fit."""
    n = len(sendbufs)
    recvbufs = list(sendbufs) if recvbufs is None else recvbufs
    if len(recvbufs) != n:
        raise ValueError("one output buffer per rank")
    dt = _dtype_name(sendbufs[0])
    M = sendbufs[0].numel()
    dev = sendbufs[0].device
    _check_tensors("sendbufs", sendbufs, dt, M, dev)
    _check_tensors("recvbufs", recvbufs, dt, M, dev)
    need = noalloc_scratch_needed(M, n, dt)
    if need > NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"{n} shards of {vc_shard_count(M, n)} {dt} elements need {need} bytes "
                         f"of scratch; the library's static scratch holds "
                         f"{NOALLOC_SCRATCH_BYTES} bytes (use vc_all_reduce_decomposed with "
                         f"caller-allocated shards)")
    L = lib()
    fn = L.vc_all_reduce_decomposed_noalloc
    vpp = ctypes.POINTER(ctypes.c_void_p)
    fn.argtypes = [vpp, vpp, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    with _OnDevice(dev):
        check_status(fn(_ptrs(sendbufs), _ptrs(recvbufs), n, M, DTYPES[dt], OPS[op], ORDERS[order],
                        _stream(stream, dev)))


# ------------------------------------------------------------ fused buckets --

class BucketPlan:
    """A gradient bucket whose tensors stay where they are (vc_bucket_plan):
    tensors[r][k] is tensor k of rank r, out[r][k] its AllReduce output
    (None: in place).  The bucket holds the tensors in the order given, each
    on a 16-byte boundary.  all_reduce() (also the call operator) gives every
    element the bits the ring-order AllReduce of that bucket gives it;
    reduce_scatter() writes shard r of the bucket's ring-order ReduceScatter
    to rank r's shard; all_gather() writes the shards back into every rank's
    output tensors.  Planned once (pointer checks, aliasing, tiles); each
    call is one launch.  The plan keeps the tensors' addresses: make a new
    one if they change."""

    def __init__(self, tensors, out=None, order: str = "ring"):
        import torch
        n = len(tensors)
        if n < 1 or n > MAX_RANKS:
            raise ValueError(f"1 <= ranks <= {MAX_RANKS}")
        out = tensors if out is None else out
        nt = len(tensors[0])
        if any(len(t) != nt for t in tensors) or len(out) != n or any(len(o) != nt for o in out):
            raise ValueError("every rank needs the same number of tensors, inputs and outputs")
        if nt == 0:
            raise ValueError("a bucket needs at least one tensor")
        dt = _dtype_name(tensors[0][0])
        dev = tensors[0][0].device
        counts = [tensors[0][k].numel() for k in range(nt)]
        for r in range(n):
            for k in range(nt):
                for name, t in (("tensors", tensors[r][k]), ("out", out[r][k])):
                    if not (t.is_cuda and t.device == dev and t.is_contiguous()
                            and _dtype_name(t) == dt and t.numel() == counts[k]):
                        raise ValueError(f"{name}[{r}][{k}] does not match tensor {k} of rank 0 "
                                         f"(device, dtype, contiguity, numel)")
        L = lib()
        ins = [tensors[r][k].data_ptr() for k in range(nt) for r in range(n)]
        outs = [out[r][k].data_ptr() for k in range(nt) for r in range(n)]
        in_tab = (ctypes.c_void_p * len(ins))(*ins)
        out_tab = (ctypes.c_void_p * len(outs))(*outs)
        cnt = (ctypes.c_size_t * nt)(*counts)
        vpp = ctypes.POINTER(ctypes.c_void_p)
        ntiles, bucket_count = ctypes.c_int(0), ctypes.c_size_t(0)
        args = (ctypes.cast(in_tab, vpp), ctypes.cast(out_tab, vpp), cnt, nt, n, DTYPES[dt],
                ORDERS[order])
        check_status(L.vc_bucket_plan(*args, None, 0, ctypes.byref(ntiles),
                                      ctypes.byref(bucket_count)))
        tiles = (BucketTile * max(1, ntiles.value))()
        check_status(L.vc_bucket_plan(*args, tiles, ntiles.value, ctypes.byref(ntiles),
                                      ctypes.byref(bucket_count)))
        self.ntiles, self.bucket_count, self.nranks, self.dtype = (ntiles.value,
                                                                  bucket_count.value, n, dt)
        self.device = dev
        raw = bytes(memoryview(tiles).cast("B"))[:ctypes.sizeof(BucketTile) * ntiles.value]
        self.tiles = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(dev)
        self.in_ptrs = torch.tensor(ins, dtype=torch.int64).to(dev)
        self.out_ptrs = torch.tensor(outs, dtype=torch.int64).to(dev)
        self._keep = (tensors, out)
        self._checked_shards = None
        self.host_tiles = tiles

    def _check_shards(self, shards):
        """One shard per rank, of the bucket's dtype, device and shard length,
        overlapping no planned tensor (checked once per set of buffers)."""
        if len(shards) != self.nranks:
            raise ValueError("one shard per rank")
        key = tuple(t.data_ptr() for t in shards)
        if key == self._checked_shards:
            return
        _check_tensors("shards", shards, self.dtype, self.shard_count, self.device)
        for t in shards:
            for rows in self._keep:
                for row in rows:
                    for g in row:
                        if g.numel() and _overlaps(t, g):
                            raise ValueError("a shard overlaps a bucket tensor")
        self._checked_shards = key

    @property
    def shard_count(self) -> int:
        """q: the elements of one rank's shard of the bucket."""
        return vc_shard_count(self.bucket_count, self.nranks)

    def __call__(self, op: str = "sum", stream=None):
        self.all_reduce(op=op, stream=stream)

    def reduce_scatter(self, shards, op: str = "sum", stream=None):
        """shards[r]: rank r's output, shard_count elements of the bucket's
        dtype on its device; disjoint from each other and from the tensors."""
        self._check_shards(shards)
        with _OnDevice(self.device):
            check_status(lib().vc_reduce_scatter_bucket(
                ctypes.c_void_p(self.tiles.data_ptr()), self.ntiles,
                ctypes.c_void_p(self.in_ptrs.data_ptr()), _ptrs(shards), self.nranks,
                self.bucket_count, DTYPES[self.dtype], OPS[op], _stream(stream, self.device)))

    def all_gather(self, shards, stream=None):
        """shards[r] (shard_count elements) gathered back into every rank's
        output tensors: out[r][k] receives the bucket's elements of tensor k
        from the shards that hold them."""
        self._check_shards(shards)
        with _OnDevice(self.device):
            check_status(lib().vc_all_gather_bucket(
                ctypes.c_void_p(self.tiles.data_ptr()), self.ntiles, _ptrs(shards),
                ctypes.c_void_p(self.out_ptrs.data_ptr()), self.nranks, self.bucket_count,
                DTYPES[self.dtype], _stream(stream, self.device)))

    def all_reduce(self, op: str = "sum", stream=None):
        with _OnDevice(self.device):
            check_status(lib().vc_all_reduce_bucket(
                ctypes.c_void_p(self.tiles.data_ptr()), self.ntiles,
                ctypes.c_void_p(self.in_ptrs.data_ptr()), ctypes.c_void_p(self.out_ptrs.data_ptr()),
                self.nranks, self.bucket_count, DTYPES[self.dtype], OPS[op],
                _stream(stream, self.device)))


def _overlaps(a, b) -> bool:
    """Whether two tensors' byte ranges overlap."""
    a0, b0 = a.data_ptr(), b.data_ptr()
    return a0 < b0 + b.numel() * b.element_size() and b0 < a0 + a.numel() * a.element_size()
