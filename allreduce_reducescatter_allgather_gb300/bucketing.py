"""Gradient buckets for the virtual-rank AllReduce.

What the pages say ("Ring AllReduce 核心流程" 4; "通信与互联（01）" 三.1 and
九.1): small tensors are merged into buckets before the collective, so one
large message replaces many small ones.  DDP fills a bucket while backward
runs and sends it when it is full.  Its caps are 25 MiB per bucket
(kDefaultBucketBytesCap), and 1 MiB for the first bucket
(kDefaultFirstBucketBytes) so that something can be sent early.  On one GPU the
saving is one kernel launch per bucket instead of one per tensor, and a
bucket large enough to run at the HBM rate.

Three ways to feed a bucket:
 - views (no copy): every gradient tensor is a view into its rank's flat
   bucket buffer (what DDP calls gradients as bucket views); the AllReduce
   runs in place on the buckets and the views hold the results;
 - fused: tensors that live elsewhere are reduced where they are, one launch
   per bucket (vc_bucket_plan + vc_all_reduce_bucket), with the bits the
   bucket's AllReduce gives them: integers in every order, floats in ring
   order;
 - packing: tensors are copied into the buckets and back with
   vc_copy_tiles around the bucket's AllReduce, three launches per bucket
   (any order).

Assignment rule (the pages give only the caps; this is the plain reading):
tensors are taken in reverse order, the order backward produces their
gradients.  A bucket closes when the next tensor would take it past its cap.
The first bucket's cap is the small one.  A tensor larger than the cap gets a
bucket of its own.  Inside a bucket every tensor starts on a 16-byte boundary.
Padding elements are zero and are reduced like the rest (zero in, identity
out for SUM; never read back).
"""
from __future__ import annotations

from dataclasses import dataclass

from . import _binding

FIRST_BUCKET_BYTES = 1 << 20  # kDefaultFirstBucketBytes
BUCKET_BYTES = 25 << 20       # kDefaultBucketBytesCap
ALIGN_BYTES = 16
TILE_BYTES = 1 << 16          # VC_COPY_TILE_MAX_BYTES


def assign_buckets(nbytes, first_cap: int = FIRST_BUCKET_BYTES, cap: int = BUCKET_BYTES):
    """Bucket membership for tensors of the given sizes (bytes, in forward
    order): a list of buckets, each a list of tensor indices in the order
    they are filled (reverse tensor order)."""
    buckets, cur, size = [], [], 0
    limit = first_cap
    for t in reversed(range(len(nbytes))):
        b = int(nbytes[t])
        if cur and size + b > limit:
            buckets.append(cur)
            cur, size = [], 0
            limit = cap
        cur.append(t)
        size += b
    if cur:
        buckets.append(cur)
    return buckets


@dataclass
class _Bucket:
    tensors: list      # tensor indices in the bucket, in fill order
    offsets: list      # element offset of each of them in the bucket buffer
    count: int         # elements in the bucket buffer (padding included)
    buffers: list      # one flat device buffer per rank
    pack_tiles: object = None    # device table for vc_copy_tiles (tensors -> bucket)
    unpack_tiles: object = None  # (bucket -> tensors)
    ntiles: int = 0
    fused: object = None         # BucketPlan over the bound tensors, in place
    shards: object = None        # ReduceScatter outputs, one per rank


class GradientBuckets:
    """Flat bucket buffers for `nranks` virtual ranks, each holding tensors
    of the given shapes (the same on every rank) and dtype."""

    def __init__(self, shapes, dtype, nranks: int, device, first_cap: int = FIRST_BUCKET_BYTES,
                 cap: int = BUCKET_BYTES):
        import torch
        self.torch = torch
        self.shapes = [tuple(s) for s in shapes]
        self.numels = [int(torch.Size(s).numel()) for s in self.shapes]
        self.dtype = dtype
        self.nranks = nranks
        self.device = torch.device(device)
        es = torch.empty(0, dtype=dtype).element_size()
        self.es = es
        align = ALIGN_BYTES // es
        self.buckets = []
        self._prepared = {}
        self.where = [None] * len(self.shapes)  # tensor -> (bucket, offset)
        for members in assign_buckets([n * es for n in self.numels], first_cap, cap):
            offsets, off = [], 0
            for t in members:
                off = (off + align - 1) // align * align
                offsets.append(off)
                off += self.numels[t]
            count = max(1, (off + align - 1) // align * align)
            bufs = [torch.zeros(count, dtype=dtype, device=self.device) for _ in range(nranks)]
            b = _Bucket(members, offsets, count, bufs)
            for t, o in zip(members, offsets):
                self.where[t] = (len(self.buckets), o)
            self.buckets.append(b)

    # ---------------------------------------------------------- views --
    def views(self, rank: int):
        """Tensors of `rank` as views into its bucket buffers (forward order):
        write gradients into them, then call all_reduce()."""
        out = []
        for t, shape in enumerate(self.shapes):
            bi, off = self.where[t]
            buf = self.buckets[bi].buffers[rank]
            out.append(buf[off:off + self.numels[t]].view(shape))
        return out

    def _calls(self, op: str, order: str):
        """The buckets' in-place AllReduce calls, prepared once per op and
        order (a call is then one C call per bucket)."""
        key = (op, order)
        calls = self._prepared.get(key)
        if calls is None:
            calls = [_binding.prepare_all_reduce(b.buffers, None, op=op, order=order)
                     for b in self.buckets]
            self._prepared[key] = calls
        return calls

    def all_reduce(self, op: str = "sum", order: str = "ring", stream=None):
        """One in-place AllReduce per bucket."""
        for c in self._calls(op, order):
            c(stream=stream)

    # --------------------------------------------------- ReduceScatter --
    def shards(self, bucket: int):
        """Rank r's shard of bucket `bucket` (ceil(count / N) elements each),
        the output of the ReduceScatter calls; allocated on first use."""
        b = self.buckets[bucket]
        if getattr(b, "shards", None) is None:
            q = _binding.vc_shard_count(b.count, self.nranks)
            b.shards = [self.torch.empty(q, dtype=self.dtype, device=self.device)
                        for _ in range(self.nranks)]
        return b.shards

    def reduce_scatter(self, op: str = "sum", order: str = "ring", stream=None):
        """ZeRO-style: one ReduceScatter per bucket, from the bucket buffers
        into shards(bucket); returns the shards of every bucket."""
        key = ("rs", op, order)
        calls = self._prepared.get(key)
        if calls is None:
            calls = [_binding.prepare_reduce_scatter(b.buffers, self.shards(i), op=op, order=order)
                     for i, b in enumerate(self.buckets)]
            self._prepared[key] = calls
        for c in calls:
            c(stream=stream)
        return [self.shards(i) for i in range(len(self.buckets))]

    # -------------------------------------------------------- packing --
    def _tiles(self, b: _Bucket, grads, to_bucket: bool):
        rows = []
        for r in range(self.nranks):
            base = b.buffers[r].data_ptr()
            for t, off in zip(b.tensors, b.offsets):
                g = grads[r][t]
                nbytes = self.numels[t] * self.es
                tp, bp = g.data_ptr(), base + off * self.es
                for k in range(0, nbytes, TILE_BYTES):
                    n = min(TILE_BYTES, nbytes - k)
                    rows.append((tp + k, bp + k, n) if to_bucket else (bp + k, tp + k, n))
        return rows

    def bind(self, grads):
        """Build the pack / unpack tables for grads[rank][tensor] (tensors
        outside the buckets, contiguous, of the given shapes and dtype).  The
        tables hold the tensors' addresses: rebind if the tensors change."""
        torch = self.torch
        for r in range(self.nranks):
            for t, g in enumerate(grads[r]):
                if not (g.is_cuda and g.is_contiguous() and g.dtype == self.dtype
                        and g.numel() == self.numels[t] and g.device == self.device):
                    raise ValueError(f"grads[{r}][{t}] does not match the bucket layout")
        for b in self.buckets:
            pack = self._tiles(b, grads, True)
            unpack = self._tiles(b, grads, False)
            b.pack_tiles = torch.tensor(pack, dtype=torch.int64).to(self.device)
            b.unpack_tiles = torch.tensor(unpack, dtype=torch.int64).to(self.device)
            b.ntiles = len(pack)
            # the fused call lays the bucket out the same way: its tensors in
            # fill order, each on a 16-byte boundary
            b.fused = _binding.BucketPlan(
                [[grads[r][t] for t in b.tensors] for r in range(self.nranks)])
            assert b.fused.bucket_count == b.count or not any(self.numels[t] for t in b.tensors)
        self.bound = grads

    def fused_supported(self, order: str) -> bool:
        """Whether all_reduce_tensors(fused=True) takes one launch per bucket
        for this order: always for integers (order-free), the ring for floats."""
        return order == "ring" or self.dtype not in (self.torch.float32, self.torch.bfloat16)

    def all_reduce_tensors(self, op: str = "sum", order: str = "ring", stream=None,
                           fused: bool = True):
        """For the bound tensors, in place.  fused (when the order allows it,
        see fused_supported): one launch per bucket that reduces the tensors
        where they are.  Otherwise, per bucket: pack (one launch), AllReduce
        in place (one launch), unpack (one launch).  Both give the bits of
        the bucket views path."""
        torch = self.torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        if fused and self.fused_supported(order):
            if order == "recursive_halving" and self.nranks & (self.nranks - 1):
                raise ValueError("recursive halving needs a power-of-two rank count")
            for b in self.buckets:
                b.fused(op=op, stream=stream)
            return
        import ctypes
        L = _binding.lib()
        s = ctypes.c_void_p(stream.cuda_stream)
        for b, c in zip(self.buckets, self._calls(op, order)):
            with _binding._OnDevice(self.device):
                _binding.check_status(L.vc_copy_tiles(ctypes.c_void_p(b.pack_tiles.data_ptr()),
                                                      b.ntiles, s))
            c(stream=stream)
            with _binding._OnDevice(self.device):
                _binding.check_status(L.vc_copy_tiles(
                    ctypes.c_void_p(b.unpack_tiles.data_ptr()), b.ntiles, s))

    def all_gather_tensors(self, stream=None):
        """FSDP's unpack: every bucket's shards (shards(bucket), e.g. after
        the optimizer updated them) gathered back into the bound tensors of
        every rank, one launch per bucket.  After reduce_scatter_tensors it
        completes the decomposed AllReduce of the buckets."""
        torch = self.torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        for i, b in enumerate(self.buckets):
            b.fused.all_gather(self.shards(i), stream=stream)

    def reduce_scatter_tensors(self, op: str = "sum", order: str = "ring", stream=None,
                               fused: bool = True):
        """For the bound tensors: the bucket's ReduceScatter into
        shards(bucket), with the bits of packing them first.  fused (when the
        order allows it, see fused_supported): one launch per bucket, the
        tensors read where they are; otherwise pack (one launch) and
        ReduceScatter the bucket buffer (one launch).  Returns the shards."""
        torch = self.torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        if fused and self.fused_supported(order):
            if order == "recursive_halving" and self.nranks & (self.nranks - 1):
                raise ValueError("recursive halving needs a power-of-two rank count")
            for i, b in enumerate(self.buckets):
                b.fused.reduce_scatter(self.shards(i), op=op, stream=stream)
            return [self.shards(i) for i in range(len(self.buckets))]
        import ctypes
        L = _binding.lib()
        s = ctypes.c_void_p(stream.cuda_stream)
        for b in self.buckets:
            with _binding._OnDevice(self.device):
                _binding.check_status(L.vc_copy_tiles(ctypes.c_void_p(b.pack_tiles.data_ptr()),
                                                      b.ntiles, s))
        return self.reduce_scatter(op=op, order=order, stream=stream)
