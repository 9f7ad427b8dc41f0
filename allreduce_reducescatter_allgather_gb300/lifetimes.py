"""Buffer lifetimes around the collectives: the ZeRO-style ReduceScatter that
keeps only the shards, and the decomposed AllReduce that releases its inputs
before it allocates its outputs.

Background ("NCCL 专家课程 07", 显存实验必须区分 steady 与 peak; ZeRO/FSDP 为什么
停在 ReduceScatter): with 256 MiB per rank a direct AllReduce peaks at 256 MiB,
RS-only keeps a 64 MiB shard (peak 320), and RS + AG in a naive lifetime
peaks at 576 MiB because input, shard and output are alive at once.  Freeing
the input before the AllGather allocates brings the peak back to 320 MiB.  The
page frees after an explicit synchronize and notes that production code relies
on stream-ordered allocation and stream recording instead.  That is what these
helpers do: PyTorch's caching allocator hands memory freed on a stream to the
next allocation on the same stream in stream order, and record_stream() keeps
memory that another stream still uses from being reused early.  No
synchronize is needed and the collectives still run in the library's kernels.

Every helper takes ownership of the input list it is given: it empties the
list, and the inputs' memory is released once the caller holds no other
reference to those tensors.
"""
from __future__ import annotations

from . import _binding


def _current(torch, device):
    return torch.cuda.current_stream(device)


def _release(torch, tensors: list, stream) -> None:
    """Drop the list's references; memory last used on another stream is
    tied to `stream` first, so the allocator waits for it."""
    for t in tensors:
        t.record_stream(stream)
    tensors.clear()


def reduce_scatter_keep_shards(inputs: list, op: str = "sum", order: str = "ring"):
    """ZeRO-style ReduceScatter: returns the N shards (q elements each) and
    releases the inputs, so the steady state holds shards only."""
    import torch
    dev = inputs[0].device
    n, M = len(inputs), inputs[0].numel()
    q = _binding.vc_shard_count(M, n)
    shards = [torch.empty(q, dtype=inputs[0].dtype, device=dev) for _ in range(n)]
    stream = _current(torch, dev)
    _binding.vc_reduce_scatter(inputs, shards, op=op, order=order, stream=stream)
    _release(torch, inputs, stream)
    return shards


def all_gather_new(shards: list, count: int, release_shards: bool = True):
    """AllGather into freshly allocated outputs of `count` elements; releases
    the shards when asked."""
    import torch
    dev = shards[0].device
    n = len(shards)
    outs = [torch.empty(count, dtype=shards[0].dtype, device=dev) for _ in range(n)]
    stream = _current(torch, dev)
    _binding.vc_all_gather(shards, outs, count=count, stream=stream)
    if release_shards:
        _release(torch, shards, stream)
    return outs


def all_reduce_decomposed_low_peak(inputs: list, op: str = "sum", order: str = "ring"):
    """The decomposed AllReduce with the short lifetime: ReduceScatter into
    new shards, release the inputs, allocate the outputs (which may reuse the
    inputs' memory, in stream order), AllGather, release the shards.  Peak =
    inputs + shards instead of inputs + shards + outputs.  Same bits as
    vc_all_reduce in the same order."""
    M = inputs[0].numel()
    shards = reduce_scatter_keep_shards(inputs, op=op, order=order)
    return all_gather_new(shards, M, release_shards=True)
