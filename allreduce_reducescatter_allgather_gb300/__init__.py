"""AllReduce, ReduceScatter and AllGather over N virtual ranks on one GB300.

N "ranks" are N device buffers in one GPU's memory.  The collectives run as
hand-written sm_103a kernels (libvc.so, C ABI in include/vc.h) that read the
N buffers with 16-byte vector loads and reduce them in registers in a fixed
order (ring, recursive halving or tree).  This package is the thin ctypes
binding with the same names as the C entry points.
"""
from ._binding import (  # noqa: F401
    BucketPlan,
    DTYPES,
    MAX_RANKS,
    OPS,
    ORDERS,
    VcError,
    Prepared,
    lib,
    prepare_all_gather,
    prepare_all_reduce,
    prepare_all_reduce_decomposed,
    prepare_reduce_scatter,
    vc_all_gather,
    vc_all_reduce,
    vc_all_reduce_decomposed,
    vc_all_reduce_decomposed_noalloc,
    vc_broadcast,
    vc_reduce,
    vc_reduce_scatter,
    vc_shard_count,
)
