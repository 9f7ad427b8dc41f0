/*
 * vc.h -- AllReduce, ReduceScatter and AllGather over N virtual ranks held
 * in one GPU's memory.
 *
 * A "virtual rank" is one device buffer.  Every call takes host arrays of N
 * device pointers (one per rank), the logical per-rank element count M, the
 * element type, the reduction op and the reduction order, and enqueues one
 * kernel (two for the decomposed AllReduce) on the caller's CUDA stream.
 *
 * Definitions ("NCCL 专家课程 07：AllReduce 等价分解、显存生命周期与 Kernel
 * 证据", section 数学证明; q = ceil(M/N)):
 *   AllReduce      y^(r)_i        = (+)_{s=0}^{N-1} x^(s)_i,   0 <= i < M, every r
 *   ReduceScatter  z^(r)_j        = (+)_{s=0}^{N-1} x^(s)_{rq+j}, 0 <= j < q
 *   AllGather      yhat^(r)_{sq+j} = z^(s)_j   (source-rank-major), trimmed to M
 * with the inputs padded from M to Nq with the op's identity (same page,
 * 条件三: 0 for sum, 1 for prod, the type's minimum / -inf for max, the
 * maximum / +inf for min; never 0 for max).  The padding is virtual: indices
 * >= M are read as the identity and never stored anywhere.
 *
 * Counts follow NCCL's rule that the ReduceScatter output count is the
 * AllGather input count (same page, 源码一): every call takes the logical M;
 * ReduceScatter writes q elements per rank and AllGather reads q per rank.
 *
 * Ownership and lifetime: the caller owns every buffer; the library never
 * allocates device memory and keeps no pointer after a call returns (the
 * pointer tables are copied by value into the kernel's parameters).  Calls
 * are asynchronous on `stream`; results are valid once the stream has
 * passed the call.  Every buffer must be aligned to its element size; when
 * every base pointer involved is also 16-byte aligned the kernels use
 * 16-byte vector accesses for the bulk of the data (otherwise they fall back
 * to element-wise accesses, on the GPU).
 *
 * Errors: arguments are checked on the host before anything is enqueued; on
 * any error the call returns a non-zero status and launches nothing (the
 * pages' capacity check also rejects before any kernel, 源码五 and Contract
 * 实验四).  VC_ERR_CUDA reports a failed launch; nothing else is retried.
 * All entry points are thread-safe; calls enqueued on different streams
 * that write overlapping memory race, as any two kernels would.
 */
#ifndef VC_H
#define VC_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The largest number of virtual ranks one call takes. */
#define VC_MAX_RANKS 64

/* Element types.  Integers accumulate in 64 bits and wrap modulo 2^64
 * (int32 results are the low 32 bits), so an integer result is the same in
 * every reduction order (every order is computed with the ring's kernels);
 * float32 accumulates in float32;
 * bfloat16 is widened exactly to float32, accumulated in float32 and rounded
 * once to nearest-even at the store.  (The pages fix no accumulator for
 * bf16; they note that float reduction is not associative, 条件五.) */
typedef enum {
    VC_INT32 = 0,
    VC_INT64 = 1,
    VC_FLOAT32 = 2,
    VC_BFLOAT16 = 3
} vc_dtype_t;

/* Reduction ops ("通信与互联（01）：集合通信原语与代价模型", 二.1: sum, max,
 * min, prod, avg).  AVG is the SUM in the chosen order divided once by N:
 * one IEEE single division for float types, truncation toward zero for
 * integers.  MAX/MIN keep the running value on ties.  NaN inputs are outside
 * the contract. */
typedef enum {
    VC_SUM = 0,
    VC_PROD = 1,
    VC_MAX = 2,
    VC_MIN = 3,
    VC_AVG = 4
} vc_op_t;

/* Reduction orders.  For integers and for MAX/MIN every order gives the same
 * bits; for float SUM/PROD/AVG the order is part of the result (条件五).
 * Element i lies in chunk c = floor(i/q).
 *  RING: the ring ReduceScatter schedule ("Ring AllReduce 核心流程" and
 *    "通信与互联（01）" 五.2: at step s rank r sends chunk (r-s+1) mod N and
 *    adds the chunk it receives into its own copy; rank r ends owning chunk
 *    (r+1) mod N).  Chunk c's value is
 *    (((x^(c) (+) x^(c+1)) (+) x^(c+2)) ... (+) x^(c+N-1)), ranks mod N.
 *    Any N from 1 to VC_MAX_RANKS.
 *  RECURSIVE_HALVING: step j pairs ranks at distance N/2^j and each keeps
 *    the combination of its half with its partner's ("ReduceScatter" page,
 *    Recursive Halving; N=8 pairs (0,4)(1,5)(2,6)(3,7), (0,2)..., (0,1)...).
 *    The value is the balanced pairwise tree over the ranks in bit-reversed
 *    order, e.g. ((x0(+)x4)(+)(x2(+)x6))(+)((x1(+)x5)(+)(x3(+)x7)).  N must be
 *    a power of two (the page's hypercube condition).
 *  PAIRWISE_TREE: the binary tree of "通信与互联（01）" 六.1 (rank 0 the root
 *    with a single child; rank r's level is its lowest set bit L and its
 *    parent is (r-L) | 2L; odd ranks are leaves).  An inner node's value is
 *    (left subtree (+) right subtree) (+) its own operand, the lower-ranked
 *    child on the left.  The page draws N = 8 only; for any N, a rank whose
 *    parent label (r-L) | 2L is not a rank (>= N) hangs under r-L instead,
 *    which keeps the tree binary with a single-child root and depth
 *    ceil(log2 N).  Any N from 1 to VC_MAX_RANKS.
 *  DOUBLE_BINARY_TREE: two trees, each carrying half of the data
 *    ("通信与互联（01）" 六.3): the first ceil(count/2) elements in the
 *    PAIRWISE_TREE order (tree A), the others in tree B, in which node k of
 *    tree A is played by rank (k+1) mod N for even N (rank numbers shifted by
 *    one: root rank 1, its child rank N/2 + 1, ...) and by rank N-1-k for odd
 *    N (the mirror image).  Any N from 1 to VC_MAX_RANKS. */
typedef enum {
    VC_ORDER_RING = 0,
    VC_ORDER_RECURSIVE_HALVING = 1,
    VC_ORDER_PAIRWISE_TREE = 2,
    VC_ORDER_DOUBLE_BINARY_TREE = 3
} vc_order_t;

typedef enum {
    VC_SUCCESS = 0,
    /* a NULL pointer table or buffer, a buffer not aligned to its element
     * size, nranks outside [1, VC_MAX_RANKS], an unknown enum value, or a
     * count whose byte size exceeds 2^62 */
    VC_ERR_INVALID_ARGUMENT = 1,
    /* RECURSIVE_HALVING with nranks not a power of two */
    VC_ERR_UNSUPPORTED = 2,
    /* an output range overlaps an input range or another output range (the
     * only overlap allowed is the in-place AllReduce, recvbufs[r] ==
     * sendbufs[r] exactly) */
    VC_ERR_ALIAS = 3,
    /* the CUDA runtime refused the launch or a device query.  (Setting the
     * environment variable VC_TEST_FAIL_LAUNCH to a non-zero value makes
     * every call that passes its checks return this without launching: a
     * test hook for the error path.) */
    VC_ERR_CUDA = 4
} vc_status_t;

/* A cudaStream_t, passed as an opaque pointer; NULL is the legacy default
 * stream. */
typedef void *vc_stream_t;

/* q = ceil(count / nranks): the shard length ReduceScatter writes and
 * AllGather reads per rank.  Returns 0 when nranks < 1. */
size_t vc_shard_count(size_t count, int nranks);

/* ReduceScatter.  sendbufs[s] (s < nranks): device buffer of `count`
 * elements, rank s's input x^(s).  recvbufs[r]: device buffer of
 * q = vc_shard_count(count, nranks) elements, receives z^(r); positions j with
 * r*q + j >= count receive the op's identity (0 for AVG).  No recv buffer may
 * overlap any send buffer or another recv buffer.  count == 0 returns
 * VC_SUCCESS without launching. */
vc_status_t vc_reduce_scatter(const void *const *sendbufs, void *const *recvbufs, int nranks,
                              size_t count, vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                              vc_stream_t stream);

/* AllGather.  sendbufs[s]: device buffer of q = vc_shard_count(count,
 * nranks) elements, shard s.  recvbufs[r]: device buffer of `count`
 * elements; receives shard s at offset s*q for every s, trimmed to `count`
 * (elements of the last shard past `count` are not read).  No recv buffer
 * may overlap a send buffer or another recv buffer.  AllGather moves bits
 * only; it takes no op or order. */
vc_status_t vc_all_gather(const void *const *sendbufs, void *const *recvbufs, int nranks,
                          size_t count, vc_dtype_t dtype, vc_stream_t stream);

/* AllReduce in one kernel: every element is read once from each of the N
 * inputs, reduced in registers and written to all N outputs (the single-GPU
 * counterpart of a ring AllReduce that fuses its last reduction with the
 * first forward of the gather phase, "NCCL 专家课程 07" 源码三).
 * sendbufs[s], recvbufs[r]: device buffers of `count` elements.  In place is
 * allowed per rank (recvbufs[r] == sendbufs[r]); any other overlap is
 * VC_ERR_ALIAS. */
vc_status_t vc_all_reduce(const void *const *sendbufs, void *const *recvbufs, int nranks,
                          size_t count, vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                          vc_stream_t stream);

/* AllReduce as two kernels: ReduceScatter into shardbufs (N buffers of q
 * elements, scratch owned by the caller), then AllGather from them into
 * recvbufs ("NCCL 专家课程 07", 源码四/五: two separate collectives).  Gives
 * the same bits as vc_all_reduce in the same order.  recvbufs[r] ==
 * sendbufs[r] is allowed; shard buffers may overlap nothing. */
vc_status_t vc_all_reduce_decomposed(const void *const *sendbufs, void *const *shardbufs,
                                     void *const *recvbufs, int nranks, size_t count,
                                     vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                                     vc_stream_t stream);

/* Reduce: the AllReduce value of every element, written to one buffer only
 * (the root's): y_i = (+)_s x^(s)_i for 0 <= i < count, in `order`, with the
 * same bits vc_all_reduce gives ("通信与互联（01）" 二.1, reduce with root 0;
 * 二.2: all_reduce = reduce + broadcast).  sendbufs[s]: device buffers of
 * `count` elements; recvbuf: device buffer of `count` elements, which may be
 * exactly one of the inputs (the root reducing in place) and must not
 * otherwise overlap them. */
vc_status_t vc_reduce(const void *const *sendbufs, void *recvbuf, int nranks, size_t count,
                      vc_dtype_t dtype, vc_op_t op, vc_order_t order, vc_stream_t stream);

/* Broadcast: recvbufs[r][i] = sendbuf[i] for every r and 0 <= i < count
 * ("通信与互联（01）" 二.1, broadcast from root 0).  sendbuf: the root's
 * device buffer of `count` elements; recvbufs: nranks device buffers of
 * `count` elements, pairwise disjoint.  One of them may be sendbuf itself
 * (the root's own buffer), which is left as it is; no other may overlap it.
 * Moves bits only. */
vc_status_t vc_broadcast(const void *sendbuf, void *const *recvbufs, int nranks, size_t count,
                         vc_dtype_t dtype, vc_stream_t stream);

/* One byte range to copy: `bytes` bytes from src to dst (device memory). */
typedef struct {
    const void *src;
    void *dst;
    size_t bytes;
} vc_copy_tile_t;

/* The largest tile vc_copy_tiles takes; longer ranges are split by the
 * caller into several tiles. */
#define VC_COPY_TILE_MAX_BYTES (1u << 16)

/* Copies many independent byte ranges in one launch: the packing of many
 * small tensors into a bucket buffer before its AllReduce, and the unpacking
 * after it (the pages' DDP buckets: gradients are merged into 25 MiB buckets,
 * the first one 1 MiB, so one large collective replaces many small ones --
 * "通信与互联（01）" 三.1 and 九.1; "Ring AllReduce 核心流程" 4).
 * dev_tiles: a DEVICE array of ntiles entries (8-byte aligned), each with
 * 0 < bytes <= VC_COPY_TILE_MAX_BYTES, src and dst device pointers.  The
 * entries live in device memory, so the library cannot check them: ranges
 * that are invalid, overlap each other's destinations, or overlap within a
 * tile are undefined behaviour, as for any device copy.  ntiles == 0
 * launches nothing. */
vc_status_t vc_copy_tiles(const vc_copy_tile_t *dev_tiles, int ntiles, vc_stream_t stream);

/* ---- fused AllReduce of a gradient bucket --------------------------------
 *
 * The pages' DDP buckets ("通信与互联（01）" 三.1 and 九.1; "Ring AllReduce
 * 核心流程" 4): many small gradient tensors are reduced as one bucket so that
 * one large collective replaces many small ones.  When the tensors cannot
 * live inside the bucket buffer, packing them in and out around the
 * AllReduce moves every byte three times.  These two calls reduce the
 * tensors where they are, in one launch, with the bits of the packed path.
 *
 * The bucket: the tensors in the order given, tensor k at element offset
 * b_k of the bucket, where b_0 = 0 and b_{k+1} is b_k + counts[k] rounded up
 * to a multiple of 16 bytes; bucket_count is the end of the last tensor
 * rounded up the same way.  Element j of tensor k gets, on every rank, the
 * value the ring-order AllReduce (VC_ORDER_RING) of the bucket gives at
 * bucket index b_k + j, the gaps between tensors holding zeros; with the
 * tensors packed into one buffer per rank, vc_all_reduce on that buffer
 * gives the same bits. */

/* One tile of a fused bucket AllReduce, as vc_bucket_plan writes it: count
 * consecutive elements of tensor `tensor`, starting at its element
 * tensor_offset, which stand at element bucket_offset of the bucket.  A
 * tile never crosses a ring chunk boundary of the bucket (a multiple of
 * vc_shard_count(bucket_count, nranks)).  flags bit 0: every rank's input
 * and output address of the tile's first element is 16-byte aligned. */
typedef struct {
    long long bucket_offset;
    long long tensor_offset;
    long long count;
    int tensor;
    int flags;
} vc_bucket_tile_t;

/* The largest tile vc_bucket_plan makes, per rank.  (Measured on GB300 with
 * a 351 MiB set of 145 bf16 tensors on 8 ranks: 64 KiB tiles ran 13 % behind
 * the in-bucket AllReduce, 16 KiB tiles 4 %, 8 KiB tiles 2 %: more, smaller
 * tiles balance the last wave of blocks.  The bucket AllGather lost 1 % from
 * 16 to 8 KiB, the ReduceScatter did not move.) */
#define VC_BUCKET_TILE_MAX_BYTES (1u << 13)

/* Plans a fused bucket AllReduce (host only; launches nothing).
 * sendbufs, recvbufs: HOST arrays of ntensors * nranks DEVICE pointers,
 *   entry [k * nranks + r] = tensor k of rank r (counts[k] elements);
 *   recvbufs may equal sendbufs entry by entry (in place, as DDP does).
 * counts: HOST array of ntensors element counts (0 allowed).
 * dtype, order: floats take VC_ORDER_RING only (VC_ERR_UNSUPPORTED
 *   otherwise); integers take every order (their result is the same in every
 *   order), recursive halving with a power-of-two nranks.
 * tiles: HOST array of max_tiles entries receiving the plan, or NULL to ask
 *   for the number of tiles only.
 * *ntiles receives the number of tiles the plan needs, *bucket_count the
 *   bucket's element count.
 * Errors (nothing written to tiles): VC_ERR_INVALID_ARGUMENT for a bad
 * argument, a NULL or misaligned pointer of a non-empty tensor, or
 * max_tiles < *ntiles (with *ntiles still set); VC_ERR_ALIAS when an output
 * range overlaps another output range, or an input range other than its own
 * input in place; VC_ERR_UNSUPPORTED as above. */
vc_status_t vc_bucket_plan(const void *const *sendbufs, void *const *recvbufs,
                           const size_t *counts, int ntensors, int nranks, vc_dtype_t dtype,
                           vc_order_t order, vc_bucket_tile_t *tiles, int max_tiles,
                           int *ntiles, size_t *bucket_count);

/* Runs a plan from vc_bucket_plan in one launch on `stream`.
 * dev_tiles: DEVICE array of the ntiles tiles (8-byte aligned).
 * dev_sendbufs, dev_recvbufs: DEVICE arrays holding the same ntensors *
 *   nranks pointer tables that were planned.
 * bucket_count: the value the plan returned.
 * op: any vc_op_t (AVG divides by nranks).
 * The tables live in device memory, so the library checks only the scalar
 * arguments here; tables that differ from the planned ones are undefined
 * behaviour, as for any device copy.  One guard runs on the device, in all
 * three bucket calls: a tile that does not lie inside [0, bucket_count) and
 * inside one ring chunk of this bucket (tiles planned with another
 * bucket_count or nranks) is skipped, so a mismatched bucket_count leaves
 * those elements unwritten instead of reaching a shard that does not exist.
 * ntiles == 0 launches nothing. */
vc_status_t vc_all_reduce_bucket(const vc_bucket_tile_t *dev_tiles, int ntiles,
                                 const void *const *dev_sendbufs, void *const *dev_recvbufs,
                                 int nranks, size_t bucket_count, vc_dtype_t dtype, vc_op_t op,
                                 vc_stream_t stream);

/* The ReduceScatter of the same bucket, as ZeRO does with gradients ("NCCL
 * 专家课程 07", ZeRO/FSDP 为什么停在 ReduceScatter): rank r receives shard r,
 * the q = vc_shard_count(bucket_count, nranks) elements from bucket index
 * r*q, reduced in ring order: the bits vc_reduce_scatter gives on the
 * packed bucket (the gaps between tensors are zeros, which every op
 * reduces to zero; positions from bucket_count to nranks*q hold the op's
 * identity, 0 for AVG).  One launch; the tensors are read where they are.
 * dev_tiles, dev_sendbufs, bucket_count: as for vc_all_reduce_bucket (the
 *   tiles in the order vc_bucket_plan wrote them).
 * recvbufs: HOST array of nranks DEVICE pointers, shard r of q elements,
 *   pairwise disjoint (checked) and disjoint from the planned tensors (not
 *   checked: those pointers live in device memory).
 * ntiles == 0 launches nothing. */
vc_status_t vc_reduce_scatter_bucket(const vc_bucket_tile_t *dev_tiles, int ntiles,
                                     const void *const *dev_sendbufs, void *const *recvbufs,
                                     int nranks, size_t bucket_count, vc_dtype_t dtype,
                                     vc_op_t op, vc_stream_t stream);

/* The AllGather of the bucket's shards back into the tensors (FSDP's
 * unpack; after vc_reduce_scatter_bucket it completes the decomposed
 * AllReduce of the bucket, with the bits of vc_all_reduce_bucket): element
 * j of tensor k, at bucket index b = b_k + j, receives element b - c*q of
 * shard c = floor(b / q) on every rank.  One launch.
 * dev_tiles, bucket_count: from vc_bucket_plan, planned with the output
 *   tensors (as both sendbufs and recvbufs, or as recvbufs).
 * sendbufs: HOST array of nranks DEVICE pointers, shard r of
 *   q = vc_shard_count(bucket_count, nranks) elements.
 * dev_recvbufs: DEVICE array of the planned output pointer table
 *   ([k * nranks + r]).
 * The shards must not overlap the output tensors (not checked: those
 * pointers live in device memory).  ntiles == 0 launches nothing. */
vc_status_t vc_all_gather_bucket(const vc_bucket_tile_t *dev_tiles, int ntiles,
                                 const void *const *sendbufs, void *const *dev_recvbufs,
                                 int nranks, size_t bucket_count, vc_dtype_t dtype,
                                 vc_stream_t stream);

/* Size of the device scratch array behind vc_all_reduce_decomposed_noalloc:
 * 32 MiB on every GPU where that entry point has been called (or on every GPU
 * the library's context is set up on, with eager module loading), held until
 * the process exits. */
#define VC_NOALLOC_SCRATCH_BYTES (32u << 20)

/* The decomposed AllReduce for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point: the pages' collectives
 * always work on buffers the framework has allocated.
 *
 * Some callers cannot call cudaMalloc where they need the AllReduce: code
 * whose device memory is owned and budgeted by a framework's caching
 * allocator (a raw cudaMalloc would bypass the budget), latency-critical
 * paths that cannot afford cudaMalloc/cudaFree and the synchronisation they
 * imply, or plugins that are handed only their input and output buffers.
 * vc_all_reduce_decomposed needs N shard buffers from its caller; this
 * variant keeps them instead in a scratch array compiled into the library,
 * so the caller passes only sendbufs and recvbufs (same meaning, layout and
 * in-place rule as vc_all_reduce_decomposed) and gets the same bits.  The
 * call allocates nothing.
 *
 * Limit: each of the N shards (q = vc_shard_count(count, nranks) elements)
 * is rounded up to a multiple of 256 bytes, and together they must fit in
 * VC_NOALLOC_SCRATCH_BYTES; a larger count returns VC_ERR_INVALID_ARGUMENT
 * and launches nothing.  (A 25 MiB gradient bucket fits.)
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  The array sits in a device-code
 * module of its own.  With CUDA's lazy module loading (the default on Linux)
 * that module, and with it the 32 MiB, is placed on a device only when it is
 * first needed there: at this first call.  The memory then comes out of the
 * device like any other allocation, so make the first call early, before a
 * caching allocator has filled the GPU; a device that cannot hold the array
 * makes the call return VC_ERR_CUDA.  (With eager loading,
 * CUDA_MODULE_LOADING=EAGER, the array is placed when the library's CUDA
 * context is set up.)  The cached address belongs to the device's primary
 * context: after cudaDeviceReset it is stale, and this entry point must not
 * be called again in that process.
 *
 * Sharing: every call uses the same array, which keeps the shards of the
 * last call.  Nothing in it needs to start at zero: the ReduceScatter writes
 * every shard element, padding included, before the AllGather reads it.
 * Calls that overlap on the GPU (on different streams, or from host threads
 * that do not order their streams) race on the array and corrupt each
 * other's results; serialise them. */
vc_status_t vc_all_reduce_decomposed_noalloc(const void *const *sendbufs, void *const *recvbufs,
                                             int nranks, size_t count, vc_dtype_t dtype,
                                             vc_op_t op, vc_order_t order, vc_stream_t stream);

/* A static, human-readable name for a status code. */
const char *vc_status_string(vc_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* VC_H */
