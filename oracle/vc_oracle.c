/*
 * Plain CPU oracle for AllReduce / ReduceScatter / AllGather over N virtual
 * ranks.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline (and its reference arm) may load this library.  It shares no code,
 * header or constant with the CUDA library; it is slow on purpose and written
 * to be checked against the pages by eye: one element at a time, every
 * operand read from a (virtually) padded buffer, the reduction order spelled
 * out as the schedule that defines it.
 *
 * Sources (page title, section):
 *  - "NCCL 专家课程 07：AllReduce 等价分解、显存生命周期与 Kernel 证据",
 *    section 数学证明: y_i = (+)_s x^(s)_i (Direct AllReduce),
 *    z^(r)_j = (+)_s x^(s)_{rq+j} (ReduceScatter, rank-major shards),
 *    yhat^(r)_{sq+j} = z^(s)_j (AllGather, source-rank-major).
 *  - same page, 等价成立的条件 条件三: q = ceil(M/N), pad to Nq with the
 *    reduction identity (MAX: the dtype's minimum / -inf, never 0), trim to M.
 *  - same page, 条件五: floating-point reduction is not associative, so the
 *    order is part of the result; the arithmetic is in the buffer's type.
 *  - "通信与互联（01）：集合通信原语与代价模型", 二.1: op set
 *    {sum, max, min, prod, avg}.
 *  - ring order: "Ring AllReduce 核心流程" (pseudocode: the chunk a rank sends
 *    at step s is (rank - s) mod N, the receiver adds it into its own copy) and
 *    "通信与互联（01）" 五.2 (rule: at step s rank r sends chunk (r-s+1) mod N;
 *    rank r ends owning chunk (r+1) mod N).  Chunk c therefore starts at rank
 *    c and picks up ranks c+1, c+2, ... c+N-1 (mod N), one per step.
 *  - recursive halving: "ReduceScatter" page, Recursive Halving table: step j
 *    pairs ranks at distance N/2^j ((0,4)(1,5)(2,6)(3,7), then (0,2)..., then
 *    (0,1)... for N=8); needs N = 2^k.
 *  - tree: "通信与互联（01）" 六.1 figure: rank 0 is the root with one child,
 *    a rank's level is the lowest set bit of its number, odd ranks are leaves;
 *    an inner node receives both children, adds itself, sends to its parent;
 *    the tree is binary and takes 2*ceil(log2 N) steps.
 *  - double binary tree: same page, 六.3: two trees, each carrying half of the
 *    data; for even N the second is the first with every rank number shifted
 *    by one, for odd N its mirror image.
 *
 * Readings where the pages are silent:
 *  - integer ops accumulate in 64 bits and wrap modulo 2^64 (int32 results
 *    are the low 32 bits);
 *  - AVG is the SUM in the chosen order followed by one division by N: an
 *    IEEE single division for float/bf16, C truncation toward zero for ints;
 *    its padding value is 0;
 *  - bf16 operands are widened exactly to fp32, accumulated in fp32 and
 *    rounded once, to nearest-even, at the store;
 *  - MAX/MIN keep the running value on ties;
 *  - tree inner node: (left subtree (+) right subtree) (+) own value, the
 *    lower-numbered child on the left (parity unpinned: the pages fix only
 *    the tree's shape);
 *  - recursive halving is defined for N a power of two only;
 *  - tree with N not a power of two: a rank whose parent label (r - L) | 2L
 *    is not a rank (>= N) hangs under r - L instead.  This keeps what the
 *    figure states for every N (a binary tree, a root with one child, odd
 *    ranks as leaves, depth ceil(log2 N)), and it is the tree of the next
 *    power of two with the missing ranks passing their one subtree through;
 *  - double binary tree: tree A reduces the first ceil(M/2) elements of the
 *    buffer, tree B the rest, padding included; in tree B node k is played
 *    by rank (k+1) mod N (even N) or N-1-k (odd N).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { OR_INT32 = 0, OR_INT64 = 1, OR_FLOAT32 = 2, OR_BFLOAT16 = 3 };
enum { OR_SUM = 0, OR_PROD = 1, OR_MAX = 2, OR_MIN = 3, OR_AVG = 4 };
enum { OR_RING = 0, OR_RECURSIVE_HALVING = 1, OR_PAIRWISE_TREE = 2,
       OR_SEQUENTIAL = 3, OR_DOUBLE_TREE = 4 };

enum { OR_OK = 0, OR_BAD_ARGUMENT = -1, OR_UNSUPPORTED = -2, OR_NO_MEMORY = -3 };

#define OR_MAX_RANKS 64

/* One operand or partial result: an int64 for the integer types, an IEEE
 * single for float32 and bfloat16. */
typedef struct {
    int is_float;
    int64_t i;
    float f;
} val_t;

static int elem_size(int dtype)
{
    switch (dtype) {
    case OR_INT32: return 4;
    case OR_INT64: return 8;
    case OR_FLOAT32: return 4;
    case OR_BFLOAT16: return 2;
    default: return 0;
    }
}

static int is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

/* ---- bfloat16 <-> float32 ------------------------------------------------ */

/* bf16 is the upper half of an IEEE single: widening is exact. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an IEEE single to bf16, to nearest with ties to even: keep the upper
 * 16 bits, and add one unit in their last place when the dropped lower half
 * is above one half, or exactly one half with an odd kept part.  A carry out
 * of the mantissa moves into the exponent, which rounds the largest finite
 * values up to infinity as IEEE rounding does.  NaN stays a (quiet) NaN. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ---- operands ------------------------------------------------------------ */

static val_t load(int dtype, const void *buf, int64_t idx)
{
    val_t v = {0, 0, 0.0f};
    const unsigned char *p = (const unsigned char *)buf;
    switch (dtype) {
    case OR_INT32: {
        int32_t t;
        memcpy(&t, p + idx * 4, 4);
        v.i = t;
        break;
    }
    case OR_INT64: {
        int64_t t;
        memcpy(&t, p + idx * 8, 8);
        v.i = t;
        break;
    }
    case OR_FLOAT32: {
        float t;
        memcpy(&t, p + idx * 4, 4);
        v.is_float = 1;
        v.f = t;
        break;
    }
    case OR_BFLOAT16: {
        uint16_t t;
        memcpy(&t, p + idx * 2, 2);
        v.is_float = 1;
        v.f = bf16_to_float(t);
        break;
    }
    }
    return v;
}

static void store(int dtype, void *buf, int64_t idx, val_t v)
{
    unsigned char *p = (unsigned char *)buf;
    switch (dtype) {
    case OR_INT32: {
        /* low 32 bits, two's complement */
        uint32_t t = (uint32_t)(uint64_t)v.i;
        memcpy(p + idx * 4, &t, 4);
        break;
    }
    case OR_INT64: {
        int64_t t = v.i;
        memcpy(p + idx * 8, &t, 8);
        break;
    }
    case OR_FLOAT32: {
        float t = v.f;
        memcpy(p + idx * 4, &t, 4);
        break;
    }
    case OR_BFLOAT16: {
        uint16_t t = float_to_bf16_rne(v.f);
        memcpy(p + idx * 2, &t, 2);
        break;
    }
    }
}

/* The identity e(op, dtype) used for the padding (条件三): 0 for SUM and AVG,
 * 1 for PROD, the smallest value (-inf for floats) for MAX, the largest
 * (+inf) for MIN. */
static val_t identity(int dtype, int op)
{
    val_t v = {0, 0, 0.0f};
    v.is_float = (dtype == OR_FLOAT32 || dtype == OR_BFLOAT16);
    switch (op) {
    case OR_SUM:
    case OR_AVG:
        v.i = 0;
        v.f = 0.0f;
        break;
    case OR_PROD:
        v.i = 1;
        v.f = 1.0f;
        break;
    case OR_MAX:
        v.i = (dtype == OR_INT32) ? (int64_t)INT32_MIN : INT64_MIN;
        v.f = -INFINITY;
        break;
    case OR_MIN:
        v.i = (dtype == OR_INT32) ? (int64_t)INT32_MAX : INT64_MAX;
        v.f = INFINITY;
        break;
    }
    return v;
}

/* a (+) b.  Integers wrap modulo 2^64 (computed unsigned); floats are single
 * precision IEEE operations; MAX/MIN keep a on ties. */
static val_t combine(int op, val_t a, val_t b)
{
    val_t r = a;
    if (a.is_float) {
        switch (op) {
        case OR_SUM:
        case OR_AVG: r.f = a.f + b.f; break;
        case OR_PROD: r.f = a.f * b.f; break;
        case OR_MAX: r.f = (b.f > a.f) ? b.f : a.f; break;
        case OR_MIN: r.f = (b.f < a.f) ? b.f : a.f; break;
        }
    } else {
        switch (op) {
        case OR_SUM:
        case OR_AVG: r.i = (int64_t)((uint64_t)a.i + (uint64_t)b.i); break;
        case OR_PROD: r.i = (int64_t)((uint64_t)a.i * (uint64_t)b.i); break;
        case OR_MAX: r.i = (b.i > a.i) ? b.i : a.i; break;
        case OR_MIN: r.i = (b.i < a.i) ? b.i : a.i; break;
        }
    }
    return r;
}

/* AVG: the sum divided by N once, after the reduction. */
static val_t epilogue(int op, int n, val_t v)
{
    if (op != OR_AVG)
        return v;
    if (v.is_float)
        v.f = v.f / (float)n;
    else
        v.i = v.i / (int64_t)n;
    return v;
}

/* ---- reduction orders ---------------------------------------------------- */

/* Left fold in rank order 0, 1, ..., N-1: the plain reading of the sum in
 * y_i = (+)_{s=0}^{N-1} x^(s)_i.  Not one of the library's orders; kept to
 * compare the others against. */
static val_t fold_sequential(int op, const val_t *a, int n)
{
    val_t acc = a[0];
    for (int s = 1; s < n; ++s)
        acc = combine(op, acc, a[s]);
    return acc;
}

/* Ring: the partial sum of chunk c leaves rank c at step 1 and every later
 * holder c+1, c+2, ... adds its own operand, so the value is
 * (((a_c (+) a_{c+1}) (+) a_{c+2}) ... (+) a_{c+N-1}), indices mod N. */
static val_t fold_ring(int op, const val_t *a, int n, int c)
{
    val_t acc = a[c];
    for (int k = 1; k < n; ++k)
        acc = combine(op, acc, a[(c + k) % n]);
    return acc;
}

/* Recursive halving: P_0[s] = a_s; at step j = 1..log2 N partners s and
 * s XOR N/2^j combine, P_j[s] = P_{j-1}[s] (+) P_{j-1}[s XOR N/2^j].  The
 * lower partner keeps the lower half of the chunks, so chunk r ends at rank
 * r and its value is P_{log2 N}[r]. */
static val_t fold_recursive_halving(int op, const val_t *a, int n, int owner)
{
    val_t p[OR_MAX_RANKS], next[OR_MAX_RANKS];
    for (int s = 0; s < n; ++s)
        p[s] = a[s];
    for (int d = n / 2; d >= 1; d /= 2) {
        for (int s = 0; s < n; ++s)
            next[s] = combine(op, p[s], p[s ^ d]);
        for (int s = 0; s < n; ++s)
            p[s] = next[s];
    }
    return p[owner];
}

/* Tree shape: a rank's level is its lowest set bit L; its parent is the rank
 * one level up whose subtree contains it, (r - L) | 2L.  Where that label is
 * not a rank (>= N) the parent is r - L: with N = 2^k this happens only for
 * rank N/2, which hangs under the root, rank 0. */
static int tree_parent(int r, int n)
{
    int low = r & -r;
    int p = (r - low) | (low << 1);
    return p < n ? p : r - low;
}

typedef struct {
    int count[OR_MAX_RANKS];
    int child[OR_MAX_RANKS][OR_MAX_RANKS];
} tree_t;

static void tree_build(tree_t *t, int n)
{
    memset(t, 0, sizeof *t);
    for (int r = 1; r < n; ++r) {
        int p = tree_parent(r, n);
        t->child[p][t->count[p]++] = r; /* children in increasing rank */
    }
}

/* Subtree value: the children's values combined first (lower rank on the
 * left), then the node's own operand; a leaf is its own operand. */
static val_t fold_tree_node(int op, const val_t *a, const tree_t *t, int p)
{
    if (t->count[p] == 0)
        return a[p];
    val_t acc = fold_tree_node(op, a, t, t->child[p][0]);
    for (int k = 1; k < t->count[p]; ++k)
        acc = combine(op, acc, fold_tree_node(op, a, t, t->child[p][k]));
    return combine(op, acc, a[p]);
}

/* ---- one output element -------------------------------------------------- */

typedef struct {
    int n;
    int64_t M;
    int64_t q;
    int dtype;
    int op;
    int order;
    tree_t tree;
} plan_t;

static int plan_init(plan_t *pl, int n, int64_t M, int dtype, int op, int order)
{
    if (n < 1 || n > OR_MAX_RANKS || M < 0 || elem_size(dtype) == 0)
        return OR_BAD_ARGUMENT;
    if (op < OR_SUM || op > OR_AVG)
        return OR_BAD_ARGUMENT;
    if (order < OR_RING || order > OR_DOUBLE_TREE)
        return OR_BAD_ARGUMENT;
    if (order == OR_RECURSIVE_HALVING && !is_pow2(n))
        return OR_UNSUPPORTED;
    pl->n = n;
    pl->M = M;
    pl->q = (M + n - 1) / n;
    pl->dtype = dtype;
    pl->op = op;
    pl->order = order;
    if (order == OR_PAIRWISE_TREE || order == OR_DOUBLE_TREE)
        tree_build(&pl->tree, n);
    return OR_OK;
}

/* Reduce the N operands a[0..N-1] of global index i (already padded). */
static val_t reduce_operands(const plan_t *pl, const val_t *a, int64_t i)
{
    int c = (pl->q > 0) ? (int)(i / pl->q) : 0; /* chunk = shard owner */
    val_t v;
    switch (pl->order) {
    case OR_RING: v = fold_ring(pl->op, a, pl->n, c); break;
    case OR_RECURSIVE_HALVING: v = fold_recursive_halving(pl->op, a, pl->n, c); break;
    case OR_PAIRWISE_TREE: v = fold_tree_node(pl->op, a, &pl->tree, 0); break;
    case OR_DOUBLE_TREE:
        if (i < (pl->M + 1) / 2) {
            v = fold_tree_node(pl->op, a, &pl->tree, 0); /* tree A */
        } else {
            /* tree B: the same tree with node k played by rank (k+1) mod N
             * (even N) or by rank N-1-k (odd N) */
            val_t b[OR_MAX_RANKS];
            for (int k = 0; k < pl->n; ++k)
                b[k] = a[(pl->n % 2 == 0) ? (k + 1) % pl->n : pl->n - 1 - k];
            v = fold_tree_node(pl->op, b, &pl->tree, 0);
        }
        break;
    default: v = fold_sequential(pl->op, a, pl->n); break;
    }
    return epilogue(pl->op, pl->n, v);
}

/* Element i of the padded logical buffer of every rank: x^(s)_i for i < M,
 * the identity for M <= i < Nq. */
static val_t reduce_index(const plan_t *pl, const void *const *x, int64_t i)
{
    val_t a[OR_MAX_RANKS];
    for (int s = 0; s < pl->n; ++s)
        a[s] = (i < pl->M) ? load(pl->dtype, x[s], i) : identity(pl->dtype, pl->op);
    return reduce_operands(pl, a, i);
}

/* ---- exported entry points ----------------------------------------------- */

int64_t oracle_shard_count(int64_t M, int n)
{
    if (n < 1 || M < 0)
        return -1;
    return (M + n - 1) / n;
}

int oracle_element_size(int dtype) { return elem_size(dtype); }

int oracle_identity(int dtype, int op, void *out)
{
    if (elem_size(dtype) == 0 || op < OR_SUM || op > OR_AVG)
        return OR_BAD_ARGUMENT;
    store(dtype, out, 0, identity(dtype, op));
    return OR_OK;
}

/* ReduceScatter: z^(r)_j = (+)_s x^(s)_{rq+j}, 0 <= j < q; positions with
 * rq+j >= M reduce the padding and hold the identity (0 for AVG). */
int oracle_reduce_scatter(const void *const *x, void *const *z, int n, int64_t M,
                          int dtype, int op, int order)
{
    plan_t pl;
    int rc = plan_init(&pl, n, M, dtype, op, order);
    if (rc != OR_OK)
        return rc;
    for (int r = 0; r < n; ++r)
        for (int64_t j = 0; j < pl.q; ++j)
            store(dtype, z[r], j, reduce_index(&pl, x, r * pl.q + j));
    return OR_OK;
}

/* AllGather: yhat^(r)_{sq+j} = z^(s)_j for every destination r, kept only
 * where sq+j < M (trim). */
int oracle_all_gather(const void *const *z, void *const *y, int n, int64_t M, int dtype)
{
    if (n < 1 || n > OR_MAX_RANKS || M < 0 || elem_size(dtype) == 0)
        return OR_BAD_ARGUMENT;
    int64_t q = (M + n - 1) / n;
    for (int r = 0; r < n; ++r)
        for (int s = 0; s < n; ++s)
            for (int64_t j = 0; j < q && s * q + j < M; ++j)
                store(dtype, y[r], s * q + j, load(dtype, z[s], j));
    return OR_OK;
}

/* Direct AllReduce: y^(r)_i = (+)_s x^(s)_i for every r, 0 <= i < M. */
int oracle_all_reduce(const void *const *x, void *const *y, int n, int64_t M,
                      int dtype, int op, int order)
{
    plan_t pl;
    int rc = plan_init(&pl, n, M, dtype, op, order);
    if (rc != OR_OK)
        return rc;
    for (int64_t i = 0; i < M; ++i) {
        val_t v = reduce_index(&pl, x, i);
        for (int r = 0; r < n; ++r)
            store(dtype, y[r], i, v);
    }
    return OR_OK;
}

/* AllReduce as ReduceScatter into the N shard buffers (q elements each)
 * followed by AllGather from them. */
int oracle_all_reduce_decomposed(const void *const *x, void *const *shards, void *const *y,
                                 int n, int64_t M, int dtype, int op, int order)
{
    int rc = oracle_reduce_scatter(x, shards, n, M, dtype, op, order);
    if (rc != OR_OK)
        return rc;
    return oracle_all_gather((const void *const *)shards, y, n, M, dtype);
}

/* Reduce to one buffer (the root's): y_i = (+)_s x^(s)_i, the AllReduce
 * value of every element ("通信与互联（01）" 二.1, reduce with root 0). */
int oracle_reduce(const void *const *x, void *y, int n, int64_t M, int dtype, int op, int order)
{
    plan_t pl;
    int rc = plan_init(&pl, n, M, dtype, op, order);
    if (rc != OR_OK)
        return rc;
    for (int64_t i = 0; i < M; ++i)
        store(dtype, y, i, reduce_index(&pl, x, i));
    return OR_OK;
}

/* Broadcast from the root's buffer: y^(r)_i = x_i for every r (same page,
 * broadcast with root 0). */
int oracle_broadcast(const void *x, void *const *y, int n, int64_t M, int dtype)
{
    if (n < 1 || n > OR_MAX_RANKS || M < 0 || elem_size(dtype) == 0)
        return OR_BAD_ARGUMENT;
    for (int r = 0; r < n; ++r)
        for (int64_t i = 0; i < M; ++i)
            store(dtype, y[r], i, load(dtype, x, i));
    return OR_OK;
}

/* Reduce selected global indices only.  xs[s] holds the K operands of rank s
 * at indices idx[0..K-1] (gathered by the caller; an index >= M takes the
 * identity whatever xs holds there); out receives the K results. */
int oracle_reduce_points(const void *const *xs, const int64_t *idx, int64_t K, int n,
                         int64_t M, int dtype, int op, int order, void *out)
{
    plan_t pl;
    int rc = plan_init(&pl, n, M, dtype, op, order);
    if (rc != OR_OK)
        return rc;
    val_t a[OR_MAX_RANKS];
    for (int64_t k = 0; k < K; ++k) {
        int64_t i = idx[k];
        if (i < 0 || i >= (int64_t)n * pl.q)
            return OR_BAD_ARGUMENT;
        for (int s = 0; s < n; ++s)
            a[s] = (i < M) ? load(dtype, xs[s], k) : identity(dtype, op);
        store(dtype, out, k, reduce_operands(&pl, a, i));
    }
    return OR_OK;
}

/* fp32 -> bf16 rounding as the oracle does it, exposed for its own pins. */
void oracle_bf16_round(const float *in, uint16_t *out, int64_t K)
{
    for (int64_t k = 0; k < K; ++k)
        out[k] = float_to_bf16_rne(in[k]);
}

/* Tree parent table (for the shape pin): parent[r] for r in 1..N-1, -1 for
 * the root. */
int oracle_tree_parents(int n, int *parent)
{
    if (n < 1 || n > OR_MAX_RANKS)
        return OR_BAD_ARGUMENT;
    parent[0] = -1;
    for (int r = 1; r < n; ++r)
        parent[r] = tree_parent(r, n);
    return OR_OK;
}
