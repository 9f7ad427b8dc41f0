/*
 * The C ABI from plain C (no C++, no Python): compiled with gcc -std=c11
 * against include/vc.h and linked with libvc.so.
 *
 *   vc_from_c checks   argument checks only (no GPU needed; run with
 *                      VC_TEST_FAIL_LAUNCH=1 so a call that passes its
 *                      checks reports VC_ERR_CUDA instead of launching)
 *   vc_from_c run      the worked example of "NCCL 专家课程 07" (4 ranks,
 *                      20 int64, x = 100r + i: every output 600 + 4i, shard
 *                      r = 600 + 4(5r + j)) through vc_all_reduce,
 *                      vc_reduce_scatter and vc_all_gather on device memory
 *                      from cudaMalloc
 *
 * Exit status 0 on success; prints the first failure otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "vc.h"

#ifdef VC_WITH_CUDA
#include <cuda_runtime_api.h>
#endif

static int fail(const char *what, long a, long b)
{
    printf("FAIL %s: %ld != %ld\n", what, a, b);
    return 1;
}

static int checks(void)
{
    void *send[4], *recv[4];
    for (int r = 0; r < 4; ++r) {
        send[r] = (void *)(uintptr_t)(((uintptr_t)1 << 40) + ((uintptr_t)r << 24));
        recv[r] = (void *)(uintptr_t)(((uintptr_t)1 << 41) + ((uintptr_t)r << 24));
    }
    if (vc_shard_count(1003, 4) != 251) return fail("shard count", (long)vc_shard_count(1003, 4), 251);
    if (vc_all_reduce((const void *const *)send, recv, 0, 100, VC_FLOAT32, VC_SUM,
                      VC_ORDER_RING, NULL) != VC_ERR_INVALID_ARGUMENT)
        return fail("nranks 0", 0, VC_ERR_INVALID_ARGUMENT);
    if (vc_all_reduce((const void *const *)send, recv, 3, 100, VC_FLOAT32, VC_SUM,
                      VC_ORDER_RECURSIVE_HALVING, NULL) != VC_ERR_UNSUPPORTED)
        return fail("recursive halving, 3 ranks", 0, VC_ERR_UNSUPPORTED);
    void *alias[4] = {recv[0], recv[1], recv[1], recv[3]};
    if (vc_all_reduce((const void *const *)send, alias, 4, 100, VC_FLOAT32, VC_SUM,
                      VC_ORDER_RING, NULL) != VC_ERR_ALIAS)
        return fail("aliased outputs", 0, VC_ERR_ALIAS);
    if (vc_all_reduce((const void *const *)send, recv, 4, 100, VC_FLOAT32, VC_SUM,
                      VC_ORDER_RING, NULL) != VC_ERR_CUDA)
        return fail("launch hook", 0, VC_ERR_CUDA);
    if (vc_all_reduce((const void *const *)send, recv, 4, 0, VC_FLOAT32, VC_SUM, VC_ORDER_RING,
                      NULL) != VC_SUCCESS)
        return fail("count 0", 0, VC_SUCCESS);
    if (strlen(vc_status_string(VC_ERR_ALIAS)) == 0) return fail("status string", 0, 1);
    printf("checks ok\n");
    return 0;
}

#ifdef VC_WITH_CUDA
static int run(void)
{
    enum { N = 4, M = 20, Q = 5 };
    int64_t host[N][M], out[M], shard[Q];
    void *x[N], *y[N], *z[N], *g[N];
    for (int r = 0; r < N; ++r) {
        for (int i = 0; i < M; ++i) host[r][i] = 100 * r + i;
        if (cudaMalloc(&x[r], sizeof host[r]) != cudaSuccess ||
            cudaMalloc(&y[r], sizeof host[r]) != cudaSuccess ||
            cudaMalloc(&z[r], sizeof shard) != cudaSuccess ||
            cudaMalloc(&g[r], sizeof host[r]) != cudaSuccess)
            return fail("cudaMalloc", 0, 0);
        cudaMemcpy(x[r], host[r], sizeof host[r], cudaMemcpyHostToDevice);
    }
    vc_status_t s = vc_all_reduce((const void *const *)x, y, N, M, VC_INT64, VC_SUM,
                                  VC_ORDER_RING, NULL);
    if (s != VC_SUCCESS) return fail("vc_all_reduce", s, VC_SUCCESS);
    s = vc_reduce_scatter((const void *const *)x, z, N, M, VC_INT64, VC_SUM, VC_ORDER_RING, NULL);
    if (s != VC_SUCCESS) return fail("vc_reduce_scatter", s, VC_SUCCESS);
    s = vc_all_gather((const void *const *)z, g, N, M, VC_INT64, NULL);
    if (s != VC_SUCCESS) return fail("vc_all_gather", s, VC_SUCCESS);
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("cudaDeviceSynchronize", 0, 0);
    for (int r = 0; r < N; ++r) {
        cudaMemcpy(out, y[r], sizeof out, cudaMemcpyDeviceToHost);
        for (int i = 0; i < M; ++i)
            if (out[i] != 600 + 4 * i) return fail("AllReduce element", (long)out[i], 600 + 4 * i);
        cudaMemcpy(shard, z[r], sizeof shard, cudaMemcpyDeviceToHost);
        for (int j = 0; j < Q; ++j)
            if (shard[j] != 600 + 4 * (Q * r + j))
                return fail("ReduceScatter shard", (long)shard[j], 600 + 4 * (Q * r + j));
        cudaMemcpy(out, g[r], sizeof out, cudaMemcpyDeviceToHost);
        for (int i = 0; i < M; ++i)
            if (out[i] != 600 + 4 * i) return fail("AllGather element", (long)out[i], 600 + 4 * i);
    }
    for (int r = 0; r < N; ++r) {
        cudaFree(x[r]);
        cudaFree(y[r]);
        cudaFree(z[r]);
        cudaFree(g[r]);
    }
    printf("run ok\n");
    return 0;
}
#endif

int main(int argc, char **argv)
{
    if (argc > 1 && strcmp(argv[1], "checks") == 0) return checks();
#ifdef VC_WITH_CUDA
    if (argc > 1 && strcmp(argv[1], "run") == 0) return run();
#endif
    printf("usage: vc_from_c checks|run\n");
    return 2;
}
