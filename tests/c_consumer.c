/*
 * A plain C program that uses libdpr through include/dpr.h only -- no Python,
 * no PyTorch -- with device memory from the CUDA runtime.  Built and run by
 * tests/test_gpu_c_consumer.py on a GPU.
 *
 * It runs the worked example of "Ring All-Reduce illustrated" and CMU 11-868
 * Lecture 14 (K = 4 ranks; rank r's chunk c holds (c + 1) * 2^r, so every
 * partial sum is exact and the sum of chunk c is (2^K - 1)(c + 1)) through the
 * reduce-scatter (both summation modes, x 1/K), the all-gather and the
 * all-reduce, with every chunk several tiles long, and checks each result
 * against that closed form.  It also checks that a call with N not a multiple
 * of K is refused without effect.  Prints "C_CONSUMER_OK" and exits 0 on
 * success; prints the first mismatch and exits 1 otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dpr.h"

#define K 4
#define S (3 * 8192 + 40) /* elements per chunk: several tiles and a ragged tail */
#define N (K * S)

static uint16_t bf16_of(float f) { /* exact for the small integers used here */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static float f32_of(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static int fail(const char* what, long i, double got, double want) {
    printf("%s: element %ld is %.9g, want %.9g\n", what, i, got, want);
    return 1;
}

static int check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) {
        printf("%s failed: cudaError %d\n", what, (int)e);
        return 1;
    }
    return 0;
}

int main(void) {
    void *in[K], *out16[K];
    float* shard[K];
    uint16_t* h = (uint16_t*)malloc(N * sizeof(uint16_t));
    float* hf = (float*)malloc(S * sizeof(float));
    if (!h || !hf) return 1;
    for (int r = 0; r < K; ++r) {
        if (check(cudaMalloc(&in[r], N * 2), "cudaMalloc") ||
            check(cudaMalloc(&out16[r], N * 2), "cudaMalloc") ||
            check(cudaMalloc((void**)&shard[r], S * 4), "cudaMalloc"))
            return 1;
        for (long t = 0; t < N; ++t) h[t] = bf16_of((float)((t / S + 1) << r));
        if (check(cudaMemcpy(in[r], h, N * 2, cudaMemcpyHostToDevice), "cudaMemcpy")) return 1;
    }
    const float total = (float)((1 << K) - 1);

    /* reduce-scatter, both modes: shard j = (2^K - 1)(j + 1) / K, exactly */
    for (int mode = DPR_SUM_RING_FP32; mode <= DPR_SUM_HOP_BF16; ++mode) {
        dpr_status st = dpr_reduce_scatter((const void* const*)in, K, 1, N, shard, mode,
                                           1.0f / K, 0, NULL);
        if (st != DPR_OK) {
            printf("dpr_reduce_scatter: %s\n", dpr_strerror(st));
            return 1;
        }
        if (check(cudaDeviceSynchronize(), "synchronize")) return 1;
        for (int j = 0; j < K; ++j) {
            if (check(cudaMemcpy(hf, shard[j], S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
            const float want = total * (float)(j + 1) / K;
            for (long t = 0; t < S; ++t)
                if (hf[t] != want) return fail("reduce-scatter", t, hf[t], want);
        }
    }

    /* all-gather of bf16 shards: shard j = bf16 of chunk j of rank 0's buffer */
    {
        const void* sh[K];
        for (int j = 0; j < K; ++j) sh[j] = (const uint16_t*)in[0] + (long)j * S;
        dpr_status st = dpr_allgather(sh, K, N, out16, NULL);
        if (st != DPR_OK) {
            printf("dpr_allgather: %s\n", dpr_strerror(st));
            return 1;
        }
        if (check(cudaDeviceSynchronize(), "synchronize")) return 1;
        for (int r = 0; r < K; ++r) {
            if (check(cudaMemcpy(h, out16[r], N * 2, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
            for (long t = 0; t < N; ++t)
                if (f32_of(h[t]) != (float)(t / S + 1))
                    return fail("all-gather", t, f32_of(h[t]), (double)(t / S + 1));
        }
    }

    /* all-reduce (sum, scale 1): every replica holds (2^K - 1)(c + 1) */
    {
        dpr_status st = dpr_allreduce((const void* const*)in, K, N, out16, DPR_SUM_RING_FP32,
                                      1.0f, NULL);
        if (st != DPR_OK) {
            printf("dpr_allreduce: %s\n", dpr_strerror(st));
            return 1;
        }
        if (check(cudaDeviceSynchronize(), "synchronize")) return 1;
        for (int r = 0; r < K; ++r) {
            if (check(cudaMemcpy(h, out16[r], N * 2, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
            for (long t = 0; t < N; ++t) {
                const float want = total * (float)(t / S + 1);
                if (f32_of(h[t]) != want) return fail("all-reduce", t, f32_of(h[t]), want);
            }
        }
    }

    /* N not a multiple of K: refused, nothing written */
    {
        if (check(cudaMemcpy(hf, shard[0], S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
        const float before = hf[0];
        dpr_status st = dpr_reduce_scatter((const void* const*)in, K, 1, N - 1, shard,
                                           DPR_SUM_RING_FP32, 1.0f / K, 0, NULL);
        if (st != DPR_ERR_INVALID_ARG) {
            printf("N %% K != 0 returned %d, want DPR_ERR_INVALID_ARG\n", (int)st);
            return 1;
        }
        if (check(cudaDeviceSynchronize(), "synchronize")) return 1;
        if (check(cudaMemcpy(hf, shard[0], S * 4, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
        if (hf[0] != before) return fail("refused call wrote", 0, hf[0], before);
    }

    for (int r = 0; r < K; ++r) {
        cudaFree(in[r]);
        cudaFree(out16[r]);
        cudaFree(shard[r]);
    }
    free(h);
    free(hf);
    printf("C_CONSUMER_OK %s\n", dpr_version());
    return 0;
}
