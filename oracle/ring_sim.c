/*
 * Ring simulation in plain C -- ORACLE, TEST INFRASTRUCTURE.
 *
 * A second CPU statement of what the ZeRO gradient-bucket reduction computes,
 * written in C so that the host's cores run it faster than numpy.  Like the
 * numpy oracle beside it, it follows the pages round by round and shares no
 * code with the CUDA library; only the test suite, the package smoke check and
 * the bench's CPU legs load it.
 *
 * The ring (CMU 11-868 Lecture 14 notes, section 3.2; "Ring All-Reduce
 * illustrated", Phases 1 and 2).  K ranks, each with a buffer of N elements
 * cut into K chunks of S = N / K; rank r sends to rank (r + 1) mod K.
 *   Reduce-scatter, rounds i = 0 .. K-2: every rank r copies its chunk
 *   (r - i) mod K into the message on its outgoing link; then every
 *   receiver adds the message that reached it to its own copy of that chunk.
 *   After K - 1 rounds rank r holds the complete sum of chunk (r + 1) mod K,
 *   so chunk j is summed in ring order x_j, x_{j+1}, ..., x_{j-1}.
 *   All-gather, rounds i = 0 .. K-2: a rank holding complete chunk (r + d)
 *   mod K sends chunk (r + d - i) mod K and the receiver overwrites its copy
 *   (d = 1 after a reduce-scatter, d = 0 when rank r starts from shard r).
 * Modes ("bf16 communication", DeepSpeed issue 8364):
 *   RING_FP32 (0): rank copies and messages are binary32, one round-to-
 *                  nearest-even add per hop;
 *   HOP_BF16  (1): rank copies and messages are bf16, each hop's binary32
 *                  sum is rounded back to bf16.
 * Micro-batches (lecture section 4.2): each rank first adds its own bf16
 * micro-batch gradients left to right, rounding to bf16 after each add.
 * Average and partition write (lecture section 4.1; DeepSpeed ZeRO-3 source
 * walkthrough, sections 5.2-5.3): the landed sum of chunk j is multiplied once
 * by the fp32 scale and written to partition slot j (copy_), or added to it
 * (add_) with `accumulate`.
 * All-reduce (lecture section 2.2): reduce-scatter, then the landing rank
 * scales its complete chunk and rounds it to bf16, then the all-gather.
 * Flat-bucket gather (ZeRO-3 walkthrough, sections 3.2 and 5.1): gradient p
 * of rank r goes to [offset_p, offset_p + numel_p) of rank r's flat bucket.
 *
 * Arithmetic.  Built with -O2 -ffp-contract=off (no fused multiply-add) and
 * without fast-math, every float operation below is one IEEE binary32
 * operation rounded to nearest even, with subnormals kept.  bf16 rounding is
 * done on the bit pattern from its definition.  Within one round every
 * element is independent of every other, so the element loops of a round may
 * run on several threads (OpenMP) without changing any result.
 *
 * Status codes: 0 ok, 1 invalid argument, 2 out of host memory.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define RING_FP32 0
#define HOP_BF16 1

/* ---- bf16 bit conversions ---------------------------------------------------
 * bf16 is the upper half of a binary32.  Widening appends 16 zero bits.
 * Narrowing rounds the dropped 16 bits to nearest, ties to the even result;
 * a NaN becomes the quiet NaN 0x7FC0. */
static float widen(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t narrow(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    const uint32_t low = u & 0xFFFFu;      /* the dropped bits */
    const uint32_t high = u >> 16;
    /* round up past the halfway point, or at it when the kept part is odd; a
     * carry moves into the exponent as IEEE rounding does (up to infinity).
     * Bitwise & and | rather than && and ||: no data-dependent branch. */
    const uint32_t up = (uint32_t)(low > 0x8000u) | ((uint32_t)(low == 0x8000u) & high & 1u);
    return (uint16_t)(high + up);
}

static uint16_t add_bf16(uint16_t a, uint16_t b) { return narrow(widen(a) + widen(b)); }

static int mod(int a, int K) { return ((a % K) + K) % K; }

/* One rank's buffer: binary32 values (RING_FP32) or bf16 bits (HOP_BF16). */
typedef struct {
    float* f;
    uint16_t* h;
} rank_buf;

static void free_ranks(rank_buf* st, int K) {
    if (!st) return;
    for (int r = 0; r < K; ++r) {
        free(st[r].f);
        free(st[r].h);
    }
    free(st);
}

/* Rank-local gradient accumulation over M micro-batches, then the rank's
 * starting buffer in the ring's mode. */
static rank_buf* initial_state(int K, int M, int64_t N, const uint16_t* const* x, int mode) {
    rank_buf* st = (rank_buf*)calloc((size_t)K, sizeof *st);
    if (!st) return NULL;
    for (int r = 0; r < K; ++r) {
        uint16_t* g = (uint16_t*)malloc((size_t)N * sizeof *g);
        if (!g) { free_ranks(st, K); return NULL; }
        const uint16_t* x0 = x[r];
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < N; ++t) {
            uint16_t v = x0[t];
            for (int m = 1; m < M; ++m) v = add_bf16(v, x[m * K + r][t]);
            g[t] = v;
        }
        if (mode == HOP_BF16) {
            st[r].h = g;
        } else {
            st[r].f = (float*)malloc((size_t)N * sizeof(float));
            if (!st[r].f) { free(g); free_ranks(st, K); return NULL; }
#pragma omp parallel for schedule(static)
            for (int64_t t = 0; t < N; ++t) st[r].f[t] = widen(g[t]);
            free(g);
        }
    }
    return st;
}

/* K - 1 reduce-scatter rounds with explicit per-link messages. */
static int rs_rounds(rank_buf* st, int K, int64_t S, int mode, int64_t* counters) {
    /* msg[r]: what rank r put on its link to rank r + 1 this round */
    void** msg = (void**)calloc((size_t)K, sizeof *msg);
    if (!msg) return 2;
    const size_t esz = mode == HOP_BF16 ? sizeof(uint16_t) : sizeof(float);
    for (int r = 0; r < K; ++r) {
        msg[r] = malloc((size_t)S * esz);
        if (!msg[r]) {
            for (int q = 0; q < r; ++q) free(msg[q]);
            free(msg);
            return 2;
        }
    }
    for (int i = 0; i < K - 1; ++i) {
        for (int r = 0; r < K; ++r) {                       /* sends */
            const int64_t c = mod(r - i, K);
            if (mode == HOP_BF16) memcpy(msg[r], st[r].h + c * S, (size_t)S * esz);
            else memcpy(msg[r], st[r].f + c * S, (size_t)S * esz);
            if (counters) counters[1 + r] += S;
        }
        for (int r = 0; r < K; ++r) {                       /* receives */
            const int dst = (r + 1) % K;
            const int64_t c = mod(r - i, K);
            if (mode == HOP_BF16) {
                uint16_t* mine = st[dst].h + c * S;
                const uint16_t* in = (const uint16_t*)msg[r];
#pragma omp parallel for schedule(static)
                for (int64_t t = 0; t < S; ++t) mine[t] = add_bf16(mine[t], in[t]);
            } else {
                float* mine = st[dst].f + c * S;
                const float* in = (const float*)msg[r];
#pragma omp parallel for schedule(static)
                for (int64_t t = 0; t < S; ++t) mine[t] = mine[t] + in[t];
            }
        }
        if (counters) counters[0] += 1;
    }
    for (int r = 0; r < K; ++r) free(msg[r]);
    free(msg);
    return 0;
}

/* The complete sum of chunk j, element t, from the rank it landed on. */
static float landed(const rank_buf* st, int K, int64_t S, int j, int64_t t, int mode) {
    const rank_buf* b = &st[mod(j - 1, K)];
    return mode == HOP_BF16 ? widen(b->h[j * S + t]) : b->f[j * S + t];
}

/* K - 1 all-gather rounds on bf16 buffers: overwrite, no reduction. */
static int ag_rounds(uint16_t** buf, int K, int64_t S, int d, int64_t* counters) {
    uint16_t** msg = (uint16_t**)calloc((size_t)K, sizeof *msg);
    if (!msg) return 2;
    for (int r = 0; r < K; ++r) {
        msg[r] = (uint16_t*)malloc((size_t)S * sizeof(uint16_t));
        if (!msg[r]) {
            for (int q = 0; q < r; ++q) free(msg[q]);
            free(msg);
            return 2;
        }
    }
    for (int i = 0; i < K - 1; ++i) {
        for (int r = 0; r < K; ++r) {
            const int64_t c = mod(r + d - i, K);
            memcpy(msg[r], buf[r] + c * S, (size_t)S * sizeof(uint16_t));
            if (counters) counters[1 + r] += S;
        }
        for (int r = 0; r < K; ++r) {
            const int64_t c = mod(r + d - i, K);
            memcpy(buf[(r + 1) % K] + c * S, msg[r], (size_t)S * sizeof(uint16_t));
        }
        if (counters) counters[0] += 1;
    }
    for (int r = 0; r < K; ++r) free(msg[r]);
    free(msg);
    return 0;
}

/* x: M*K bf16 buffers of N (x[m*K + r] = rank r, micro-batch m).
 * out: K fp32 shards of N/K (slot j), read first when accumulate != 0.
 * counters (optional): [0] rounds, [1 + r] elements rank r sent. */
int oracle_reduce_scatter(int K, int M, int64_t N, const uint16_t* const* x, int mode,
                          float scale, int accumulate, float* const* out, int64_t* counters) {
    if (K < 2 || M < 1 || N <= 0 || N % K || !x || !out) return 1;
    if (mode != RING_FP32 && mode != HOP_BF16) return 1;
    const int64_t S = N / K;
    rank_buf* st = initial_state(K, M, N, x, mode);
    if (!st) return 2;
    int e = rs_rounds(st, K, S, mode, counters);
    if (e) { free_ranks(st, K); return e; }
    for (int j = 0; j < K; ++j) {
        float* o = out[j];
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < S; ++t) {
            const float v = landed(st, K, S, j, t, mode) * scale;
            o[t] = accumulate ? o[t] + v : v;
        }
    }
    free_ranks(st, K);
    return 0;
}

/* shard: K bf16 shards of S (rank j starts with shard j); out: K buffers of
 * K*S, overlapping no shard. */
int oracle_allgather(int K, int64_t S, const uint16_t* const* shard, uint16_t* const* out,
                     int64_t* counters) {
    if (K < 2 || S <= 0 || !shard || !out) return 1;
    for (int r = 0; r < K; ++r) {
        memset(out[r], 0, (size_t)(K * S) * sizeof(uint16_t));
        memcpy(out[r] + (int64_t)r * S, shard[r], (size_t)S * sizeof(uint16_t));
    }
    return ag_rounds((uint16_t**)out, K, S, 0, counters);
}

/* x: K bf16 buffers of N; out: K bf16 buffers of N (may be the inputs). */
int oracle_allreduce(int K, int64_t N, const uint16_t* const* x, int mode, float scale,
                     uint16_t* const* out, int64_t* counters) {
    if (K < 2 || N <= 0 || N % K || !x || !out) return 1;
    if (mode != RING_FP32 && mode != HOP_BF16) return 1;
    const int64_t S = N / K;
    rank_buf* st = initial_state(K, 1, N, x, mode);
    if (!st) return 2;
    int e = rs_rounds(st, K, S, mode, counters);
    if (e) { free_ranks(st, K); return e; }
    /* every rank's buffer goes on the wire as bf16; the landing rank's
     * complete chunk is scaled and rounded first */
    uint16_t* chunk = (uint16_t*)malloc((size_t)S * sizeof(uint16_t));
    if (!chunk) { free_ranks(st, K); return 2; }
    for (int r = 0; r < K; ++r) {
        const int c = (r + 1) % K;
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < S; ++t) chunk[t] = narrow(landed(st, K, S, c, t, mode) * scale);
        uint16_t* o = out[r];
        if (mode == HOP_BF16) {
            memcpy(o, st[r].h, (size_t)N * sizeof(uint16_t));
        } else {
            const float* f = st[r].f;
#pragma omp parallel for schedule(static)
            for (int64_t t = 0; t < N; ++t) o[t] = narrow(f[t]);
        }
        memcpy(o + (int64_t)c * S, chunk, (size_t)S * sizeof(uint16_t));
    }
    free(chunk);
    free_ranks(st, K);
    return ag_rounds((uint16_t**)out, K, S, 1, counters);
}

/* src: K*P gradients (src[r*P + p], numel[p] bf16 each); dst: K flat buckets of
 * bucket_numel; positions no gradient covers are left as they are. */
int oracle_flatten(int K, int P, const uint16_t* const* src, const int64_t* numel,
                   const int64_t* offset, int64_t bucket_numel, uint16_t* const* dst) {
    if (K < 1 || P < 0 || !dst || (P > 0 && (!src || !numel || !offset))) return 1;
    for (int p = 0; p < P; ++p)
        if (numel[p] < 0 || offset[p] < 0 || offset[p] + numel[p] > bucket_numel) return 1;
    for (int r = 0; r < K; ++r)
        for (int p = 0; p < P; ++p)
            memcpy(dst[r] + offset[p], src[(int64_t)r * P + p], (size_t)numel[p] * sizeof(uint16_t));
    return 0;
}

/* Threads the element loops may use (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
