// The alpha-beta cost model of collective algorithms (host only).
//
// CMU 11-868 Lecture 14 notes, section 3.4: a message of n bytes costs
// alpha + n / beta.  With K devices and N bytes per device:
//   ring all-reduce   2(K-1) (alpha + N / (K beta))
//   tree all-reduce   2 ceil(log2 K) (alpha + N / beta)
//   naive all-reduce  2 (alpha + (K-1) N / beta)       (all to device 0 and back)
// Section 3.1: a ring broadcast of N bytes cut into S segments takes
//   (K - 2 + S) (alpha + N / (S beta))                 (S = 1: unsegmented)
// Section 4.4: K-way data parallelism without overlap speeds a step of T1 up
// by T1 / (T1 / K + T_comm), T_comm the ring all-reduce time.
#include <cmath>
#include <cstdint>

#include "../../include/dpr.h"

namespace {

bool valid(int K, double bytes, double alpha, double beta) {
    return K >= 1 && bytes >= 0 && alpha >= 0 && beta > 0 && std::isfinite(bytes) &&
           std::isfinite(alpha) && std::isfinite(beta);
}

int ceil_log2(int K) {
    int c = 0;
    while ((1 << c) < K) ++c;
    return c;
}

// T(N) = c0 + c1 * N for each all-reduce algorithm
bool linear(int algo, int K, double alpha, double beta, double* c0, double* c1) {
    switch (algo) {
        case DPR_ALGO_RING:
            *c0 = 2.0 * (K - 1) * alpha;
            *c1 = 2.0 * (K - 1) / (double(K) * beta);
            return true;
        case DPR_ALGO_TREE:
            *c0 = 2.0 * ceil_log2(K) * alpha;
            *c1 = 2.0 * ceil_log2(K) / beta;
            return true;
        case DPR_ALGO_NAIVE:
            *c0 = 2.0 * alpha;
            *c1 = 2.0 * (K - 1) / beta;
            return true;
        default:
            return false;
    }
}

}  // namespace

extern "C" {

dpr_status dpr_cost_allreduce(int algo, int K, double bytes, double alpha, double beta,
                              double* seconds) {
    if (!seconds || !valid(K, bytes, alpha, beta)) return DPR_ERR_INVALID_ARG;
    double c0 = 0, c1 = 0;
    if (!linear(algo, K, alpha, beta, &c0, &c1)) return DPR_ERR_INVALID_ARG;
    *seconds = c0 + c1 * bytes;
    return DPR_OK;
}

dpr_status dpr_cost_ring_broadcast(int K, double bytes, double alpha, double beta, int64_t segments,
                                   double* seconds) {
    if (!seconds || K < 2 || segments < 1 || !valid(K, bytes, alpha, beta))
        return DPR_ERR_INVALID_ARG;
    const double S = double(segments);
    *seconds = (K - 2 + S) * (alpha + bytes / (S * beta));
    return DPR_OK;
}

dpr_status dpr_cost_best_segments(int K, double bytes, double alpha, double beta,
                                  int64_t max_segments, int64_t* segments, double* seconds) {
    if (!segments || !seconds || max_segments < 1) return DPR_ERR_INVALID_ARG;
    int64_t best = 1;
    double best_t = 0;
    dpr_status st = dpr_cost_ring_broadcast(K, bytes, alpha, beta, 1, &best_t);
    if (st != DPR_OK) return st;
    for (int64_t S = 2; S <= max_segments && S > 0; S *= 2) {
        double t = 0;
        dpr_cost_ring_broadcast(K, bytes, alpha, beta, S, &t);
        if (t < best_t) {
            best_t = t;
            best = S;
        }
    }
    *segments = best;
    *seconds = best_t;
    return DPR_OK;
}

dpr_status dpr_cost_crossover(int algo_a, int algo_b, int K, double alpha, double beta,
                              double* bytes) {
    if (!bytes || !valid(K, 0.0, alpha, beta)) return DPR_ERR_INVALID_ARG;
    double a0, a1, b0, b1;
    if (!linear(algo_a, K, alpha, beta, &a0, &a1) || !linear(algo_b, K, alpha, beta, &b0, &b1))
        return DPR_ERR_INVALID_ARG;
    if (a1 == b1) return DPR_ERR_UNSUPPORTED;           // parallel lines: no crossover
    const double n = (b0 - a0) / (a1 - b1);
    if (!(n >= 0)) return DPR_ERR_UNSUPPORTED;          // they cross at no message size
    *bytes = n;
    return DPR_OK;
}

dpr_status dpr_cost_dp_speedup(double t1, int K, double bytes, double alpha, double beta,
                               double* speedup) {
    if (!speedup || !(t1 > 0) || K < 1) return DPR_ERR_INVALID_ARG;
    double t_comm = 0;
    dpr_status st = dpr_cost_allreduce(DPR_ALGO_RING, K, bytes, alpha, beta, &t_comm);
    if (st != DPR_OK) return st;
    *speedup = t1 / (t1 / K + t_comm);
    return DPR_OK;
}

}  // extern "C"
