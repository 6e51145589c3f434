// Ring-order summation shared by the reduce-scatter, all-reduce and
// per-parameter kernels: the addends of chunk j are added starting at rank j,
// then ranks j+1, ..., j-1 (CMU 11-868 Lecture 14 notes, section 3.2; "Ring
// All-Reduce illustrated", Phase 1), with fp32 or per-hop bf16 partial sums.
#pragma once

#include "dpr_device.cuh"
#include "dpr_kernels.h"

namespace dpr {

// Folds the next addend (2W elements as W bf16x2 words) into the ring sum.
template <int MODE, int W>
__device__ __forceinline__ void ring_add(bool first, const uint32_t (&x)[W], float (&acc)[2 * W],
                                         uint32_t (&hop)[W]) {
    if constexpr (MODE == DPR_SUM_RING_FP32) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            if (first) {
                acc[2 * k] = bf_lo(x[k]);
                acc[2 * k + 1] = bf_hi(x[k]);
            } else {
                acc[2 * k] = __fadd_rn(acc[2 * k], bf_lo(x[k]));
                acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], bf_hi(x[k]));
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < W; ++k) hop[k] = first ? x[k] : add_bf16x2(hop[k], x[k]);
    }
}

// Ring-order sum of elements [e, e + 2W) of chunk j.  KC > 0: K = KC known at
// compile time; KC == 0: K at run time.  Loads are issued in groups of G
// ranks (all M micro-batches of each) before the group is added, keeping up
// to 256 bytes in flight per thread while the additions follow the ring.
// With M = 2 each rank's addend is first its local accumulation
// bf16(g0 + g1).
template <int KC, int M, int MODE, int W, bool NC>
__device__ __forceinline__ void ring_sum(const uint16_t* const* in, int K, int j, uint64_t e,
                                         float (&acc)[2 * W]) {
    constexpr int LOADS = (W == 8) ? 8 : 16;
    constexpr int G0 = LOADS / M;
    constexpr int G = (KC > 0 && KC < G0) ? KC : G0;
    static_assert(KC == 0 || KC % G == 0, "load groups must tile K");
    uint32_t hop[W];
#pragma unroll
    for (int k = 0; k < W; ++k) hop[k] = 0;
    const int Kr = KC > 0 ? KC : K;
#pragma unroll(KC > 0 ? 64 : 1)
    for (int g0 = 0; g0 < Kr; g0 += G) {
        uint32_t v[G][M][W];
#pragma unroll
        for (int s = 0; s < G; ++s) {
            if (KC > 0 || g0 + s < Kr) {
                int r = j + g0 + s;
                r = (r >= Kr) ? r - Kr : r;
#pragma unroll
                for (int m = 0; m < M; ++m) load_words<W, NC>(in[m * Kr + r] + e, v[s][m]);
            }
        }
#pragma unroll
        for (int s = 0; s < G; ++s) {
            if (KC > 0 || g0 + s < Kr) {
                uint32_t x[W];
#pragma unroll
                for (int k = 0; k < W; ++k)
                    x[k] = (M == 1) ? v[s][0][k] : add_bf16x2(v[s][0][k], v[s][M - 1][k]);
                ring_add<MODE, W>(g0 + s == 0, x, acc, hop);
            }
        }
    }
    if constexpr (MODE == DPR_SUM_HOP_BF16) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            acc[2 * k] = bf_lo(hop[k]);
            acc[2 * k + 1] = bf_hi(hop[k]);
        }
    }
}

// Scaled fp32 shard store of 2W values: out = acc*scale, or out + acc*scale
// (two roundings, never fused).
template <int W>
__device__ __forceinline__ void store_shard(float* o, const float (&acc)[2 * W], float scale,
                                            int accumulate) {
    float r[2 * W];
#pragma unroll
    for (int k = 0; k < 2 * W; ++k) r[k] = __fmul_rn(acc[k], scale);
    if (accumulate) {
#pragma unroll
        for (int q = 0; q < 2 * W; q += 4) {
            const float4 a = *reinterpret_cast<const float4*>(o + q);
            r[q] = __fadd_rn(a.x, r[q]);
            r[q + 1] = __fadd_rn(a.y, r[q + 1]);
            r[q + 2] = __fadd_rn(a.z, r[q + 2]);
            r[q + 3] = __fadd_rn(a.w, r[q + 3]);
        }
    }
    if constexpr (W == 8) {
        st_f8(o, r);
        st_f8(o + 8, r + 8);
    } else {
        st_f4(o, r[0], r[1], r[2], r[3]);
        st_f4(o + 4, r[4], r[5], r[6], r[7]);
    }
}

}  // namespace dpr
