// Device-side helpers shared by the libdpr kernels: 16-byte loads and stores,
// bf16 <-> fp32 conversions.  All arithmetic is IEEE round-to-nearest-even with
// no contraction (the library is built with -fmad=false and uses the _rn
// intrinsics explicitly) and no flush of subnormals.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "dpr_kernels.h"

namespace dpr {

// 16-byte load through the non-coherent read-only path, not kept in L1:
// every input element is read exactly once.  Only used on buffers that no
// thread of the same kernel writes.  Volatile keeps a group of loads in
// program order, so the group is in flight together before it is consumed.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// 16-byte coherent load, not kept in L1 (for kernels that may write the
// buffers they read, i.e. in-place forms).
__device__ __forceinline__ uint4 ld_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_f4(float* p, float a, float b, float c, float d) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// 32-byte accesses (sm_100 and later): the fastest way to stream HBM on GB300.
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

__device__ __forceinline__ void ld_v8(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ void st_f8(float* p, const float* f) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(f[0]),
                 "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7])
                 : "memory");
}

// W 32-bit words (2W bf16 elements) per rank and access: W = 8 moves 32 bytes
// (buffers 32-byte aligned), W = 4 moves 16 bytes (16-byte aligned).
template <int W, bool NC>
__device__ __forceinline__ void load_words(const uint16_t* p, uint32_t (&w)[W]) {
    static_assert(W == 4 || W == 8, "16- or 32-byte accesses");
    if constexpr (W == 8) {
        if constexpr (NC) ld_nc_v8(p, w);
        else ld_v8(p, w);
    } else {
        const uint4 v = NC ? ld_nc_v4(p) : ld_v4(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
}

template <int W>
__device__ __forceinline__ void store_words(uint16_t* p, const uint32_t (&w)[W]) {
    if constexpr (W == 8) st_v8(p, w);
    else st_v4(p, make_uint4(w[0], w[1], w[2], w[3]));
}

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf_1(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

// two fp32 -> two bf16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
    return uint16_t(pack_bf16x2(x, 0.0f) & 0xFFFFu);
}

// bf16 + bf16 -> bf16 on two packed lanes: the fp32 sum of the widened
// operands, rounded once to bf16.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    return pack_bf16x2(__fadd_rn(bf_lo(a), bf_lo(b)), __fadd_rn(bf_hi(a), bf_hi(b)));
}

__device__ __forceinline__ uint4 add_bf16x8(uint4 a, uint4 b) {
    return make_uint4(add_bf16x2(a.x, b.x), add_bf16x2(a.y, b.y), add_bf16x2(a.z, b.z),
                      add_bf16x2(a.w, b.w));
}

__device__ __forceinline__ uint16_t add_bf16(uint16_t a, uint16_t b) {
    return to_bf16(__fadd_rn(bf_1(a), bf_1(b)));
}

// Programmatic dependent launch (griddepcontrol, sm_90 and later).  A grid
// launched with programmatic stream serialization may start while the grid
// before it on the stream is still draining.
//  - grid_wait() blocks until every prerequisite grid has completed and its
//    memory operations are visible; it returns at once for a grid launched
//    without the attribute.
//  - grid_release() lets the next grid on the stream be scheduled once every
//    block of this grid has released it (or exited).
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Called by every thread on entry: a kBesidePrevious grid lets the next grid
// be scheduled at once (it waits for nothing, so nothing behind it can run
// ahead of what it itself depends on).
__device__ __forceinline__ void order_start(int order) {
    if (order == kBesidePrevious) grid_release();
}

// Called by every thread before its first access to a caller buffer, after
// any reads of its plan's fixed tables: a kAfterPrevious grid waits for the
// previous grid here and only then lets the next grid be scheduled (a batch
// member behind it relies on that wait for the buffers written before the
// batch).
__device__ __forceinline__ void order_enter(int order) {
    if (order == kAfterPrevious) {
        grid_wait();
        grid_release();
    }
}

// Called by every thread after its last access.  In a kBesidePrevious grid
// the first block waits here for the previous grid, so this grid cannot
// complete before it; the other blocks exit at once and free their SM slots
// for the grids behind them (one waiting block is enough, since a grid
// completes only when its last block exits).
__device__ __forceinline__ void order_exit(int order) {
    if (order == kBesidePrevious && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        grid_wait();
}

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

}  // namespace dpr
