// Device-side helpers shared by the libdpr kernels: 16-byte loads and stores,
// bf16 <-> fp32 conversions.  All arithmetic is IEEE round-to-nearest-even with
// no contraction (the library is built with -fmad=false and uses the _rn
// intrinsics explicitly) and no flush of subnormals.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

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

__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

}  // namespace dpr
