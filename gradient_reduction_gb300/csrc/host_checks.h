// Host-side helpers shared by the libdpr entry points: address spans and the
// overlap and alignment tests that run before any launch, and the one-time
// upload of a plan's tables.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

namespace dpr {

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
};

inline bool overlaps(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }

inline Span span_of(const void* p, uint64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + uintptr_t(bytes)};
}

inline bool pairwise_disjoint(std::vector<Span> v) {
    std::sort(v.begin(), v.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    for (size_t i = 1; i < v.size(); ++i)
        if (v[i].lo < v[i - 1].hi) return false;
    return true;
}

// Does any span of `b` overlap any span of `a`?  `a` must be pairwise
// disjoint (as pairwise_disjoint checks).
inline bool any_overlap(std::vector<Span> a, const std::vector<Span>& b) {
    std::sort(a.begin(), a.end(), [](const Span& x, const Span& y) { return x.lo < y.lo; });
    for (const Span& x : b) {
        // the first span of `a` that ends after x starts (ends are sorted too)
        auto it = std::upper_bound(a.begin(), a.end(), x.lo,
                                   [](uintptr_t v, const Span& y) { return v < y.hi; });
        if (it != a.end() && overlaps(*it, x)) return true;
    }
    return false;
}

// A span with the index of the batch member it belongs to.
struct OwnedSpan {
    Span s;
    int owner;
};

// Does `x` (of member `owner`) overlap a span of `sorted` that belongs to
// another member?  `sorted` must be pairwise disjoint and sorted by start.
inline bool overlaps_other(const std::vector<OwnedSpan>& sorted, const Span& x, int owner) {
    auto it = std::upper_bound(sorted.begin(), sorted.end(), x.lo,
                               [](uintptr_t v, const OwnedSpan& y) { return v < y.s.hi; });
    for (; it != sorted.end() && it->s.lo < x.hi; ++it)
        if (it->owner != owner && overlaps(it->s, x)) return true;
    return false;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// cudaMalloc a device copy of `src` and enqueue the copy on `st`.
template <typename T>
cudaError_t upload(T** dst, const std::vector<T>& src, cudaStream_t st) {
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), src.size() * sizeof(T));
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice, st);
    return e;
}

}  // namespace dpr
