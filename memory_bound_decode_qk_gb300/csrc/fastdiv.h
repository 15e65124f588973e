// fastdiv.h -- unsigned 32-bit division by a loop-invariant divisor.
//
// Method: T. Granlund and P. L. Montgomery, "Division by invariant integers
// using multiplication" (PLDI 1994), section 4 (unsigned division).  With
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, for every 32-bit n:
//     t = mulhi(m, n),  n / d = (t + ((n - t) >> 1)) >> (l - 1)     (l >= 1)
// and n / 1 = n.  Used to turn a flattened index into (row, column) without
// a hardware divide.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define EDGE_HD __host__ __device__ __forceinline__
#else
#define EDGE_HD inline
#endif

namespace edge {

struct FastDiv {
    uint32_t d;   // divisor (>= 1)
    uint32_t m;   // magic multiplier
    uint32_t l;   // ceil(log2 d)
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while (l < 32 && (uint64_t(1) << l) < d) ++l;
    f.l = l;
    f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
    return f;
}

EDGE_HD uint32_t mulhi32(uint32_t a, uint32_t b) {
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * b) >> 32);
#endif
}

EDGE_HD uint32_t fast_div(uint32_t n, const FastDiv& f) {
    if (f.l == 0) return n;
    uint32_t t = mulhi32(f.m, n);
    return (t + ((n - t) >> 1)) >> (f.l - 1);
}

}  // namespace edge
