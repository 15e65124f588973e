// edge_common.cuh -- device helpers shared by the decode-seam kernels.
//
// Element types, 16-byte vector packing, rounding to the activation dtype, the
// static-scale FP8 E4M3 epilogue, warp reductions and the programmatic
// dependent launch hooks.  Every op keeps its fp32 arithmetic in registers and
// rounds once at the output ("thox-edge-ops v2", section 3, R1).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace edge {

// ---------------------------------------------------------------- types

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kBytes = 4;
};
template <> struct Elem<__half> {
    static constexpr int kBytes = 2;
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
};

// Elements of T in one 16-byte vector.
template <typename T> __host__ __device__ constexpr int vec_elems() { return 16 / Elem<T>::kBytes; }

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Round an fp32 value to T and back (the intermediate rounding of the prologue).
template <typename T> __device__ __forceinline__ float round_to(float v) { return to_f(from_f<T>(v)); }

// ---------------------------------------------------------------- 16-byte vectors

// Unpack a 16-byte vector of T into fp32.
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 p;
        if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            p = __half22float2(h);
        } else {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            p = __bfloat1622float2(h);
        }
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}

template <typename T, int N>
__device__ __forceinline__ void unpack_vec(const uint4& v, float (&f)[N]) {
    if constexpr (N == 4) {
        unpack(v, f);
    } else {
        unpack16<T>(v, f);
    }
}

// Pack N fp32 values into a 16-byte vector of T, rounding each to nearest even.
template <typename T, int N>
__device__ __forceinline__ uint4 pack_vec(const float (&f)[N]) {
    uint4 v;
    if constexpr (N == 4) {
        v.x = __float_as_uint(f[0]);
        v.y = __float_as_uint(f[1]);
        v.z = __float_as_uint(f[2]);
        v.w = __float_as_uint(f[3]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (std::is_same<T, __half>::value) {
                __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            } else {
                __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            }
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return v;
}

// ---------------------------------------------------------------- fp32 pairs

// A 16-byte vector as N/2 fp32 pairs, for the packed two-lane fp32
// instructions of the sm_100 family (__fadd2_rn, __fmul2_rn, __ffma2_rn).  Each
// lane of one of them rounds exactly as the scalar __fadd_rn / __fmul_rn /
// __fmaf_rn does, so an elementwise step gives the same bits with half the
// instructions.  Measured on GB300: 5-9% faster for the issue-bound tanh-GELU
// gate, 2-12% for the RMSNorm rows and 5% for LayerNorm at many rows; slower
// for the four-threads-per-head prologue, whose 128-register budget the pairs
// strain into spills, and for the plain quantize, which keep scalar forms.
template <typename T, int N>
__device__ __forceinline__ void unpack_pairs(const uint4& v, float2 (&f)[N / 2]) {
    if constexpr (N == 4) {
        f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (std::is_same<T, __half>::value) {
                f[i] = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            } else {
                f[i] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            }
        }
    }
}

// N/2 fp32 pairs -> a 16-byte vector of T, each value rounded to nearest even.
template <typename T, int N>
__device__ __forceinline__ uint4 pack_pairs(const float2 (&f)[N / 2]) {
    if constexpr (N == 4) {
        return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y),
                          __float_as_uint(f[1].x), __float_as_uint(f[1].y));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (std::is_same<T, __half>::value) {
                __half2 h = __float22half2_rn(f[i]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            } else {
                __nv_bfloat162 h = __float22bfloat162_rn(f[i]);
                w[i] = *reinterpret_cast<uint32_t*>(&h);
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// ---------------------------------------------------------------- FP8 epilogue

// Two fp32 values -> two E4M3 codes (round to nearest even, saturate to
// +-448); the first value lands in the low byte.
__device__ __forceinline__ uint32_t fp8x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// N fp32 results -> N E4M3 codes of (y * inv_scale) packed in N bytes, four
// codes per 32-bit word.  The product is taken in fp32 like the rest of the
// epilogue.
template <int N> struct Fp8Pack;
template <> struct Fp8Pack<4> {
    using type = uint32_t;
};
template <> struct Fp8Pack<8> {
    using type = uint2;
};

template <int N>
__device__ __forceinline__ typename Fp8Pack<N>::type quantize_vec(const float (&y)[N], float inv) {
    uint32_t w[N / 4];
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        uint32_t lo = fp8x2(__fmul_rn(y[4 * i], inv), __fmul_rn(y[4 * i + 1], inv));
        uint32_t hi = fp8x2(__fmul_rn(y[4 * i + 2], inv), __fmul_rn(y[4 * i + 3], inv));
        w[i] = lo | (hi << 16);
    }
    if constexpr (N == 4) {
        return w[0];
    } else {
        return make_uint2(w[0], w[1]);
    }
}

// quantize_vec from fp32 pairs: the same codes, the products by inv_scale
// packed two to an instruction.
template <int N>
__device__ __forceinline__ typename Fp8Pack<N>::type quantize_pairs(const float2 (&y)[N / 2],
                                                                    float inv) {
    uint32_t w[N / 4];
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float2 a = __fmul2_rn(y[2 * i], splat2(inv));
        const float2 b = __fmul2_rn(y[2 * i + 1], splat2(inv));
        w[i] = fp8x2(a.x, a.y) | (fp8x2(b.x, b.y) << 16);
    }
    if constexpr (N == 4) {
        return w[0];
    } else {
        return make_uint2(w[0], w[1]);
    }
}

__device__ __forceinline__ uint8_t quantize1(float y, float inv) {
    return (uint8_t)(fp8x2(__fmul_rn(y, inv), 0.0f) & 0xFFu);
}

// ---------------------------------------------------------------- reductions

// Sum over aligned groups of G lanes (G a power of two <= 32), of float or
// double values.
template <int G, typename V>
__device__ __forceinline__ V group_sum(V v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 1 / sqrt(ss / n + eps), with inv_n = 1/n rounded to fp32 on the host and
// the hardware reciprocal square root (rsqrtf, at most 2 ulp).  Its relative
// error, a few fp32 ulps, is far inside the tolerance band of every output.
__device__ __forceinline__ float inv_rms(float ss, float inv_n, float eps) {
    return rsqrtf(__fmaf_rn(ss, inv_n, eps));
}

// ---------------------------------------------------------------- PDL hooks

// Programmatic dependent launch.  Both instructions are no-ops unless the
// kernel was launched with programmatic stream serialization.  wait() blocks
// until the preceding grid in the stream has completed and its writes are
// visible, so every kernel calls it before its first global load whose value
// it uses.  Before it, a kernel only computes addresses and prefetches into
// L2.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- L2 prefetch

// Ask L2 to fetch the bytes [base + lo, base + hi) from HBM (at most the
// first kPrefetchMax of them).  Issued by one thread before pdl_wait(), the
// fetch overlaps the HBM latency of a CTA's first loads with the tail of the
// preceding grid.  A prefetch is a hint that returns no data: the loads that
// read the bytes still come after the wait, and L2 stays coherent with every
// SM's writes, so the preceding grid's writes to the range are still seen.
// The start is rounded up and the end down to 16 bytes (the bulk prefetch
// wants 16-byte-aligned addresses and sizes), so nothing outside the range is
// touched.
constexpr uint32_t kPrefetchPiece = 16u << 10;
constexpr uint32_t kPrefetchMax = 64u << 10;
__device__ __forceinline__ void prefetch_l2(const void* base, int64_t lo, int64_t hi) {
    if (base == nullptr || hi <= lo) return;
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    uintptr_t s = (b + (uintptr_t)lo + 15u) & ~(uintptr_t)15u;
    uintptr_t e = (b + (uintptr_t)hi) & ~(uintptr_t)15u;
    if (e > s + kPrefetchMax) e = s + kPrefetchMax;
    while (s < e) {
        const uint32_t n = (uint32_t)(e - s < kPrefetchPiece ? e - s : kPrefetchPiece);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s), "r"(n) : "memory");
        s += n;
    }
}

// Prefetch into L2 the line holding *p (no alignment needed).
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
    if (p != nullptr) asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// Prefetch into this SM's L1 the line holding *p, which must lie inside an
// allocation (only issued after the kernel's wait, for data it will load).
__device__ __forceinline__ void prefetch_l1_line(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p) : "memory");
}


}  // namespace edge
