// glu.cu -- SiLU / tanh-GELU gated activations of a merged gate+up row (sm_103a).
//
// What it computes ("thox-edge-ops v2", section 5.1; FlashRT
// gate_geglu_merged_fp8): out[t, i] = act(g) * u with g = gate_up[t, i],
// u = gate_up[t, d + i].  The gate is the first half of each row.
//   silu(g)      = g * sigma(g)
//   gelu_tanh(g) = 0.5 g (1 + tanh z) = g * sigma(2z),
//                  z = sqrt(2/pi) (g + 0.044715 g^3)
// The second form is an exact identity, since 0.5 (1 + tanh z) equals the
// logistic sigma(2z).  It avoids the cancellation of 1 + tanh z for negative
// z.  sigma(v) is evaluated as num / (1 + e^-|v|) with num = 1 for v >= 0 and
// e^-|v| otherwise, so nothing overflows.
//
// Two precisions of the exponential, both from this identity:
//   - fp32 outputs: libm expf, an IEEE divide, and the GELU argument 2z
//     carried as an unevaluated sum of two floats.  This keeps the relative
//     error within a few fp32 ulps for every g.
//   - bf16 / fp16 / FP8 outputs: e^-a = 2^(-a log2 e) through ex2.approx and
//     a reciprocal through rcp.approx.  The error is a few fp32 ulps (plus
//     the |2z| * 2^-24 of the argument's rounding), far inside half an ulp of
//     the output in most cases.  This keeps the kernel HBM-bound rather than
//     issue-bound at full bandwidth.
//
// GB300 design.  It is a pure stream: it reads 2 elements and writes 1 per
// output.  The rows are flattened into one index space of 16-byte vectors.
// Each thread issues its U gate and U up loads before any arithmetic.  A
// multiply-high divide turns a flat index into (row, column).  Stores are
// 16 bytes, or 8 bytes of E4M3 codes: four codes per 32-bit word.
#include "edge_common.cuh"
#include "fastdiv.h"
#include "launch.h"

namespace edge {
namespace {

constexpr int kSilu = 0;
constexpr int kGelu = 1;

// Constants from their definitions, split into a float and its remainder.
constexpr double kLog2eD = 1.4426950408889634073599246810019;   // log2(e)
constexpr double kK2D = 1.5957691216057307117597842397375;      // 2 sqrt(2/pi)
constexpr double kCD = 0.044715;
constexpr float kLog2e = (float)kLog2eD;
constexpr float kK2 = (float)kK2D;
// 2 sqrt(2/pi) log2(e): the fast tanh-GELU forms its exponent in base 2
// directly, one product fewer per element
constexpr float kK2L = (float)(kK2D * kLog2eD);
constexpr float kK2lo = (float)(kK2D - (double)(float)kK2D);
constexpr float kC = (float)kCD;
constexpr float kClo = (float)(kCD - (double)(float)kCD);

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Reciprocal of x in [1, 2] (its only use: 1 / (1 + e^-|v|)).  Neither x nor
// 1/x is subnormal there, so the flush-to-zero form gives the same result
// without the subnormal handling of the plain form (measured on GB300: 1.17x
// on the issue-bound tanh-GELU gate with FP8 output).
__device__ __forceinline__ float rcp_approx_1to2(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// act(g) * u, fast form (bf16 / fp16 / FP8 outputs).  vl is the logistic
// argument times log2(e), so that e^-|v| = 2^-|vl|.
template <int ACT>
__device__ __forceinline__ float gate_fast(float g, float u) {
    float vl;
    if constexpr (ACT == kSilu) {
        vl = __fmul_rn(g, kLog2e);
    } else {
        const float c2 = __fmul_rn(__fmul_rn(kC, g), g);
        vl = __fmul_rn(__fmul_rn(kK2L, g), __fadd_rn(1.0f, c2));
    }
    const float t = ex2_approx(-fabsf(vl));
    const float num = vl >= 0.0f ? 1.0f : t;
    // g * sigma(v) first, u last: g * u could overflow where sigma(v) = 0
    return __fmul_rn(__fmul_rn(g, __fmul_rn(num, rcp_approx_1to2(__fadd_rn(1.0f, t)))), u);
}

// gate_fast on a pair of elements: the products and sums as packed two-lane
// instructions (each lane rounded as gate_fast rounds it, so the results are
// the same bits), the exponential and the reciprocal per lane.
template <int ACT>
__device__ __forceinline__ float2 gate_fast2(float2 g, float2 u) {
    float2 vl;
    if constexpr (ACT == kSilu) {
        vl = __fmul2_rn(g, splat2(kLog2e));
    } else {
        const float2 c2 = __fmul2_rn(__fmul2_rn(splat2(kC), g), g);
        vl = __fmul2_rn(__fmul2_rn(splat2(kK2L), g), __fadd2_rn(splat2(1.0f), c2));
    }
    const float2 t = make_float2(ex2_approx(-fabsf(vl.x)), ex2_approx(-fabsf(vl.y)));
    const float2 num = make_float2(vl.x >= 0.0f ? 1.0f : t.x, vl.y >= 0.0f ? 1.0f : t.y);
    const float2 den = __fadd2_rn(splat2(1.0f), t);
    const float2 rc = make_float2(rcp_approx_1to2(den.x), rcp_approx_1to2(den.y));
    // g * sigma(v) first, u last (see gate_fast)
    return __fmul2_rn(__fmul2_rn(g, __fmul2_rn(num, rc)), u);
}

// act(g) * u, accurate form (fp32 outputs).
template <int ACT>
__device__ __forceinline__ float gate_accurate(float g, float u) {
    float a, ae;  // |v| = a + ae, v the logistic argument
    bool neg;
    if constexpr (ACT == kSilu) {
        a = fabsf(g);
        ae = 0.0f;
        neg = g < 0.0f;
    } else {
        // v = 2z = K g (1 + C g^2) in double-float arithmetic.  Past |g| = 2^20,
        // |v| > 2^56 and sigma(v) is exactly 0 or 1 in fp32, so g is clamped
        // there: the double-float terms would overflow to inf - inf.
        const float gc = fminf(fmaxf(g, -1048576.0f), 1048576.0f);
        const float g2 = __fmul_rn(gc, gc);
        const float g2e = __fmaf_rn(gc, gc, -g2);
        const float c = __fmul_rn(kC, g2);
        const float ce = __fmaf_rn(kC, g2, -c) + __fmaf_rn(kC, g2e, __fmul_rn(kClo, g2));
        const float s = __fadd_rn(1.0f, c);
        const float bb = __fsub_rn(s, 1.0f);
        const float se = __fadd_rn(__fadd_rn(__fsub_rn(1.0f, __fsub_rn(s, bb)), __fsub_rn(c, bb)), ce);
        const float pq = __fmul_rn(gc, s);
        const float pe = __fmaf_rn(gc, s, -pq) + __fmul_rn(gc, se);
        const float z = __fmul_rn(kK2, pq);
        const float ze = __fmaf_rn(kK2, pq, -z) + __fmaf_rn(kK2, pe, __fmul_rn(kK2lo, pq));
        neg = z < 0.0f;
        a = fabsf(z);
        ae = neg ? -ze : ze;
    }
    // e^-(a + ae) = e^-a * e^-ae ~= e^-a (1 - ae), |ae| <= a few ulp of a.
    // Wherever e^-a is nonzero (a < 104), |ae| < 2^-15; the clamp only keeps
    // t = +0 past that, where a's ulp can exceed 1.
    const float t = __fmul_rn(expf(-a), __fsub_rn(1.0f, fminf(fmaxf(ae, -0.25f), 0.25f)));
    const float num = neg ? t : 1.0f;
    // g * sigma first, u last (see gate_fast)
    return __fmul_rn(__fmul_rn(g, __fdiv_rn(num, __fadd_rn(1.0f, t))), u);
}

template <typename T, bool FP8, int ACT>
__device__ __forceinline__ float gate(float g, float u) {
    if constexpr (std::is_same<T, float>::value && !FP8) {
        return gate_accurate<ACT>(g, u);
    } else {
        return gate_fast<ACT>(g, u);
    }
}

struct GluP {
    const char* gu;
    char* out;
    uint32_t total;   // rows * dvec (vector path) or rows * d (generic, 64-bit below)
    FastDiv dv;       // 16-byte vectors per half row
    int64_t rows;
    int64_t d;
    float inv;
};

template <typename T, bool FP8, int ACT, int U>
__global__ void __launch_bounds__(256) glu_vec_kernel(GluP p) {
    constexpr int N = vec_elems<T>();
    const uint32_t dv = p.dv.d;
    const uint4* gu = reinterpret_cast<const uint4*>(p.gu);
    const uint32_t stride = gridDim.x * blockDim.x * U;

    if (threadIdx.x == 0) {
        // this CTA's first vectors into L2 while the preceding grid drains:
        // flat vectors [i0, i1) lie in rows r0..r1, gate then up in each row
        const uint32_t i0 = blockIdx.x * blockDim.x * U;
        const uint32_t i1 = i0 + blockDim.x * U < p.total ? i0 + blockDim.x * U : p.total;
        if (i0 < i1) {
            const int64_t r0 = fast_div(i0, p.dv), r1 = fast_div(i1 - 1, p.dv);
            const int64_t row = 32 * (int64_t)dv;  // bytes of one [g | u] row
            if (r1 > r0 + 1) {
                prefetch_l2(p.gu, r0 * row, (r1 + 1) * row);
            } else {
                for (int64_t r = r0; r <= r1; ++r) {
                    const int64_t c0 = (int64_t)i0 > r * dv ? (int64_t)i0 - r * dv : 0;
                    const int64_t c1 = (int64_t)i1 < (r + 1) * dv ? (int64_t)i1 - r * dv : dv;
                    prefetch_l2(p.gu, r * row + 16 * c0, r * row + 16 * c1);
                    prefetch_l2(p.gu, r * row + 16 * (dv + c0), r * row + 16 * (dv + c1));
                }
            }
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    for (uint32_t b0 = blockIdx.x * blockDim.x * U + threadIdx.x; b0 < p.total; b0 += stride) {
        uint4 gv[U], uv[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t i = b0 + k * blockDim.x;
            if (i < p.total) {
                const uint32_t row = fast_div(i, p.dv);
                const uint32_t col = i - row * dv;
                const uint4* g = gu + (size_t)row * 2 * dv + col;
                gv[k] = __ldcs(g);
                uv[k] = __ldcs(g + dv);
            } else {
                gv[k] = make_uint4(0u, 0u, 0u, 0u);
                uv[k] = gv[k];
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t i = b0 + k * blockDim.x;
            if (i >= p.total) continue;
            if constexpr (std::is_same<T, float>::value && !FP8) {
                float g[N], u[N], y[N];
                unpack_vec<T, N>(gv[k], g);
                unpack_vec<T, N>(uv[k], u);
#pragma unroll
                for (int e = 0; e < N; ++e) y[e] = gate_accurate<ACT>(g[e], u[e]);
                reinterpret_cast<uint4*>(p.out)[i] = pack_vec<T, N>(y);
            } else {
                // the fast form on element pairs
                float2 g[N / 2], u[N / 2], y[N / 2];
                unpack_pairs<T, N>(gv[k], g);
                unpack_pairs<T, N>(uv[k], u);
#pragma unroll
                for (int j = 0; j < N / 2; ++j) y[j] = gate_fast2<ACT>(g[j], u[j]);
                if constexpr (FP8) {
                    auto q8 = quantize_pairs<N>(y, p.inv);
                    reinterpret_cast<decltype(q8)*>(p.out)[i] = q8;
                } else {
                    reinterpret_cast<uint4*>(p.out)[i] = pack_pairs<T, N>(y);
                }
            }
        }
    }
}

template <typename T, bool FP8, int ACT>
__global__ void __launch_bounds__(256) glu_generic_kernel(GluP p) {
    const T* gu = reinterpret_cast<const T*>(p.gu);
    const int64_t total = p.rows * p.d;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;

    pdl_wait();
    pdl_launch_dependents();

    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t row = i / p.d;
        const int64_t col = i - row * p.d;
        const float g = to_f(gu[row * 2 * p.d + col]);
        const float u = to_f(gu[row * 2 * p.d + p.d + col]);
        const float y = gate<T, FP8, ACT>(g, u);
        if constexpr (FP8) {
            reinterpret_cast<uint8_t*>(p.out)[i] = quantize1(y, p.inv);
        } else {
            reinterpret_cast<T*>(p.out)[i] = from_f<T>(y);
        }
    }
}

template <typename T, bool FP8, int ACT>
cudaError_t launch_typed(const GluArgs& a, GluP& p, cudaStream_t s) {
    constexpr int N = vec_elems<T>();
    auto aligned = [](const void* ptr, uintptr_t n) {
        return (reinterpret_cast<uintptr_t>(ptr) % n) == 0;
    };
    const int sms = sm_count();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;

    const int64_t dvec = a.d / N;
    const bool vec = (a.d * (int64_t)sizeof(T)) % 16 == 0 && aligned(a.gate_up, 16) &&
                     aligned(a.out, FP8 ? N : 16) && a.rows * dvec <= kMaxUnits;
    if (vec) {
        p.dv = make_fastdiv((uint32_t)dvec);
        p.total = (uint32_t)(a.rows * dvec);
        const int threads = 256;
        // one vector per thread and a one-shot grid (measured on GB300: 2 or 4
        // vectors per thread were slower at every size timed on its own,
        // 1.1x to 1.2x for the tanh-GELU gate with FP8 output)
        int64_t blocks = ((int64_t)p.total + threads - 1) / threads;
        const int64_t cap = (int64_t)sms * (2048 / threads) * 64;
        if (blocks > cap) blocks = cap;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(threads);
        return cudaLaunchKernelEx(&cfg, glu_vec_kernel<T, FP8, ACT, 1>, p);
    }
    const int64_t total = a.rows * a.d;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)sms * 64;
    if (blocks > cap) blocks = cap;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, glu_generic_kernel<T, FP8, ACT>, p);
}

template <typename T>
cudaError_t launch_dt(const GluArgs& a, GluP& p, cudaStream_t s) {
    const bool fp8 = a.out_dt == kFP8;
    if (a.act == kSilu) {
        return fp8 ? launch_typed<T, true, kSilu>(a, p, s) : launch_typed<T, false, kSilu>(a, p, s);
    }
    return fp8 ? launch_typed<T, true, kGelu>(a, p, s) : launch_typed<T, false, kGelu>(a, p, s);
}

}  // namespace

cudaError_t launch_glu(const GluArgs& a, cudaStream_t s) {
    GluP p;
    p.gu = static_cast<const char*>(a.gate_up);
    p.out = static_cast<char*>(a.out);
    p.total = 0;
    p.dv = make_fastdiv(1);
    p.rows = a.rows;
    p.d = a.d;
    p.inv = a.inv_scale;
    switch (a.dt) {
        case kF32: return launch_dt<float>(a, p, s);
        case kF16: return launch_dt<__half>(a, p, s);
        default: return launch_dt<__nv_bfloat16>(a, p, s);
    }
}

}  // namespace edge
