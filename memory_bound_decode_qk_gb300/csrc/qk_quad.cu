// qk_quad.cu -- QK-norm + RoPE prologue, four threads per head (many heads).
//
// Same operation as the lane-group path in qk_norm_rope.cu ("thox-edge-ops
// v2", sections 5.1 and 5.4; ninfer text profile).  It is for widths where the
// work is many heads rather than few.
//
// Why a second path.  With one head per lane group, each lane holds only 8
// elements.  The per-head overhead is then repeated by every lane:
//   - a 5-level shuffle reduction;
//   - the reciprocal square root;
//   - address decoding;
//   - reloading the weight and the cache row;
//   - divergent rotation paths.
// That overhead outweighs the per-element work: about 290 warp-instructions
// per head were measured on GB300, and the kernel was issue-bound (issue
// active 74%), not HBM-bound.
//
// Here K = 4 threads share a head, and thread k owns the 16-byte chunks
// k, k+4, k+8, ...:
//   - a head load is 4 x 16 contiguous bytes per instruction;
//   - the reduction is two shuffle levels;
//   - the weights (w + delta, fp32) sit in shared memory;
//   - when the rotary width is a multiple of 2 * 4 * N, every rotate-half pair
//     (c, c + half/N) belongs to the same thread, so the rotation needs no
//     shuffle.  Thread k's first HVQ chunks are first members and its next
//     HVQ chunks their partners; for the interleaved layout, pairs lie inside
//     a chunk.
// The rotated chunk count RQ is a template parameter, so every chunk's role is
// known at compile time.  About 50 warp-instructions per head remain.  All C
// loads of a thread are issued before any arithmetic, so a warp (8 heads) has
// 4 KB in flight.
#include "qk_common.cuh"

namespace edge {
namespace {

constexpr int K = 4;  // threads per head

// RQ: rotate-half: chunks per thread that are first members (HVQ); interleaved:
// chunks per thread that rotate.  0: no channel rotates.
template <typename T, bool FP8, int C, int LAYOUT, int RQ>
__global__ void __launch_bounds__(256, FP8 ? 2 : 3) qk_quad_kernel(QKP p) {
    constexpr int N = vec_elems<T>();
    constexpr int D = C * K * N;
    static_assert(LAYOUT == kInterleaved ? RQ <= C : 2 * RQ <= C, "rotated chunks exceed the head");
    __shared__ __align__(16) float wsm[2][D];

    pdl_wait();
    pdl_launch_dependents();

    // w + delta in fp32 (1 when no weight), for q heads and k heads
    for (int e = threadIdx.x; e < D; e += blockDim.x) {
        const float dq = p.wq ? __fadd_rn(to_f(reinterpret_cast<const T*>(p.wq)[e]), p.delta) : 1.0f;
        const float dk = p.wk ? __fadd_rn(to_f(reinterpret_cast<const T*>(p.wk)[e]), p.delta) : 1.0f;
        wsm[0][e] = dq;
        wsm[1][e] = dk;
    }
    __syncthreads();

    const int kt = threadIdx.x & (K - 1);
    const int hs = threadIdx.x / K;           // head slot in the CTA
    const int heads_per_cta = blockDim.x / K;
    const uint32_t hb = (uint32_t)D * sizeof(T);

    for (uint32_t base = blockIdx.x * heads_per_cta; base < p.units;
         base += gridDim.x * heads_per_cta) {
        const uint32_t u = base + hs;
        const bool active = u < p.units;
        const bool isq = u < p.qrows;
        const uint32_t row = isq ? u : u - p.qrows;
        const uint32_t t = active ? fast_div(row, isq ? p.qdiv : p.kdiv) : 0;
        const char* src = (isq ? p.q : p.k) + (size_t)row * hb;
        char* dst = (isq ? p.qo : p.ko) + (size_t)row * D * p.out_bytes;

        uint4 raw[C];
#pragma unroll
        for (int i = 0; i < C; ++i) {
            raw[i] = active ? __ldcs(reinterpret_cast<const uint4*>(src) + kt + K * i)
                            : make_uint4(0u, 0u, 0u, 0u);
        }
        int64_t pos = -1;
        if (RQ > 0 && active) pos = __ldg(p.pos + t);

        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            float x[N];
            unpack_vec<T, N>(raw[i], x);
#pragma unroll
            for (int e = 0; e < N; ++e) ss = __fmaf_rn(x[e], x[e], ss);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        // without normalization (standalone rotary) r = 1 and w = 1: m = x
        const float r = (p.mode & kModeNorm) ? inv_rms(ss, p.invD, p.eps) : 1.0f;

        // normalized value rounded to the dtype, packed (exactly) over the
        // loaded vectors, which are no longer needed
        const float* w = wsm[isq ? 0 : 1];
        uint4 (&mp)[C] = raw;
#pragma unroll
        for (int i = 0; i < C; ++i) {
            float x[N], m[N];
            unpack_vec<T, N>(raw[i], x);
            const float4* wc = reinterpret_cast<const float4*>(w + (kt + K * i) * N);
#pragma unroll
            for (int v = 0; v < N / 4; ++v) {
                const float4 ww = wc[v];
                m[4 * v + 0] = __fmul_rn(__fmul_rn(x[4 * v + 0], r), ww.x);
                m[4 * v + 1] = __fmul_rn(__fmul_rn(x[4 * v + 1], r), ww.y);
                m[4 * v + 2] = __fmul_rn(__fmul_rn(x[4 * v + 2], r), ww.z);
                m[4 * v + 3] = __fmul_rn(__fmul_rn(x[4 * v + 3], r), ww.w);
            }
            mp[i] = pack_vec<T, N>(m);
        }

        const bool rot = RQ > 0 && pos >= 0 && pos < p.cache_len;
        if (!active) continue;
        char* out = dst;
        auto emit = [&](int i, const float (&y)[N]) {
            if constexpr (FP8) {
                auto q8 = quantize_vec<N>(y, p.inv);
                reinterpret_cast<decltype(q8)*>(out)[kt + K * i] = q8;
            } else {
                reinterpret_cast<uint4*>(out)[kt + K * i] = pack_vec<T, N>(y);
            }
        };
        auto emit_m = [&](int i) {
            if constexpr (FP8) {
                float y[N];
                unpack_vec<T, N>(mp[i], y);
                emit(i, y);
            } else {
                reinterpret_cast<uint4*>(out)[kt + K * i] = mp[i];
            }
        };

        if constexpr (LAYOUT == kInterleaved) {
#pragma unroll
            for (int i = 0; i < C; ++i) {
                if (i < RQ && rot) {
                    const int c = kt + K * i;
                    float m[N], y[N], cs[N / 2], sn[N / 2];
                    unpack_vec<T, N>(mp[i], m);
                    const float* crow = p.cs + pos * p.half + c * (N / 2);
                    const float* srow = p.sn + pos * p.half + c * (N / 2);
                    if constexpr (N == 8) {
                        const float4 c4 = __ldg(reinterpret_cast<const float4*>(crow));
                        const float4 s4 = __ldg(reinterpret_cast<const float4*>(srow));
                        cs[0] = c4.x; cs[1] = c4.y; cs[2] = c4.z; cs[3] = c4.w;
                        sn[0] = s4.x; sn[1] = s4.y; sn[2] = s4.z; sn[3] = s4.w;
                    } else {
                        const float2 c2 = __ldg(reinterpret_cast<const float2*>(crow));
                        const float2 s2 = __ldg(reinterpret_cast<const float2*>(srow));
                        cs[0] = c2.x; cs[1] = c2.y;
                        sn[0] = s2.x; sn[1] = s2.y;
                    }
#pragma unroll
                    for (int j = 0; j < N / 2; ++j) {
                        const float a = m[2 * j], b = m[2 * j + 1];
                        y[2 * j] = __fmaf_rn(a, cs[j], -__fmul_rn(b, sn[j]));
                        y[2 * j + 1] = __fmaf_rn(b, cs[j], __fmul_rn(a, sn[j]));
                    }
                    emit(i, y);
                } else {
                    emit_m(i);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < C; ++i) {
                if (i < RQ && rot) {
                    // chunk i (first members) with chunk i + RQ (their partners),
                    // four channels at a time to keep few values live
                    const int c = kt + K * i;
                    float a[N], b[N];
                    unpack_vec<T, N>(mp[i], a);
                    unpack_vec<T, N>(mp[i + RQ], b);
                    const float4* c4 = reinterpret_cast<const float4*>(p.cs + pos * p.half + c * N);
                    const float4* s4 = reinterpret_cast<const float4*>(p.sn + pos * p.half + c * N);
#pragma unroll
                    for (int v = 0; v < N / 4; ++v) {
                        const float4 cc = __ldg(c4 + v), sv = __ldg(s4 + v);
                        const float cs[4] = {cc.x, cc.y, cc.z, cc.w};
                        const float sn[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float ae = a[4 * v + e], be = b[4 * v + e];
                            a[4 * v + e] = __fmaf_rn(ae, cs[e], -__fmul_rn(be, sn[e]));
                            b[4 * v + e] = __fmaf_rn(be, cs[e], __fmul_rn(ae, sn[e]));
                        }
                    }
                    emit(i, a);
                    emit(i + RQ, b);
                } else if (i < RQ || i >= 2 * RQ || !rot) {
                    emit_m(i);
                }
            }
        }
    }
}

using QuadFn = void (*)(QKP);

// The instantiated (C, layout, RQ) combinations: head sizes of 2, 4 or 8
// chunks per thread (D*s = 128, 256 or 512 bytes), every rotary width that
// keeps pairs thread-local.
template <typename T, bool FP8, int C>
QuadFn pick_rq(int layout, int rq) {
    if (rq == 0) return qk_quad_kernel<T, FP8, C, kRotateHalf, 0>;
    if (layout == kInterleaved) {
        switch (rq) {
            case 1: return qk_quad_kernel<T, FP8, C, kInterleaved, 1>;
            case 2: return C >= 2 ? qk_quad_kernel<T, FP8, C, kInterleaved, (C >= 2 ? 2 : 1)> : nullptr;
            case 4: return C >= 4 ? qk_quad_kernel<T, FP8, C, kInterleaved, (C >= 4 ? 4 : 1)> : nullptr;
            case 8: return C >= 8 ? qk_quad_kernel<T, FP8, C, kInterleaved, (C >= 8 ? 8 : 1)> : nullptr;
            default: return nullptr;
        }
    }
    switch (rq) {
        case 1: return qk_quad_kernel<T, FP8, C, kRotateHalf, 1>;
        case 2: return C >= 4 ? qk_quad_kernel<T, FP8, C, kRotateHalf, (C >= 4 ? 2 : 1)> : nullptr;
        case 4: return C >= 8 ? qk_quad_kernel<T, FP8, C, kRotateHalf, (C >= 8 ? 4 : 1)> : nullptr;
        default: return nullptr;
    }
}

}  // namespace

template <typename T, bool FP8>
cudaError_t launch_qk_quad(const QKArgs& a, const QKP& p, cudaLaunchConfig_t cfg, bool* handled) {
    constexpr int N = vec_elems<T>();
    *handled = false;
    if (a.mode & kModeUnrounded) return cudaSuccess;  // served by the lane-group path
    const int64_t hb = (int64_t)a.head_dim * (int64_t)sizeof(T);
    if (hb % (16 * K) != 0) return cudaSuccess;
    const int C = (int)(hb / (16 * K));
    if (C != 2 && C != 4 && C != 8) return cudaSuccess;
    auto aligned = [](const void* ptr, uintptr_t n) {
        return ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) % n) == 0;
    };
    if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.q_out, FP8 ? N : 16) ||
        !aligned(a.k_out, FP8 ? N : 16)) {
        return cudaSuccess;
    }
    int rq = 0;
    if (p.rot > 0) {
        const int unit = (a.layout == kInterleaved ? 1 : 2) * K * N;
        if (p.rot % unit != 0) return cudaSuccess;
        if (!aligned(a.cos, a.layout == kInterleaved ? 8 * (N / 4) : 16) ||
            !aligned(a.sin, a.layout == kInterleaved ? 8 * (N / 4) : 16)) {
            return cudaSuccess;
        }
        rq = p.rot / unit;
    }
    QuadFn fn = nullptr;
    switch (C) {
        case 2: fn = pick_rq<T, FP8, 2>(a.layout, rq); break;
        case 4: fn = pick_rq<T, FP8, 4>(a.layout, rq); break;
        default: fn = pick_rq<T, FP8, 8>(a.layout, rq); break;
    }
    if (fn == nullptr) return cudaSuccess;
    *handled = true;
    const int threads = 256;
    const int64_t per_block = threads / K;
    int64_t blocks = ((int64_t)p.units + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 64;
    if (blocks > cap) blocks = cap;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

bool qk_quad_preferred(const QKArgs& a, int sms) {
    // Measured crossover on GB300 (bf16, head_dim 256): the lane-group path
    // wins below about 40 heads per SM (decode widths, where its one-shot grid
    // puts every head in flight at once), this path above (it issues ~4x fewer
    // instructions per head).
    const int64_t units = a.tokens * (int64_t)(a.q_heads + a.k_heads);
    return units >= (int64_t)sms * 40;
}

template cudaError_t launch_qk_quad<float, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<float, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__half, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__half, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__nv_bfloat16, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__nv_bfloat16, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);

}  // namespace edge
