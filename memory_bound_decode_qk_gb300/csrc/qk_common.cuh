// qk_common.cuh -- definitions shared by the QK-norm + RoPE kernels.
#pragma once

#include "edge_common.cuh"
#include "fastdiv.h"
#include "launch.h"

namespace edge {

constexpr int kRotateHalf = 0;
constexpr int kInterleaved = 1;

// Prologue modes (QKArgs::mode): kModeNorm normalizes each head first (the
// fused prologue; without it the op is the standalone rotary embedding);
// kModeUnrounded rotates the fp32 normalized value instead of its rounding to
// the dtype (the variant asked for in the ninfer review, item 1).
constexpr int kModeNorm = 1;
constexpr int kModeUnrounded = 2;

// Kernel parameters of the prologue (validated by the C ABI layer).
struct QKP {
    const char* q;
    const char* k;
    char* qo;
    char* ko;
    const char* wq;
    const char* wk;
    const int64_t* pos;
    const float* cs;
    const float* sn;
    int64_t cache_len;
    int64_t tokens;
    uint32_t units;        // tokens * (q_heads + k_heads)
    FastDiv heads;         // q_heads + k_heads
    FastDiv qdiv, kdiv;    // q_heads, k_heads (k_heads >= 1 for the divisor)
    uint32_t qrows;        // tokens * q_heads
    int q_heads, k_heads, D, rot, half;
    int in_bytes, out_bytes;  // element sizes of input and output
    float eps, delta, inv, invD;  // invD = 1 / head_dim (fp32)
    int mode;                     // kModeNorm | kModeUnrounded
};

struct Unit {
    const char* src;
    char* dst;
    const char* w;
    int64_t t;
};

// Prefetch into L2 what a CTA's first head units [u0, u1) read, before the
// dependent-launch wait.  Token-major units (q heads then k heads of each
// token) when `token_major`, else all q rows first and then all k rows.  CTA 0
// also fetches the two norm weights.
__device__ __forceinline__ void prefetch_heads(const QKP& p, uint32_t u0, uint32_t u1,
                                               bool token_major) {
    if (u1 > p.units) u1 = p.units;
    if (u0 >= u1) return;
    const int64_t hb = (int64_t)p.D * p.in_bytes;
    if (token_major) {
        const int64_t t0 = fast_div(u0, p.heads), t1 = fast_div(u1 - 1, p.heads) + 1;
        prefetch_l2(p.q, t0 * p.q_heads * hb, t1 * p.q_heads * hb);
        prefetch_l2(p.k, t0 * p.k_heads * hb, t1 * p.k_heads * hb);
        if (p.rot > 0) prefetch_l2_line(p.pos + t0);
    } else {
        const uint32_t qr = p.qrows;
        if (u0 < qr) prefetch_l2(p.q, (int64_t)u0 * hb, (int64_t)(u1 < qr ? u1 : qr) * hb);
        if (u1 > qr) prefetch_l2(p.k, (int64_t)(u0 > qr ? u0 - qr : 0) * hb, (int64_t)(u1 - qr) * hb);
    }
    if (blockIdx.x == 0) {
        prefetch_l2(p.wq, 0, hb);
        prefetch_l2(p.wk, 0, hb);
    }
}

__device__ __forceinline__ Unit locate(const QKP& p, uint32_t u) {
    uint32_t t = fast_div(u, p.heads);
    int h = (int)(u - t * p.heads.d);
    Unit r;
    r.t = t;
    int64_t row;
    if (h < p.q_heads) {
        row = (int64_t)t * p.q_heads + h;
        r.src = p.q + row * p.D * p.in_bytes;
        r.dst = p.qo + row * p.D * p.out_bytes;
        r.w = p.wq;
    } else {
        row = (int64_t)t * p.k_heads + (h - p.q_heads);
        r.src = p.k + row * p.D * p.in_bytes;
        r.dst = p.ko + row * p.D * p.out_bytes;
        r.w = p.wk;
    }
    return r;
}


// ---------------------------------------------------------------- shared head math

// Cache entries a lane needs: rotate-half lanes hold N consecutive channels of
// one half (N entries); interleaved lanes hold N/2 pairs (N/2 entries).
template <typename T, int LAYOUT>
struct CacheRegs {
    static constexpr int N = vec_elems<T>();
    static constexpr int kCount = LAYOUT == kInterleaved ? N / 2 : N;
    float c[kCount], s[kCount];
};

// Role of a lane's vector in the rotation: 0 none, 1 first member, 2 second.
template <typename T, int LAYOUT>
__device__ __forceinline__ int rotary_role(const QKP& p, int sub) {
    constexpr int N = vec_elems<T>();
    const int e0 = sub * N;
    if constexpr (LAYOUT == kInterleaved) {
        return e0 < p.rot ? 1 : 0;
    } else {
        return e0 < p.half ? 1 : (e0 < p.rot ? 2 : 0);
    }
}

// Load this lane's cos/sin entries of cache row `pos` (role != 0 only).
template <typename T, int LAYOUT>
__device__ __forceinline__ void load_cache(const QKP& p, int64_t pos, int sub, int role,
                                           CacheRegs<T, LAYOUT>& cr) {
    constexpr int N = vec_elems<T>();
    const int e0 = sub * N;
    if constexpr (LAYOUT == kInterleaved) {
        const float* crow = p.cs + pos * p.half + e0 / 2;
        const float* srow = p.sn + pos * p.half + e0 / 2;
        if constexpr (N == 8) {
            float4 c4 = __ldg(reinterpret_cast<const float4*>(crow));
            float4 s4 = __ldg(reinterpret_cast<const float4*>(srow));
            cr.c[0] = c4.x; cr.c[1] = c4.y; cr.c[2] = c4.z; cr.c[3] = c4.w;
            cr.s[0] = s4.x; cr.s[1] = s4.y; cr.s[2] = s4.z; cr.s[3] = s4.w;
        } else {
            float2 c2 = __ldg(reinterpret_cast<const float2*>(crow));
            float2 s2 = __ldg(reinterpret_cast<const float2*>(srow));
            cr.c[0] = c2.x; cr.c[1] = c2.y;
            cr.s[0] = s2.x; cr.s[1] = s2.y;
        }
    } else {
        const int j0 = role == 1 ? e0 : e0 - p.half;
        const float4* c4 = reinterpret_cast<const float4*>(p.cs + pos * p.half + j0);
        const float4* s4 = reinterpret_cast<const float4*>(p.sn + pos * p.half + j0);
#pragma unroll
        for (int v = 0; v < N / 4; ++v) {
            float4 cc = __ldg(c4 + v), sv = __ldg(s4 + v);
            cr.c[4 * v] = cc.x; cr.c[4 * v + 1] = cc.y; cr.c[4 * v + 2] = cc.z; cr.c[4 * v + 3] = cc.w;
            cr.s[4 * v] = sv.x; cr.s[4 * v + 1] = sv.y; cr.s[4 * v + 2] = sv.z; cr.s[4 * v + 3] = sv.w;
        }
    }
}

// Normalize, round to the dtype, rotate and store one head held as one
// 16-byte vector per lane of an LPH-lane group.  w holds w + delta.  All 32
// lanes of the warp call this together (the rotate-half partner comes over a
// warp shuffle); inactive groups carry zeros and store nothing.  `role` is
// this lane's rotation role for this head's token (0 when it does not rotate).
//  copy: pass the head through unnormalized and unrotated (the v heads of
//  the fused QKV op); the lane group still joins the warp-wide reduction.
template <typename T, bool FP8, int LPH, int LAYOUT>
__device__ __forceinline__ void qk_core(const QKP& p, char* dst, bool active, int lane, int sub,
                                        const uint4& raw, const float (&w)[vec_elems<T>()], int role,
                                        const CacheRegs<T, LAYOUT>& cr, bool copy = false) {
    constexpr int N = vec_elems<T>();
    constexpr int P = N / 2;
    // the elementwise steps on fp32 pairs (packed two-lane instructions, each
    // lane rounded as the scalar form rounds it)
    float2 x[P];
    unpack_pairs<T, N>(raw, x);
    // normalized value n (fp32); without normalization n = x
    float2 n[P];
    if (p.mode & kModeNorm) {
        float2 s2 = splat2(0.0f);
#pragma unroll
        for (int j = 0; j < P; ++j) s2 = __ffma2_rn(x[j], x[j], s2);
        const float ss = group_sum<LPH>(__fadd_rn(s2.x, s2.y));
        const float2 r2 = splat2(inv_rms(ss, p.invD, p.eps));
#pragma unroll
        for (int j = 0; j < P; ++j) {
            n[j] = copy ? x[j] : __fmul2_rn(__fmul2_rn(x[j], r2), make_float2(w[2 * j], w[2 * j + 1]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < P; ++j) n[j] = x[j];
    }
    // m: n rounded to the activation dtype (packed exactly as `mine`).  The
    // rotation consumes m, or n itself in the unrounded mode; channels that
    // do not rotate emit m.
    const bool unrounded = (p.mode & kModeUnrounded) != 0;
    const uint4 mine = pack_pairs<T, N>(n);
    float2 m[P], src[P];
    unpack_pairs<T, N>(mine, m);
#pragma unroll
    for (int j = 0; j < P; ++j) src[j] = unrounded ? n[j] : m[j];

    float2 y[P];
#pragma unroll
    for (int j = 0; j < P; ++j) y[j] = m[j];

    if constexpr (LAYOUT == kInterleaved) {
        if (role != 0) {
            // pair (a, b) -> (a c - b s, b c + a s): the products
            // (b, a) * (-s, s), then one fma per pair
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 t = __fmul2_rn(make_float2(src[j].y, src[j].x), make_float2(-cr.s[j], cr.s[j]));
                y[j] = __ffma2_rn(src[j], splat2(cr.c[j]), t);
            }
        }
    } else {
        // rotate-half: channel e pairs with e + half; the partner vector is
        // held by the lane half/N positions away in the same lane group
        const int hv = p.half / N;
        const int from = role == 1 ? lane + hv : (role == 2 ? lane - hv : lane);
        float2 pm[P];
        if (unrounded) {
#pragma unroll
            for (int j = 0; j < P; ++j) {
                pm[j].x = __shfl_sync(0xffffffffu, src[j].x, from);
                pm[j].y = __shfl_sync(0xffffffffu, src[j].y, from);
            }
        } else {
            uint4 other;
            other.x = __shfl_sync(0xffffffffu, mine.x, from);
            other.y = __shfl_sync(0xffffffffu, mine.y, from);
            other.z = __shfl_sync(0xffffffffu, mine.z, from);
            other.w = __shfl_sync(0xffffffffu, mine.w, from);
            unpack_pairs<T, N>(other, pm);
        }
        if (role != 0) {
            // first member: x c - x' s; second: x c + x' s (the sine's sign
            // folded into the product, which rounds symmetrically)
            const float sg = role == 1 ? -1.0f : 1.0f;
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 sn = make_float2(sg * cr.s[2 * j], sg * cr.s[2 * j + 1]);
                y[j] = __ffma2_rn(src[j], make_float2(cr.c[2 * j], cr.c[2 * j + 1]), __fmul2_rn(pm[j], sn));
            }
        }
    }

    if (active) {
        if constexpr (FP8) {
            auto q8 = quantize_pairs<N>(y, p.inv);
            reinterpret_cast<decltype(q8)*>(dst)[sub] = q8;
        } else {
            reinterpret_cast<uint4*>(dst)[sub] = pack_pairs<T, N>(y);
        }
    }
}

template <typename T>
__device__ __forceinline__ void weights_plus_delta(const QKP& p, const char* wptr, int sub,
                                                   float (&w)[vec_elems<T>()]) {
    constexpr int N = vec_elems<T>();
    if (wptr != nullptr) {
        uint4 wr = __ldg(reinterpret_cast<const uint4*>(wptr) + sub);
        unpack_vec<T, N>(wr, w);
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = __fadd_rn(w[i], p.delta);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = 1.0f;
    }
}

// qk_core for a head held as two 16-byte vectors per lane of an LPH-lane
// group: vectors sub (raw0, weights w0) and sub + LPH (raw1, w1).  Rotate-half
// heads whose rotary channels all lie in the first LPH vectors, in the
// rounded mode, so only the first vector rotates (partner over the same
// shuffle as qk_core).  All 32 lanes of the warp call this together.
//  copy: pass the head through unnormalized and unrotated (the v heads of the
//  fused QKV op); the lane group still joins the warp-wide reduction.
template <typename T, bool FP8, int LPH>
__device__ __forceinline__ void qk_core2(const QKP& p, char* dst, bool active, int lane, int sub,
                                         const uint4& raw0, const uint4& raw1,
                                         const float (&w0)[vec_elems<T>()],
                                         const float (&w1)[vec_elems<T>()], int role,
                                         const CacheRegs<T, kRotateHalf>& cr, bool copy = false) {
    constexpr int N = vec_elems<T>();
    constexpr int P = N / 2;
    // normalized values n (x itself without normalization or for a copy),
    // rounded to the dtype as `mine` (first vector) and `mine1` (second); the
    // values of a copy are already in the dtype, so its packs are exact
    float2 x0[P], x1[P], n0[P], n1[P];
    unpack_pairs<T, N>(raw0, x0);
    unpack_pairs<T, N>(raw1, x1);
#pragma unroll
    for (int j = 0; j < P; ++j) {
        n0[j] = x0[j];
        n1[j] = x1[j];
    }
    if (p.mode & kModeNorm) {
        float2 s2 = splat2(0.0f);
#pragma unroll
        for (int j = 0; j < P; ++j) s2 = __ffma2_rn(x0[j], x0[j], s2);
#pragma unroll
        for (int j = 0; j < P; ++j) s2 = __ffma2_rn(x1[j], x1[j], s2);
        const float ss = group_sum<LPH>(__fadd_rn(s2.x, s2.y));
        const float2 r2 = splat2(inv_rms(ss, p.invD, p.eps));
        if (!copy) {
#pragma unroll
            for (int j = 0; j < P; ++j) {
                n0[j] = __fmul2_rn(__fmul2_rn(x0[j], r2), make_float2(w0[2 * j], w0[2 * j + 1]));
                n1[j] = __fmul2_rn(__fmul2_rn(x1[j], r2), make_float2(w1[2 * j], w1[2 * j + 1]));
            }
        }
    }
    const uint4 mine = pack_pairs<T, N>(n0);
    const uint4 mine1 = pack_pairs<T, N>(n1);
    float2 m[P], y[P];
    unpack_pairs<T, N>(mine, m);
#pragma unroll
    for (int j = 0; j < P; ++j) y[j] = m[j];

    // rotate-half on the first vector: the partner is half/N lanes away
    const int hv = p.half / N;
    const int from = role == 1 ? lane + hv : (role == 2 ? lane - hv : lane);
    uint4 other;
    other.x = __shfl_sync(0xffffffffu, mine.x, from);
    other.y = __shfl_sync(0xffffffffu, mine.y, from);
    other.z = __shfl_sync(0xffffffffu, mine.z, from);
    other.w = __shfl_sync(0xffffffffu, mine.w, from);
    float2 pm[P];
    unpack_pairs<T, N>(other, pm);
    if (role != 0) {
        // first member: x c - x' s; second: x c + x' s (the sine's sign
        // folded into the product, which rounds symmetrically)
        const float sg = role == 1 ? -1.0f : 1.0f;
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const float2 sn = make_float2(sg * cr.s[2 * j], sg * cr.s[2 * j + 1]);
            y[j] = __ffma2_rn(m[j], make_float2(cr.c[2 * j], cr.c[2 * j + 1]), __fmul2_rn(pm[j], sn));
        }
    }
    if (active) {
        if constexpr (FP8) {
            float2 m1[P];
            unpack_pairs<T, N>(mine1, m1);
            auto q0 = quantize_pairs<N>(y, p.inv);
            auto q1 = quantize_pairs<N>(m1, p.inv);
            reinterpret_cast<decltype(q0)*>(dst)[sub] = q0;
            reinterpret_cast<decltype(q1)*>(dst)[sub + LPH] = q1;
        } else {
            reinterpret_cast<uint4*>(dst)[sub] = role != 0 ? pack_pairs<T, N>(y) : mine;
            reinterpret_cast<uint4*>(dst)[sub + LPH] = mine1;
        }
    }
}

// Threads-per-head path for many heads (qk_quad.cu).  *handled is false when
// the geometry is outside its instantiations; the caller then takes the
// lane-group path.
// ---------------------------------------------------------------- generic head

template <typename T>
__device__ __forceinline__ float ld_elem(const char* base, int i) {
    return to_f(reinterpret_cast<const T*>(base)[i]);
}

// One head of any size or alignment, by one warp, staged as fp32 in hm[D]
// (shared memory).  With `norm` the head is normalized and weighted, and the
// staged value is what the rotation consumes: rounded to T, or left in fp32
// in the unrounded mode.  The first p.rot channels rotate when token t's
// position is inside the cache.  Every output is rounded once to T (or takes
// the FP8 epilogue).
template <typename T, bool FP8>
__device__ void generic_head(const QKP& p, const char* src, char* dst, const char* w, int64_t t,
                             bool norm, float* hm, int lane, int layout) {
    float ss = 0.0f;
    for (int e = lane; e < p.D; e += 32) {
        const float v = ld_elem<T>(src, e);
        hm[e] = v;
        ss = __fmaf_rn(v, v, ss);
    }
    if (norm) {
        ss = group_sum<32>(ss);
        const float r = inv_rms(ss, p.invD, p.eps);
        const bool unrounded = (p.mode & kModeUnrounded) != 0;
        for (int e = lane; e < p.D; e += 32) {
            const float wd = w ? __fadd_rn(ld_elem<T>(w, e), p.delta) : 1.0f;
            const float n = __fmul_rn(__fmul_rn(hm[e], r), wd);
            hm[e] = unrounded ? n : round_to<T>(n);
        }
    }
    __syncwarp();
    int64_t pos = -1;
    if (p.rot > 0) pos = p.pos[t];
    const bool rot = pos >= 0 && pos < p.cache_len;
    for (int e = lane; e < p.D; e += 32) {
        float y = round_to<T>(hm[e]);
        if (rot && e < p.rot) {
            int j, partner;
            bool first;
            if (layout == kInterleaved) {
                j = e >> 1;
                partner = e ^ 1;
                first = (e & 1) == 0;
            } else {
                first = e < p.half;
                j = first ? e : e - p.half;
                partner = first ? e + p.half : e - p.half;
            }
            const float c = p.cs[pos * p.half + j];
            const float sn = p.sn[pos * p.half + j];
            const float own = hm[e], other = hm[partner];
            y = first ? __fmaf_rn(own, c, -__fmul_rn(other, sn))
                      : __fmaf_rn(own, c, __fmul_rn(other, sn));
        }
        if constexpr (FP8) {
            reinterpret_cast<uint8_t*>(dst)[e] = quantize1(y, p.inv);
        } else {
            reinterpret_cast<T*>(dst)[e] = from_f<T>(y);
        }
    }
    __syncwarp();
}

template <typename T, bool FP8>
cudaError_t launch_qk_quad(const QKArgs& a, const QKP& p, cudaLaunchConfig_t cfg, bool* handled);

// Whether the four-threads-per-head path suits a geometry at all (past the
// geometry's quad_min_waves of the lane-group grid).
bool quad_suits(int layout, int rotary_dim, int64_t head_bytes);

// Waves of the lane-group grid beyond which the four-threads-per-head path
// takes over the prologue (measured per geometry).
double quad_min_waves(int elem_bytes, int layout, int rotary_dim, int64_t head_bytes);

// Arguments of the fused QKV kernels: the prologue's QKP (q = the fused qkv
// rows, qo = q_out; k and ko unused) and the cache side.
struct QKVP {
    QKP p;
    char* kc;              // k_cache
    char* vc;              // v_cache
    const int64_t* slots;  // nullable: no cache rows
    int64_t num_slots;
    int64_t row_bytes;     // bytes of one qkv row
    FastDiv per_token;     // Hq + 2 Hk
};

// The four-threads-per-head path for the fused QKV op; *handled is false
// when the geometry or alignment is outside the path (nothing launched).
template <typename T>
cudaError_t launch_qkv_quad(const QKVArgs& a, const QKVP& k, cudaLaunchConfig_t cfg,
                            bool* handled);

}  // namespace edge
