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
// known at compile time.  A head's cos/sin lines are prefetched into L1 as its
// arithmetic begins, so the rotation reads them without another round trip.  About 50 warp-instructions per head remain.  All C
// loads of a thread are issued before any arithmetic, so a warp (8 heads) has
// 4 KB in flight.
//
// The same body serves the fused QKV op (qkv_cache.cu): a mapper gives each
// head unit its source, destination and kind.  Value heads take the body with
// a unit weight and no norm or rotation, so a warp never diverges on them and
// their bits are copied exactly.
#include "qk_common.cuh"

namespace edge {
namespace {

constexpr int K = 4;  // threads per head

// Register budget per thread, stated as CTAs of 256 threads per SM (65536
// registers per SM); the 64- and 128-thread CTAs used at launch hold the same
// registers per thread.  Fewer elements per thread leave fewer live values,
// so more threads fit: 5 CTAs (51 registers) for 128-byte heads and 4 (64)
// for 256-byte heads, both without spills; 3 (85) for 512-byte heads; 2 (128)
// with the FP8 epilogue, and for 16-bit 512-byte heads (64 elements per
// thread) that are interleaved or have more than two rotate-half chunks per
// thread.  Measured on GB300: those 16-bit heads ran faster at 2 CTAs than at
// 3 with spills, while fp32 512-byte heads (32 elements per thread) ran
// faster at 3 CTAs, spilling about a hundred bytes, than at 2.
// With PIPE a thread holds two heads' chunks, so each size steps down one
// CTA count: 4 for 128-byte heads, 3 for 256-byte heads, 2 for 512-byte heads.
template <typename T, bool FP8, int C, int LAYOUT, int RQ, bool PIPE>
__host__ __device__ constexpr int quad_min_blocks() {
    return FP8 ? 2
           : PIPE ? (C <= 2 ? 4 : C <= 4 ? 3 : 2)
                  : C <= 2 ? 5
                  : C <= 4 ? 4
                  : (sizeof(T) == 2 && (LAYOUT == kInterleaved || 2 * RQ > 2)) ? 2 : 3;
}

// Which variants run the resident, load-ahead form.  Measured on GB300 at
// T = 1024 to 4096: 10-24% faster for 512-byte heads with at most two
// rotate-half chunks per thread (the text profiles, fp32 heads of 128),
// slower for 256-byte heads (whose one-pass form already holds 4 CTAs per SM)
// and no faster for 16-bit 512-byte heads that are interleaved or rotate
// fully (whose one-pass form already runs at 2 CTAs).
template <typename T, int C, int LAYOUT, int RQ>
__host__ __device__ constexpr bool quad_pipe() {
    return C == 8 && !(sizeof(T) == 2 && (LAYOUT == kInterleaved || 2 * RQ > 2));
}

constexpr int kKindQ = 0, kKindK = 1, kKindV = 2;

// One head unit: where its chunks come from and go to.
struct QuadUnit {
    const char* src;
    char* dst;     // nullptr: nothing to store (a cache head without a slot)
    uint32_t t;    // token
    int kind;      // kKindQ, kKindK or kKindV
};

// The two-tensor prologue: all q rows, then all k rows.  Every unit is a
// query or key head with a destination.
struct QKMap {
    static constexpr bool kHasV = false;
    __device__ __forceinline__ QuadUnit unit(const QKP& p, uint32_t u, uint32_t hb) const {
        const bool isq = u < p.qrows;
        const uint32_t row = isq ? u : u - p.qrows;
        QuadUnit r;
        r.t = fast_div(row, isq ? p.qdiv : p.kdiv);
        r.src = (isq ? p.q : p.k) + (size_t)row * hb;
        r.dst = (isq ? p.qo : p.ko) + (size_t)row * (size_t)p.D * p.out_bytes;
        r.kind = isq ? kKindQ : kKindK;
        return r;
    }
    __device__ __forceinline__ void prefetch(const QKP& p, uint32_t u0, uint32_t u1) const {
        prefetch_heads(p, u0, u1, false);
    }
};

// Fused QKV rows [Hq q heads | Hk k heads | Hk v heads] per token, token-major;
// k and v heads go to row slots[t] of their cache (nowhere when out of range).
struct QKVMap {
    static constexpr bool kHasV = true;  // value heads, and units with no destination
    const QKVP* a;
    __device__ __forceinline__ QuadUnit unit(const QKP& p, uint32_t u, uint32_t hb) const {
        const uint32_t t = fast_div(u, a->per_token);
        const int h = (int)(u - t * a->per_token.d);
        QuadUnit r;
        r.t = t;
        r.src = p.q + (int64_t)t * a->row_bytes + (int64_t)h * hb;
        if (h < p.q_heads) {
            r.kind = kKindQ;
            r.dst = p.qo + ((int64_t)t * p.q_heads + h) * hb;
        } else {
            const bool isv = h >= p.q_heads + p.k_heads;
            const int j = isv ? h - p.q_heads - p.k_heads : h - p.q_heads;
            r.kind = isv ? kKindV : kKindK;
            const int64_t slot = a->slots != nullptr ? __ldg(a->slots + t) : -1;
            r.dst = (slot >= 0 && slot < a->num_slots)
                        ? (isv ? a->vc : a->kc) + (slot * p.k_heads + j) * hb
                        : nullptr;
        }
        return r;
    }
    __device__ __forceinline__ void prefetch(const QKP& p, uint32_t u0, uint32_t u1) const {
        if (u1 > p.units) u1 = p.units;
        if (u0 >= u1) return;
        const int64_t t0 = fast_div(u0, a->per_token), t1 = fast_div(u1 - 1, a->per_token) + 1;
        prefetch_l2(p.q, t0 * a->row_bytes, t1 * a->row_bytes);
    }
};

// One head unit's loaded chunks and what the arithmetic needs besides them.
template <int C>
struct QuadHead {
    uint4 raw[C];
    QuadUnit un;
    int64_t pos;
    bool active, isv;
};

// RQ: rotate-half: chunks per thread that are first members (HVQ); interleaved:
// chunks per thread that rotate.  0: no channel rotates.
// PIPE: a resident grid in which every thread issues its next head's loads
// before the arithmetic of the current one, so that memory and arithmetic
// overlap across iterations instead of alternating in lockstep waves.
// UNR: the unrounded form (the rotation takes the fp32 normalized value; one
// rounding after it), for the instantiated geometries only.
template <typename T, bool FP8, int C, int LAYOUT, int RQ, bool PIPE, class Map, bool UNR = false>
__device__ __forceinline__ void quad_body(const QKP& p, const Map& map) {
    constexpr int N = vec_elems<T>();
    constexpr int D = C * K * N;
    // chunks whose fp32 normalized values the unrounded rotation needs
    constexpr int RC = UNR ? (LAYOUT == kInterleaved ? RQ : 2 * RQ) : 0;
    static_assert(LAYOUT == kInterleaved ? RQ <= C : 2 * RQ <= C, "rotated chunks exceed the head");
    // w + delta in fp32 (1 when no weight) for q heads, k heads, and 1 for v
    __shared__ __align__(16) float wsm[3][D];

    const int heads_per_cta = blockDim.x / K;
    if (threadIdx.x == 0) {
        map.prefetch(p, blockIdx.x * heads_per_cta, (blockIdx.x + 1) * heads_per_cta);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int kt = threadIdx.x & (K - 1);
    const int hs = threadIdx.x / K;           // head slot in the CTA
    const uint32_t hb = (uint32_t)D * sizeof(T);
    const uint32_t stride = gridDim.x * heads_per_cta;

    // The weights are staged while the first heads are in flight in the
    // prologue (measured 3-10% faster on GB300), and before the first heads in
    // the fused QKV op, whose value-head bookkeeping leaves no registers for
    // the overlap (measured 7% faster that way).
    auto stage = [&]() {
        for (int e = threadIdx.x; e < D; e += blockDim.x) {
            const float dq =
                p.wq ? __fadd_rn(to_f(reinterpret_cast<const T*>(p.wq)[e]), p.delta) : 1.0f;
            const float dk =
                p.wk ? __fadd_rn(to_f(reinterpret_cast<const T*>(p.wk)[e]), p.delta) : 1.0f;
            wsm[kKindQ][e] = dq;
            wsm[kKindK][e] = dk;
            wsm[kKindV][e] = 1.0f;
        }
        __syncthreads();
    };

    // issue every load of the unit in slot hs of the pass at `base`
    auto load = [&](uint32_t base, QuadHead<C>& h) {
        const uint32_t u = base + hs;
        h.active = u < p.units;
        h.un = map.unit(p, h.active ? u : base, hb);
#pragma unroll
        for (int i = 0; i < C; ++i) {
            h.raw[i] = h.active ? __ldcs(reinterpret_cast<const uint4*>(h.un.src) + kt + K * i)
                                : make_uint4(0u, 0u, 0u, 0u);
        }
        h.isv = Map::kHasV && h.un.kind == kKindV;
        h.pos = -1;
        if (RQ > 0 && h.active && !h.isv) h.pos = __ldg(p.pos + h.un.t);
    };

    // the arithmetic and stores of one loaded unit
    auto process = [&](QuadHead<C>& h) {
        uint4 (&raw)[C] = h.raw;
        const QuadUnit& un = h.un;
        const bool active = h.active, isv = h.isv;
        const int64_t pos = h.pos;
        const bool rot = RQ > 0 && pos >= 0 && pos < p.cache_len;
        if (rot) {
            // the cos/sin lines of the rotated chunks into L1 now, so that
            // their round trip overlaps the normalization below
#pragma unroll
            for (int i = 0; i < (RQ > 0 ? RQ : 1); ++i) {
                const int64_t e = pos * p.half + (kt + K * i) * (LAYOUT == kInterleaved ? N / 2 : N);
                prefetch_l1_line(p.cs + e);
                prefetch_l1_line(p.sn + e);
            }
        }
        // beyond 32 terms per thread, two running sums alternating by chunk
        // (at most 4N sequential terms each, for the error bound of the
        // tolerance)
        constexpr bool kSplit = C * N > 32;
        float ssp[2] = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < C; ++i) {
            float x[N];
            unpack_vec<T, N>(raw[i], x);
#pragma unroll
            for (int e = 0; e < N; ++e) {
                ssp[kSplit ? (i & 1) : 0] = __fmaf_rn(x[e], x[e], ssp[kSplit ? (i & 1) : 0]);
            }
        }
        float ss = kSplit ? __fadd_rn(ssp[0], ssp[1]) : ssp[0];
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        // without normalization (standalone rotary, the unnormalized QKV
        // form, value heads) r = 1 and w = 1: m = x exactly
        const bool norm = (p.mode & kModeNorm) && !isv;
        const float r = norm ? inv_rms(ss, p.invD, p.eps) : 1.0f;

        // normalized value rounded to the dtype, packed (exactly) over the
        // loaded vectors, which are no longer needed.  (The prologue's
        // unnormalized form, standalone rotary, passes no weights, so its
        // q/k rows hold 1.)
        const float* w = wsm[Map::kHasV ? (norm ? un.kind : kKindV) : un.kind];
        uint4 (&mp)[C] = raw;
        float mf[RC > 0 ? RC : 1][N];  // fp32 normalized values (unrounded form)
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
            if constexpr (RC > 0) {
                if (i < RC) {
#pragma unroll
                    for (int e = 0; e < N; ++e) mf[i < RC ? i : 0][e] = m[e];
                }
            }
            mp[i] = pack_vec<T, N>(m);
        }
        // the value a rotated chunk consumes: the dtype-rounded normalized
        // value, or its fp32 form in the unrounded mode
        auto rot_in = [&](int i, float (&a)[N]) {
            if constexpr (RC > 0) {
#pragma unroll
                for (int e = 0; e < N; ++e) a[e] = mf[i < RC ? i : 0][e];
            } else {
                unpack_vec<T, N>(mp[i], a);
            }
        };

        if (!active || (Map::kHasV && un.dst == nullptr)) return;
        char* out = un.dst;
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
                    rot_in(i, m);
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
                    rot_in(i, a);
                    rot_in(i + RQ, b);
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
    };

    uint32_t base = blockIdx.x * heads_per_cta;
    if (base >= p.units) return;  // the same for the whole CTA
    if constexpr (Map::kHasV) stage();
    QuadHead<C> h0;
    load(base, h0);
    if constexpr (!Map::kHasV) stage();
    if constexpr (PIPE) {
        // two buffers in turn: the next pass is loaded into one while the
        // other is processed (passes are the same for the whole CTA)
        QuadHead<C> h1;
        for (;;) {
            uint32_t next = base + stride;
            if (next >= p.units) {
                process(h0);
                break;
            }
            load(next, h1);
            process(h0);
            base = next;
            next = base + stride;
            if (next >= p.units) {
                process(h1);
                break;
            }
            load(next, h0);
            process(h1);
            base = next;
        }
    } else {
        for (;;) {
            process(h0);
            base += stride;
            if (base >= p.units) break;
            load(base, h0);
        }
    }
}

template <typename T, bool FP8, int C, int LAYOUT, int RQ, bool UNR = false>
__global__ void __launch_bounds__(256, (quad_min_blocks<T, FP8, C, LAYOUT, RQ,
                                                        quad_pipe<T, C, LAYOUT, RQ>()>()))
    qk_quad_kernel(QKP p) {
    quad_body<T, FP8, C, LAYOUT, RQ, quad_pipe<T, C, LAYOUT, RQ>(), QKMap, UNR>(p, QKMap{});
}

template <typename T, int C, int LAYOUT, int RQ>
__global__ void __launch_bounds__(256, (quad_min_blocks<T, false, C, LAYOUT, RQ,
                                                        quad_pipe<T, C, LAYOUT, RQ>()>()))
    qkv_quad_kernel(QKVP a) {
    quad_body<T, false, C, LAYOUT, RQ, quad_pipe<T, C, LAYOUT, RQ>()>(a.p, QKVMap{&a});
}

// Kernel selectors for pick_rq: the prologue (FP8 or not) and the fused QKV op.
template <typename T, bool FP8, int C, int LAYOUT, int RQ>
struct QKSel {
    static constexpr void (*fn)(QKP) = qk_quad_kernel<T, FP8, C, LAYOUT, RQ>;
};
template <typename T, bool FP8, int C, int LAYOUT, int RQ>
struct QKVSel {
    static constexpr void (*fn)(QKVP) = qkv_quad_kernel<T, C, LAYOUT, RQ>;
};

// The instantiated (C, layout, RQ) combinations: head sizes of 2, 4 or 8
// chunks per thread (D*s = 128, 256 or 512 bytes), every rotary width that
// keeps pairs thread-local.
template <template <typename, bool, int, int, int> class Sel, typename T, bool FP8, int C>
auto pick_rq(int layout, int rq) -> decltype(Sel<T, FP8, C, kRotateHalf, 0>::fn) {
    if (rq == 0) return Sel<T, FP8, C, kRotateHalf, 0>::fn;
    if (layout == kInterleaved) {
        switch (rq) {
            case 1: return Sel<T, FP8, C, kInterleaved, 1>::fn;
            case 2: return C >= 2 ? Sel<T, FP8, C, kInterleaved, (C >= 2 ? 2 : 1)>::fn : nullptr;
            case 4: return C >= 4 ? Sel<T, FP8, C, kInterleaved, (C >= 4 ? 4 : 1)>::fn : nullptr;
            case 8: return C >= 8 ? Sel<T, FP8, C, kInterleaved, (C >= 8 ? 8 : 1)>::fn : nullptr;
            default: return nullptr;
        }
    }
    switch (rq) {
        case 1: return Sel<T, FP8, C, kRotateHalf, 1>::fn;
        case 2: return C >= 4 ? Sel<T, FP8, C, kRotateHalf, (C >= 4 ? 2 : 1)>::fn : nullptr;
        case 4: return C >= 8 ? Sel<T, FP8, C, kRotateHalf, (C >= 8 ? 4 : 1)>::fn : nullptr;
        default: return nullptr;
    }
}

// Chunks per thread C and rotated chunks RQ of a geometry the path takes, or
// false: head bytes 128, 256 or 512; 16-byte aligned heads; a rotary width
// whose pairs stay in one thread; cache rows aligned for their vector loads.
template <typename T>
bool quad_shape(int head_dim, int rot, int layout, const void* const* bufs, int nbufs,
                const void* cs, const void* sn, int* C, int* rq) {
    constexpr int N = vec_elems<T>();
    const int64_t hb = (int64_t)head_dim * (int64_t)sizeof(T);
    if (hb % (16 * K) != 0) return false;
    *C = (int)(hb / (16 * K));
    if (*C != 2 && *C != 4 && *C != 8) return false;
    for (int i = 0; i < nbufs; ++i) {
        if (bufs[i] != nullptr && reinterpret_cast<uintptr_t>(bufs[i]) % 16 != 0) return false;
    }
    *rq = 0;
    if (rot > 0) {
        const int unit = (layout == kInterleaved ? 1 : 2) * K * N;
        if (rot % unit != 0) return false;
        const uintptr_t ca = layout == kInterleaved ? 8 * (N / 4) : 16;
        if (reinterpret_cast<uintptr_t>(cs) % ca != 0 || reinterpret_cast<uintptr_t>(sn) % ca != 0) {
            return false;
        }
        *rq = rot / unit;
    }
    return true;
}

// quad_pipe for run-time (C, layout, RQ)
template <typename T>
bool pipe_of(int C, int layout, int rq) {
    return C == 8 && !(sizeof(T) == 2 && (layout == kInterleaved || 2 * rq > 2));
}

// Threads per CTA: small CTAs spread mid-size work over every SM (16 heads
// per CTA for 512-byte heads, 32 for smaller ones).  Measured on GB300 at
// T = 128 to 4096: up to 25% faster than 64 heads per CTA at mid T, within
// a few percent at large T.
template <typename P, typename Fn>
cudaError_t launch_quad(Fn fn, const P& arg, uint32_t units, bool pipe, int C,
                        cudaLaunchConfig_t cfg) {
    const int threads = C == 8 ? 64 : 128;
    const int64_t per_block = threads / K;
    int64_t blocks = ((int64_t)units + per_block - 1) / per_block;
    // the load-ahead form needs every CTA resident for all its passes
    const int64_t cap = (int64_t)sm_count() * (pipe ? resident_ctas((const void*)fn, threads) : 64);
    if (blocks > cap) blocks = cap;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, fn, arg);
}

}  // namespace

template <typename T, bool FP8>
cudaError_t launch_qk_quad(const QKArgs& a, const QKP& p, cudaLaunchConfig_t cfg, bool* handled) {
    constexpr int N = vec_elems<T>();
    *handled = false;
    const bool unr = (a.mode & kModeUnrounded) != 0;
    // FP8 outputs are N bytes per chunk: alignment N
    if ((a.q_out && reinterpret_cast<uintptr_t>(a.q_out) % (FP8 ? N : 16) != 0) ||
        (a.k_out && reinterpret_cast<uintptr_t>(a.k_out) % (FP8 ? N : 16) != 0)) {
        return cudaSuccess;
    }
    const void* bufs[2] = {a.q, a.k};
    int C = 0, rq = 0;
    if (!quad_shape<T>(a.head_dim, p.rot, a.layout, bufs, 2, a.cos, a.sin, &C, &rq)) {
        return cudaSuccess;
    }
    void (*fn)(QKP) = nullptr;
    if (unr) {
        // the unrounded form for 16-bit rotate-half heads of 512 bytes with
        // rotary 64 (the text profiles) and of 256 bytes rotating fully;
        // other geometries take the lane-group path
        if constexpr (sizeof(T) == 2) {
            if (a.layout == kRotateHalf && C == 8 && rq == 1) {
                fn = qk_quad_kernel<T, FP8, 8, kRotateHalf, 1, true>;
            }
            if (a.layout == kRotateHalf && C == 4 && rq == 2) {
                fn = qk_quad_kernel<T, FP8, 4, kRotateHalf, 2, true>;
            }
        }
    } else {
        switch (C) {
            case 2: fn = pick_rq<QKSel, T, FP8, 2>(a.layout, rq); break;
            case 4: fn = pick_rq<QKSel, T, FP8, 4>(a.layout, rq); break;
            default: fn = pick_rq<QKSel, T, FP8, 8>(a.layout, rq); break;
        }
    }
    if (fn == nullptr) return cudaSuccess;
    *handled = true;
    return launch_quad(fn, p, p.units, pipe_of<T>(C, a.layout, rq), C, cfg);
}

template <typename T>
cudaError_t launch_qkv_quad(const QKVArgs& a, const QKVP& k, cudaLaunchConfig_t cfg,
                            bool* handled) {
    *handled = false;
    const void* bufs[4] = {a.qkv, a.q_out, a.k_cache, a.v_cache};
    int C = 0, rq = 0;
    if (!quad_shape<T>(a.head_dim, k.p.rot, a.layout, bufs, 4, a.cos, a.sin, &C, &rq)) {
        return cudaSuccess;
    }
    void (*fn)(QKVP) = nullptr;
    switch (C) {
        case 2: fn = pick_rq<QKVSel, T, false, 2>(a.layout, rq); break;
        case 4: fn = pick_rq<QKVSel, T, false, 4>(a.layout, rq); break;
        default: fn = pick_rq<QKVSel, T, false, 8>(a.layout, rq); break;
    }
    if (fn == nullptr) return cudaSuccess;
    *handled = true;
    return launch_quad(fn, k, k.p.units, pipe_of<T>(C, a.layout, rq), C, cfg);
}

double quad_min_waves(int elem_bytes, int layout, int rotary_dim, int64_t head_bytes) {
    // Measured on GB300, lane-group against four threads per head, T = 64 to
    // 2048 in back-to-back cold launches, for the text profiles (with and
    // without FP8 output), DFlash2, context-K, 16-bit 512-byte heads rotating
    // fully and fp32 heads of 128: every 16-bit geometry crosses at about one
    // wave of the lane-group grid, fp32 heads at about two.  With each buffer
    // set's own cos/sin cache the lane group wins by 3-10% up to 0.9 of a
    // wave; with one cache shared by every set (its rows L2-resident, as when
    // the layers of a step share the positions) the four-thread path wins
    // the (16,2) text profile by 4-5% from 0.57 of a wave, the one point where
    // the two disagree.
    (void)layout;
    (void)rotary_dim;
    (void)head_bytes;
    return elem_bytes == 4 ? 2.0 : 1.0;
}

bool quad_suits(int layout, int rotary_dim, int64_t head_bytes) {
    // 512-byte heads in the interleaved layout need the two-CTA register
    // budget.  Measured on GB300, this path then wins at some widths and
    // loses at others, by up to 15% each way (every partial wave of its grid
    // costs a full pass), so the lane-group path keeps them.
    return !(layout == kInterleaved && rotary_dim > 0 && head_bytes == 512);
}

template cudaError_t launch_qk_quad<float, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<float, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__half, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__half, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__nv_bfloat16, false>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qk_quad<__nv_bfloat16, true>(const QKArgs&, const QKP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qkv_quad<float>(const QKVArgs&, const QKVP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qkv_quad<__half>(const QKVArgs&, const QKVP&, cudaLaunchConfig_t, bool*);
template cudaError_t launch_qkv_quad<__nv_bfloat16>(const QKVArgs&, const QKVP&, cudaLaunchConfig_t, bool*);

}  // namespace edge
