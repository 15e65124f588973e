// qkv_cache.cu -- fused QKV split + QK-norm + RoPE + KV-cache write (sm_103a).
//
// What it computes (FlashRT "optimization-details": qkv_split_rope_kvcache;
// "thox-edge-ops v2", roadmap item 4, a KV write fused into the prologue).
// Row t of the fused projection output qkv [T, (Hq + 2 Hk) D] holds Hq query
// heads, Hk key heads and Hk value heads.
//   - Query heads get the prologue (optional per-head RMSNorm, rounded to the
//     dtype, rotary embedding of the first rotary_dim channels) into
//     q_out[t].
//   - Key heads get the same into k_cache[slots[t]].
//   - Value heads are copied unchanged into v_cache[slots[t]].
// Caches are [num_slots, Hk, D].  A token whose slot is outside [0, num_slots)
// writes no cache row, so it cannot write out of bounds; its query still goes
// to q_out.
//
// GB300 design: the lane-group layout of the decode-width prologue.  A head is
// one 16-byte vector per lane of an LPH-lane group, and a one-shot grid puts
// every head in flight, the regime of decode widths.  Units are token-major
// over the Hq + 2 Hk heads of a row.  A v head rides the same code with no
// norm and no rotation, so a warp never diverges around the shuffles.  Mid
// widths of the text-profile heads take two vectors per lane, and many
// heads four threads per head (qk_quad.cu), as in the prologue.
#include "qk_common.cuh"

namespace edge {
namespace {

template <typename T, int LPH, int LAYOUT>
__global__ void __launch_bounds__(256) qkv_vec_kernel(QKVP a) {
    constexpr int N = vec_elems<T>();
    constexpr int HPW = 32 / LPH;
    const QKP& p = a.p;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPH - 1);
    const int hb = p.D * (int)sizeof(T);
    // one-shot grid; < 2^31 + 8 HPW since units are at most 2^31 - 1
    const uint32_t u = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * HPW + lane / LPH;
    const bool active = u < p.units;
    const uint32_t t = fast_div(active ? u : 0, a.per_token);
    const int h = (int)((active ? u : 0) - t * a.per_token.d);
    const char* src = p.q + (int64_t)t * a.row_bytes + (int64_t)h * hb;
    const bool isq = h < p.q_heads;
    const bool isv = h >= p.q_heads + p.k_heads;
    const int j = isq ? h : (isv ? h - p.q_heads - p.k_heads : h - p.q_heads);

    if (threadIdx.x == 0) {
        // the qkv rows of this CTA's units into L2 while the preceding grid
        // drains
        const uint32_t per_cta = (blockDim.x >> 5) * HPW;
        const uint32_t u0 = blockIdx.x * per_cta;
        const uint32_t u1 = u0 + per_cta < p.units ? u0 + per_cta : p.units;
        if (u0 < u1) {
            const int64_t t0 = fast_div(u0, a.per_token), t1 = fast_div(u1 - 1, a.per_token) + 1;
            prefetch_l2(p.q, t0 * a.row_bytes, t1 * a.row_bytes);
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    const int lane_role = p.rot > 0 ? rotary_role<T, LAYOUT>(p, sub) : 0;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    int64_t pos = -1, slot = -1;
    if (active) {
        raw = __ldcs(reinterpret_cast<const uint4*>(src) + sub);
        if (p.rot > 0 && !isv) pos = __ldg(p.pos + t);
        if (!isq && a.slots != nullptr) slot = __ldg(a.slots + t);
    }
    char* dst = nullptr;
    if (isq) {
        dst = p.qo + ((int64_t)t * p.q_heads + j) * hb;
    } else if (slot >= 0 && slot < a.num_slots) {
        dst = (isv ? a.vc : a.kc) + (slot * p.k_heads + j) * hb;
    }
    float w[N];
    weights_plus_delta<T>(p, isq ? p.wq : p.wk, sub, w);
    const bool rot = active && !isv && pos >= 0 && pos < p.cache_len;
    const int role = rot ? lane_role : 0;
    CacheRegs<T, LAYOUT> cr;
    if (role != 0) load_cache<T, LAYOUT>(p, pos, sub, role, cr);
    qk_core<T, false, LPH, LAYOUT>(p, dst, active && dst != nullptr, lane, sub, raw, w, role, cr,
                                   isv);
}

// Two vectors per lane for mid widths, as in the prologue: lane sub of a
// 16-lane group holds vectors sub and sub + LPH of one head, two heads per
// warp.  Rotate-half heads whose rotary channels lie in the first LPH
// vectors; a v head is copied exactly (no norm, no rotation).  Held to 64
// registers: 4 CTAs of 256 threads per SM, as the prologue's form.
template <typename T, int LPH>
__global__ void __launch_bounds__(256, 4) qkv_vec2_kernel(QKVP a) {
    constexpr int N = vec_elems<T>();
    constexpr int HPW = 32 / LPH;
    const QKP& p = a.p;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPH - 1);
    const int hb = p.D * (int)sizeof(T);
    // one-shot grid; < 2^31 + 8 HPW since units are at most 2^31 - 1
    const uint32_t u = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * HPW + lane / LPH;
    const bool active = u < p.units;
    const uint32_t t = fast_div(active ? u : 0, a.per_token);
    const int h = (int)((active ? u : 0) - t * a.per_token.d);
    const char* src = p.q + (int64_t)t * a.row_bytes + (int64_t)h * hb;
    const bool isq = h < p.q_heads;
    const bool isv = h >= p.q_heads + p.k_heads;
    const int j = isq ? h : (isv ? h - p.q_heads - p.k_heads : h - p.q_heads);

    if (threadIdx.x == 0) {
        const uint32_t per_cta = (blockDim.x >> 5) * HPW;
        const uint32_t u0 = blockIdx.x * per_cta;
        const uint32_t u1 = u0 + per_cta < p.units ? u0 + per_cta : p.units;
        if (u0 < u1) {
            const int64_t t0 = fast_div(u0, a.per_token), t1 = fast_div(u1 - 1, a.per_token) + 1;
            prefetch_l2(p.q, t0 * a.row_bytes, t1 * a.row_bytes);
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    const int lane_role = p.rot > 0 ? rotary_role<T, kRotateHalf>(p, sub) : 0;
    uint4 raw0 = make_uint4(0u, 0u, 0u, 0u), raw1 = raw0;
    int64_t pos = -1, slot = -1;
    if (active) {
        raw0 = __ldcs(reinterpret_cast<const uint4*>(src) + sub);
        raw1 = __ldcs(reinterpret_cast<const uint4*>(src) + sub + LPH);
        if (p.rot > 0 && !isv) pos = __ldg(p.pos + t);
        if (!isq && a.slots != nullptr) slot = __ldg(a.slots + t);
    }
    char* dst = nullptr;
    if (isq) {
        dst = p.qo + ((int64_t)t * p.q_heads + j) * hb;
    } else if (slot >= 0 && slot < a.num_slots) {
        dst = (isv ? a.vc : a.kc) + (slot * p.k_heads + j) * hb;
    }
    float w0[N], w1[N];
    weights_plus_delta<T>(p, isq ? p.wq : p.wk, sub, w0);
    weights_plus_delta<T>(p, isq ? p.wq : p.wk, sub + LPH, w1);
    const bool rot = active && !isv && pos >= 0 && pos < p.cache_len;
    const int role = rot ? lane_role : 0;
    CacheRegs<T, kRotateHalf> cr;
    if (role != 0) load_cache<T, kRotateHalf>(p, pos, sub, role, cr);

    qk_core2<T, false, LPH>(p, dst, active && dst != nullptr, lane, sub, raw0, raw1, w0, w1, role,
                            cr, isv);
}

// Any head size or alignment: one warp per head, staged in shared memory.
template <typename T>
__global__ void __launch_bounds__(128) qkv_generic_kernel(QKVP a, int layout) {
    extern __shared__ float qkv_smem[];
    const QKP& p = a.p;
    const int lane = threadIdx.x & 31;
    float* hm = qkv_smem + (threadIdx.x >> 5) * p.D;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const int64_t hb = (int64_t)p.D * (int64_t)sizeof(T);

    pdl_wait();
    pdl_launch_dependents();

    for (uint32_t u = warp; u < p.units; u += nwarps) {
        const uint32_t t = fast_div(u, a.per_token);
        const int h = (int)(u - t * a.per_token.d);
        const char* src = p.q + (int64_t)t * a.row_bytes + h * hb;
        const bool isq = h < p.q_heads;
        const bool isv = h >= p.q_heads + p.k_heads;
        const int j = isq ? h : (isv ? h - p.q_heads - p.k_heads : h - p.q_heads);
        char* dst;
        if (isq) {
            dst = p.qo + ((int64_t)t * p.q_heads + j) * hb;
        } else {
            // no cache (slots NULL) or a slot outside it: no cache row; the
            // same for the whole warp
            const int64_t slot = a.slots != nullptr ? a.slots[t] : -1;
            if (slot < 0 || slot >= a.num_slots) continue;
            dst = (isv ? a.vc : a.kc) + (slot * p.k_heads + j) * hb;
        }
        if (isv) {
            for (int e = lane; e < p.D; e += 32) {
                reinterpret_cast<T*>(dst)[e] = reinterpret_cast<const T*>(src)[e];
            }
        } else {
            generic_head<T, false>(p, src, dst, isq ? p.wq : p.wk, t, (p.mode & kModeNorm) != 0,
                                   hm, lane, layout);
        }
    }
}

template <typename T, int LPH>
void (*qkv_vec_fn(int layout))(QKVP) {
    return layout == kInterleaved ? qkv_vec_kernel<T, LPH, kInterleaved>
                                  : qkv_vec_kernel<T, LPH, kRotateHalf>;
}

template <typename T>
cudaError_t launch_typed(const QKVArgs& a, QKVP& k, cudaStream_t s, bool* handled) {
    constexpr int N = vec_elems<T>();
    *handled = false;
    const int D = a.head_dim;
    const int nvec = (D * (int)sizeof(T)) % 16 == 0 ? D * (int)sizeof(T) / 16 : 0;
    auto aligned = [](const void* ptr, uintptr_t n) {
        return ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) % n) == 0;
    };
    bool vec = nvec > 0 && nvec <= 32 && (nvec & (nvec - 1)) == 0;
    vec = vec && aligned(a.qkv, 16) && aligned(a.wq, 16) && aligned(a.wk, 16) &&
          aligned(a.q_out, 16) && aligned(a.k_cache, 16) && aligned(a.v_cache, 16);
    if (k.p.rot > 0) {
        if (a.layout == kInterleaved) {
            vec = vec && k.p.rot % N == 0 && aligned(a.cos, 8 * (N / 4)) && aligned(a.sin, 8 * (N / 4));
        } else {
            vec = vec && (k.p.rot / 2) % N == 0 && aligned(a.cos, 16) && aligned(a.sin, 16);
        }
    }
    *handled = true;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    if (!vec) {
        const int threads = 128;
        int64_t blocks = ((int64_t)k.p.units + threads / 32 - 1) / (threads / 32);
        const int64_t cap = (int64_t)sm_count() * 16;
        if (blocks > cap) blocks = cap;
        const size_t smem = (size_t)(threads / 32) * D * sizeof(float);
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(qkv_generic_kernel<T>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        return cudaLaunchKernelEx(&cfg, qkv_generic_kernel<T>, k, a.layout);
    }
    const int lph = nvec;
    const int hpw = 32 / lph;
    void (*vfn)(QKVP) = nullptr;
    switch (lph) {
        case 1: vfn = qkv_vec_fn<T, 1>(a.layout); break;
        case 2: vfn = qkv_vec_fn<T, 2>(a.layout); break;
        case 4: vfn = qkv_vec_fn<T, 4>(a.layout); break;
        case 8: vfn = qkv_vec_fn<T, 8>(a.layout); break;
        case 16: vfn = qkv_vec_fn<T, 16>(a.layout); break;
        default: vfn = qkv_vec_fn<T, 32>(a.layout); break;
    }
    const int threads = 256;
    const int64_t per_block = (int64_t)(threads / 32) * hpw;
    int64_t blocks = ((int64_t)k.p.units + per_block - 1) / per_block;
    // the prologue's rule: the one-shot lane-group grid while it fits in one
    // wave of resident CTAs, four threads per head beyond; for 16-bit
    // rotate-half heads of 512 bytes whose rotary channels lie in the first
    // half, the prologue's three bands in waves w of the one-vector grid
    // (one vector to 0.25 and from 0.8 to 1, two vectors elsewhere up to 1.6,
    // four threads per head beyond)
    const int64_t wave = (int64_t)resident_ctas((const void*)vfn, threads) * sm_count();
    const bool two = sizeof(T) == 2 && D * (int)sizeof(T) == 512 && a.layout == kRotateHalf &&
                     k.p.rot <= D / 2;
    const double w = (double)blocks / (double)wave;
    const bool take_quad = two ? w > 1.6 : blocks > wave;
    if (take_quad && quad_suits(a.layout, k.p.rot, (int64_t)D * (int64_t)sizeof(T))) {
        bool quad = false;
        cudaError_t e = launch_qkv_quad<T>(a, k, cfg, &quad);
        if (quad || e != cudaSuccess) return e;
    }
    if constexpr (sizeof(T) == 2) {
        if (two && w > 0.25 && !(w > 0.8 && w <= 1.0)) {
            const int64_t per2 = (int64_t)(threads / 32) * 2;
            cfg.gridDim = dim3((unsigned)(((int64_t)k.p.units + per2 - 1) / per2));
            cfg.blockDim = dim3(threads);
            cfg.dynamicSmemBytes = 0;
            return cudaLaunchKernelEx(&cfg, qkv_vec2_kernel<T, 16>, k);
        }
    }
    cfg.gridDim = dim3((unsigned)blocks);  // one-shot: blocks < 2^28
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, vfn, k);
}

}  // namespace

cudaError_t launch_qkv_cache(const QKVArgs& a, cudaStream_t s, bool* handled) {
    QKVP k;
    QKP& p = k.p;
    const int es = a.dt == kF32 ? 4 : 2;
    const bool may_rotate = a.rotary_dim > 0 && a.cache_len > 0 && a.pos && a.cos && a.sin;
    p.q = static_cast<const char*>(a.qkv);
    p.k = nullptr;
    p.qo = static_cast<char*>(a.q_out);
    p.ko = nullptr;
    p.wq = static_cast<const char*>(a.wq);
    p.wk = static_cast<const char*>(a.wk);
    p.pos = a.pos;
    p.cs = a.cos;
    p.sn = a.sin;
    p.cache_len = may_rotate ? a.cache_len : 0;
    p.tokens = a.tokens;
    p.units = (uint32_t)(a.tokens * (a.q_heads + 2 * a.kv_heads));
    p.heads = make_fastdiv((uint32_t)(a.q_heads + 2 * a.kv_heads));
    p.qdiv = make_fastdiv((uint32_t)a.q_heads);
    p.kdiv = make_fastdiv((uint32_t)(a.kv_heads > 0 ? a.kv_heads : 1));
    p.qrows = (uint32_t)(a.tokens * a.q_heads);
    p.q_heads = a.q_heads;
    p.k_heads = a.kv_heads;
    p.D = a.head_dim;
    p.rot = may_rotate ? a.rotary_dim : 0;
    p.half = p.rot / 2;
    p.in_bytes = es;
    p.out_bytes = es;
    p.eps = a.eps;
    p.delta = (float)a.weight_offset;
    p.inv = 1.0f;
    p.invD = 1.0f / (float)a.head_dim;
    p.mode = a.normalize ? kModeNorm : 0;
    k.kc = static_cast<char*>(a.k_cache);
    k.vc = static_cast<char*>(a.v_cache);
    k.slots = a.slots;
    k.num_slots = a.num_slots;
    k.row_bytes = (int64_t)(a.q_heads + 2 * a.kv_heads) * a.head_dim * es;
    k.per_token = p.heads;
    switch (a.dt) {
        case kF32: return launch_typed<float>(a, k, s, handled);
        case kF16: return launch_typed<__half>(a, k, s, handled);
        default: return launch_typed<__nv_bfloat16>(a, k, s, handled);
    }
}

}  // namespace edge
