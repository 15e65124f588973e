// qk_norm_rope.cu -- fused per-head QK-RMSNorm + RoPE prologue (sm_103a).
//
// What it computes ("thox-edge-ops v2", sections 5.1 and 5.4; ninfer text
// profile, "Implementation"): every head of q (weight wq) and of k (weight wk)
// of token t is normalized by its own RMSNorm and rounded to the activation
// dtype.  If 0 <= positions[t] < cache_len, the first rotary_dim channels are
// then rotated by cos/sin row positions[t] and rounded once more.  Channels
// past rotary_dim carry the rounded normalized value.  An out-of-cache token
// is normalized, not rotated, and reads no cache row.
//
// GB300 design.  The op is HBM-bound: it reads each head once and writes it
// once, about 2 flops per byte.  One head is a "unit".  Fast path: a head of
// D elements is held by LPH = D*s/16 lanes, one 16-byte vector per lane, so a
// warp holds 32/LPH heads (bf16 D=256: one head per warp; bf16 D=128: two).
//   - The sum of squares is reduced with xor-shuffles inside the lane group.
//   - The rotate-half partner vector sits half/N lanes away and comes over a
//     shuffle.  Interleaved pairs sit inside one vector.
//   - cos/sin entries are read from L1: every head of a token shares the row.
//   - The grid is one-shot: one unit per lane group, its address computed
//     before the dependent-launch wait.
// Units are ordered token-major, so the warps of a CTA share cos/sin rows and
// the norm weights.  Streamed inputs use evict-first loads.
// Mid widths, for 16-bit 512-byte rotate-half heads whose rotary channels
// lie in the first half (the text profiles): the same layout with two
// vectors per lane, 16 lanes per head.  Many heads: the four-threads-per-head
// path (qk_quad.cu) takes over past a measured number of waves of this
// path's grid (quad_min_waves; 1.6 for the heads with the two-vector form).
// Generic path: one warp per head, staged through shared memory.  It serves
// any head_dim up to 2048, any even rotary_dim and any element-aligned
// pointer.
#include "qk_common.cuh"

namespace edge {
namespace {

// ---------------------------------------------------------------- decode-width path

// One head per lane group, a one-shot grid: every unit of the grid is one
// head, so the unit's addresses are known before the dependent-launch wait.
// Every load of a head (data, weight, position) is issued right after it; the
// cache row follows the position, an L1/L2 hit for every head of a token but
// the first.  (Measured on GB300: reading the position before the wait as an
// address hint for the row, to save that second round trip, was 0.03 to
// 0.26 us slower per launch from T = 1 to 128, and so was a grid-stride loop
// over the heads.)
template <typename T, bool FP8, int LPH, int LAYOUT>
__global__ void __launch_bounds__(256) qk_vec_kernel(QKP p) {
    constexpr int N = vec_elems<T>();
    constexpr int HPW = 32 / LPH;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPH - 1);
    // < 2^31 + 8 HPW: units are at most 2^31 - 1 (validated)
    const uint32_t u = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * HPW + lane / LPH;
    const bool active = u < p.units;
    const Unit un = locate(p, active ? u : 0);

    if (threadIdx.x == 0) {
        const uint32_t per_cta = (blockDim.x >> 5) * HPW;
        prefetch_heads(p, blockIdx.x * per_cta, (blockIdx.x + 1) * per_cta, true);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int lane_role = p.rot > 0 ? rotary_role<T, LAYOUT>(p, sub) : 0;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    int64_t pos = -1;
    if (active) {
        raw = __ldcs(reinterpret_cast<const uint4*>(un.src) + sub);
        if (p.rot > 0) pos = __ldg(p.pos + un.t);
    }
    float w[N];
    weights_plus_delta<T>(p, un.w, sub, w);
    const bool rot = active && pos >= 0 && pos < p.cache_len;
    const int role = rot ? lane_role : 0;
    CacheRegs<T, LAYOUT> cr;
    if (role != 0) load_cache<T, LAYOUT>(p, pos, sub, role, cr);
    qk_core<T, FP8, LPH, LAYOUT>(p, un.dst, active, lane, sub, raw, w, role, cr);
}

// Two vectors per lane, for mid widths: lane sub of an LPH-lane group holds
// the head's vectors sub and sub + LPH, so a warp carries 32 / LPH heads of
// 2 LPH vectors and every per-head step (address decoding, the position and
// cache loads, the shuffle tree, the partner shuffle) serves twice the data
// of the one-vector form.  Rotate-half heads whose rotary channels all lie in
// the first LPH vectors, in the rounded mode: the second vector of a lane
// never rotates (qk_core2).
template <typename T, bool FP8, int LPH>
__global__ void __launch_bounds__(256) qk_vec2_kernel(QKP p) {
    constexpr int N = vec_elems<T>();
    constexpr int HPW = 32 / LPH;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (LPH - 1);
    // < 2^31 + 8 HPW: units are at most 2^31 - 1 (validated)
    const uint32_t u = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * HPW + lane / LPH;
    const bool active = u < p.units;
    const Unit un = locate(p, active ? u : 0);

    if (threadIdx.x == 0) {
        const uint32_t per_cta = (blockDim.x >> 5) * HPW;
        prefetch_heads(p, blockIdx.x * per_cta, (blockIdx.x + 1) * per_cta, true);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int lane_role = p.rot > 0 ? rotary_role<T, kRotateHalf>(p, sub) : 0;
    uint4 raw0 = make_uint4(0u, 0u, 0u, 0u), raw1 = raw0;
    int64_t pos = -1;
    if (active) {
        raw0 = __ldcs(reinterpret_cast<const uint4*>(un.src) + sub);
        raw1 = __ldcs(reinterpret_cast<const uint4*>(un.src) + sub + LPH);
        if (p.rot > 0) pos = __ldg(p.pos + un.t);
    }
    float w0[N], w1[N];
    weights_plus_delta<T>(p, un.w, sub, w0);
    weights_plus_delta<T>(p, un.w, sub + LPH, w1);
    const bool rot = active && pos >= 0 && pos < p.cache_len;
    const int role = rot ? lane_role : 0;
    CacheRegs<T, kRotateHalf> cr;
    if (role != 0) load_cache<T, kRotateHalf>(p, pos, sub, role, cr);

    qk_core2<T, FP8, LPH>(p, un.dst, active, lane, sub, raw0, raw1, w0, w1, role, cr);
}

// ---------------------------------------------------------------- generic path

template <typename T, bool FP8>
__global__ void __launch_bounds__(128) qk_generic_kernel(QKP p, int layout) {
    extern __shared__ float smem[];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    float* hm = smem + wib * p.D;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;

    pdl_wait();
    pdl_launch_dependents();

    for (uint32_t u = warp; u < p.units; u += nwarps) {
        const Unit un = locate(p, u);
        generic_head<T, FP8>(p, un.src, un.dst, un.w, un.t, (p.mode & kModeNorm) != 0, hm, lane,
                             layout);
    }
}

// ---------------------------------------------------------------- launch

using QKFn = void (*)(QKP);

template <typename T, bool FP8, int LPH>
QKFn vec_fn(int layout) {
    return layout == kInterleaved ? qk_vec_kernel<T, FP8, LPH, kInterleaved>
                                  : qk_vec_kernel<T, FP8, LPH, kRotateHalf>;
}

template <typename T, bool FP8>
cudaError_t launch_typed(const QKArgs& a, QKP& p, cudaStream_t s) {
    constexpr int N = vec_elems<T>();
    const int D = a.head_dim;
    const int nvec = (D * (int)sizeof(T)) % 16 == 0 ? D * (int)sizeof(T) / 16 : 0;
    auto aligned = [](const void* ptr, uintptr_t n) {
        return ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) % n) == 0;
    };
    bool vec = nvec > 0 && nvec <= 32 && (nvec & (nvec - 1)) == 0;
    vec = vec && aligned(a.q, 16) && aligned(a.k, 16) && aligned(a.wq, 16) && aligned(a.wk, 16);
    vec = vec && aligned(a.q_out, FP8 ? N : 16) && aligned(a.k_out, FP8 ? N : 16);
    if (a.rotary_dim > 0) {
        if (a.layout == kInterleaved) {
            vec = vec && a.rotary_dim % N == 0 && aligned(a.cos, 8 * (N / 4)) &&
                  aligned(a.sin, 8 * (N / 4));
        } else {
            vec = vec && (a.rotary_dim / 2) % N == 0 && aligned(a.cos, 16) && aligned(a.sin, 16);
        }
    }
    const int sms = sm_count();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;

    if (vec) {
        const int lph = nvec;
        const int hpw = 32 / lph;
        QKFn vfn = nullptr;
        switch (lph) {
            case 1: vfn = vec_fn<T, FP8, 1>(a.layout); break;
            case 2: vfn = vec_fn<T, FP8, 2>(a.layout); break;
            case 4: vfn = vec_fn<T, FP8, 4>(a.layout); break;
            case 8: vfn = vec_fn<T, FP8, 8>(a.layout); break;
            case 16: vfn = vec_fn<T, FP8, 16>(a.layout); break;
            default: vfn = vec_fn<T, FP8, 32>(a.layout); break;
        }
        // decode-width path: one head per lane group, a one-shot grid (on
        // GB300 many short CTAs that each issue one round of loads keep more
        // requests in flight than fewer, fatter warps: several heads in
        // flight per group or a resident looping grid measured slower)
        const int threads = 256;
        const int64_t per_block = (int64_t)(threads / 32) * hpw;
        int64_t blocks = ((int64_t)p.units + per_block - 1) / per_block;
        // Measured on GB300 for every geometry: the one-shot grid wins up to a
        // measured number of waves of resident CTAs (one for 16-bit heads,
        // two for fp32); past that, four threads per head (about 4x fewer
        // instructions per head) win.
        const int64_t hbytes = (int64_t)D * (int64_t)sizeof(T);
        const double wave = (double)resident_ctas((const void*)vfn, threads) * sms *
                            quad_min_waves((int)sizeof(T), a.layout, a.rotary_dim, hbytes);
        // 16-bit heads of 512 bytes whose rotary channels lie in the first
        // half (the text profiles), in the rounded mode, have a third form:
        // two vectors per lane.  Measured on GB300 against both others over
        // T = 1 to 1024 for the (16,2) and (24,4) text profiles and RoPE
        // alone, in units of the one-vector grid's waves w: the one-vector
        // form wins for w <= 0.25 (by up to 4%) and at 0.8 < w <= 1, where it
        // fills one balanced wave (by 6-8%); two vectors win elsewhere up to
        // w = 1.6 (by 8-18%, over four threads per head from w = 1); four
        // threads per head beyond.
        const bool two = sizeof(T) == 2 && hbytes == 512 && a.layout == kRotateHalf &&
                         a.rotary_dim <= D / 2 && (a.mode & kModeUnrounded) == 0;
        const double w = (double)blocks / (double)(resident_ctas((const void*)vfn, threads) * sms);
        const bool take_quad = two ? w > 1.6 : (double)blocks > wave;
        if (take_quad && quad_suits(a.layout, a.rotary_dim, hbytes)) {
            bool handled = false;
            cudaError_t e = launch_qk_quad<T, FP8>(a, p, cfg, &handled);
            if (handled || e != cudaSuccess) return e;
        }
        if constexpr (sizeof(T) == 2) {
            if (two && w > 0.25 && !(w > 0.8 && w <= 1.0)) {
                // 16 lanes per head, two heads per warp, 16 heads per CTA
                const int64_t per2 = (int64_t)(threads / 32) * 2;
                cfg.gridDim = dim3((unsigned)(((int64_t)p.units + per2 - 1) / per2));
                cfg.blockDim = dim3(threads);
                cfg.dynamicSmemBytes = 0;
                return cudaLaunchKernelEx(&cfg, qk_vec2_kernel<T, FP8, 16>, p);
            }
        }
        // one-shot: units <= 2^31 - 1 (validated), so blocks < 2^28
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = 0;
        return cudaLaunchKernelEx(&cfg, vfn, p);
    }
    const int threads = 128;
    const int64_t warps_per_block = threads / 32;
    int64_t blocks = ((int64_t)p.units + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    const size_t smem = (size_t)warps_per_block * D * sizeof(float);
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(qk_generic_kernel<T, FP8>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, qk_generic_kernel<T, FP8>, p, a.layout);
}

}  // namespace

cudaError_t launch_qk(const QKArgs& args, cudaStream_t s) {
    // With no cache rows or no positions no token can rotate: run the
    // prologue with rotary width 0 so the kernels touch neither pointer.
    QKArgs a = args;
    if (a.cache_len <= 0 || a.pos == nullptr || a.cos == nullptr || a.sin == nullptr) {
        a.rotary_dim = 0;
    }
    QKP p;
    p.q = static_cast<const char*>(a.q);
    p.k = static_cast<const char*>(a.k);
    p.qo = static_cast<char*>(a.q_out);
    p.ko = static_cast<char*>(a.k_out);
    p.wq = static_cast<const char*>(a.wq);
    p.wk = static_cast<const char*>(a.wk);
    p.pos = a.pos;
    p.cs = a.cos;
    p.sn = a.sin;
    p.cache_len = a.rotary_dim > 0 ? a.cache_len : 0;
    p.tokens = a.tokens;
    p.units = (uint32_t)(a.tokens * (a.q_heads + a.k_heads));
    p.heads = make_fastdiv((uint32_t)(a.q_heads + a.k_heads));
    p.qdiv = make_fastdiv((uint32_t)a.q_heads);
    p.kdiv = make_fastdiv((uint32_t)(a.k_heads > 0 ? a.k_heads : 1));
    p.qrows = (uint32_t)(a.tokens * a.q_heads);
    p.q_heads = a.q_heads;
    p.k_heads = a.k_heads;
    p.D = a.head_dim;
    p.rot = a.rotary_dim;
    p.half = a.rotary_dim / 2;
    p.in_bytes = a.dt == kF32 ? 4 : 2;
    p.out_bytes = a.out_dt == kFP8 ? 1 : p.in_bytes;
    p.eps = a.eps;
    p.delta = (float)a.weight_offset;
    p.inv = a.inv_scale;
    p.invD = 1.0f / (float)a.head_dim;
    p.mode = a.mode;
    const bool fp8 = a.out_dt == kFP8;
    switch (a.dt) {
        case kF32:
            return fp8 ? launch_typed<float, true>(a, p, s) : launch_typed<float, false>(a, p, s);
        case kF16:
            return fp8 ? launch_typed<__half, true>(a, p, s) : launch_typed<__half, false>(a, p, s);
        default:
            return fp8 ? launch_typed<__nv_bfloat16, true>(a, p, s)
                       : launch_typed<__nv_bfloat16, false>(a, p, s);
    }
}

}  // namespace edge
