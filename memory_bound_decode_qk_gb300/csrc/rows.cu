// rows.cu -- RMSNorm and fused residual-add RMSNorm over rows (sm_103a).
//
// What they compute ("thox-edge-ops v2", section 3 R1 and section 5.1;
// FlashRT rms_norm_fp8_static, residual_add_rms_norm_fp8_static and the
// no-weight RMSNorm):
//   residual <- round_dt(fp32(x) + fp32(residual))    (fused form only)
//   out      =  s * r * (w + delta),  r = 1 / sqrt(mean(s^2) + eps)
// s is x for the plain form and the rounded sum for the fused form.  The
// output is rounded once to the activation dtype, or takes the static-scale
// FP8 epilogue.
//
// GB300 design.  Both ops move about 3 or 4 bytes of HBM traffic for every 2
// flops.  A row is held in registers from its load to its store, so it makes
// one HBM pass.  A CTA is a (32 W) x R block: threadIdx.y picks one of its R
// rows and the W warps along x share that row, each thread holding up to V
// 16-byte vectors.  Every load of a thread is issued before any arithmetic,
// so it keeps V (fused form: 2V) loads in flight.  The grid is one-shot (one
// CTA per R rows, no grid-stride loop), so between the dependent-launch wait
// and the loads there is no index arithmetic beyond a multiply-add.  (Measured
// on GB300: the earlier form, which divided the thread index by a run-time
// row width and looped over rows, took 1.79 us per decode-width launch at
// T = 64 and 3.1 us at T = 512 against 1.57 and 2.2 us for this one.)  The
// sum of squares is reduced with warp shuffles, then through shared memory
// with one barrier.  The elementwise steps run on fp32 pairs (packed two-lane
// instructions).  W and V come from the row length and the row
// count: few rows spread over more warps, many rows favour more bytes in
// flight per thread.  Rows whose length or alignment does not allow 16-byte
// vectors take a scalar two-pass kernel: one CTA per row, and the second pass
// re-reads the row from L1/L2.
#include "edge_common.cuh"
#include "launch.h"

namespace edge {
namespace {

struct RowsP {
    const char* x;
    char* res;
    const char* w;          // RMSNorm weight, or LayerNorm gamma
    const char* beta;       // LayerNorm beta (nullable)
    char* out;
    int64_t rows;
    int hidden;
    int nvec;      // 16-byte vectors per row
    float eps, delta, inv, invH;  // invH = 1 / hidden (fp32)
};

// Sum of v over the W = blockDim.x / 32 warps that share this thread's row
// (threadIdx.y): a shuffle tree per warp, then shared memory and one barrier.
// Every thread of the CTA calls it.  The barrier is taken even when W = 1 (a
// row per warp): the unconditional form measured 0.06 us faster per launch
// on GB300 at decode widths than one branching around it.  A kernel that
// reduces twice passes two buffers, so that no slot is rewritten before every
// reader has passed the barrier that follows its first write.
__device__ __forceinline__ float row_sum(float v, float* buf) {
    v = group_sum<32>(v);
    const int W = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) buf[(threadIdx.y * blockDim.x + threadIdx.x) >> 5] = v;
    __syncthreads();
    v = 0.0f;
    for (int k = 0; k < W; ++k) v = __fadd_rn(v, buf[threadIdx.y * W + k]);
    return v;
}

template <typename T, bool FP8, bool ADD, int V>
__global__ void __launch_bounds__(512) rows_vec_kernel(RowsP p) {
    constexpr int N = vec_elems<T>();
    __shared__ float red[16];
    const int tid = threadIdx.x;
    const int tpr = blockDim.x;
    const int64_t row0 = (int64_t)blockIdx.x * blockDim.y;
    const int64_t row = row0 + threadIdx.y;
    const bool active = row < p.rows;
    const int64_t in_row = (int64_t)p.nvec * 16;
    const int64_t out_row = FP8 ? (int64_t)p.hidden : in_row;

    if (tid == 0 && threadIdx.y == 0) {
        // this CTA's rows into L2 while the preceding grid drains
        const int64_t r1 = row0 + blockDim.y < p.rows ? row0 + blockDim.y : p.rows;
        prefetch_l2(p.x, row0 * in_row, r1 * in_row);
        if (ADD) prefetch_l2(p.res, row0 * in_row, r1 * in_row);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int64_t rsafe = active ? row : row0;
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + rsafe * in_row);
    uint4* rr = ADD ? reinterpret_cast<uint4*>(p.res + rsafe * in_row) : nullptr;

    // every load of the row (x, residual and the weight) is issued before
    // any arithmetic: one memory round trip per row
    const uint4* wv = reinterpret_cast<const uint4*>(p.w);
    uint4 xv[V], rv[V], wr[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        const bool ok = active && idx < p.nvec;
        xv[i] = ok ? __ldcs(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
        if constexpr (ADD) rv[i] = ok ? __ldcs(rr + idx) : make_uint4(0u, 0u, 0u, 0u);
        wr[i] = (ok && wv != nullptr) ? __ldg(wv + idx) : make_uint4(0u, 0u, 0u, 0u);
    }

    // running sums: the two lanes of a pair, and beyond 32 terms per thread
    // two pairs alternating by vector (at most 2N sequential terms each, for
    // the error bound of the tolerance)
    constexpr int P = N / 2;
    constexpr bool kSplit = V * N > 32;
    float2 ssp[2] = {splat2(0.0f), splat2(0.0f)};
#pragma unroll
    for (int i = 0; i < V; ++i) {
        float2 a[P];
        unpack_pairs<T, N>(xv[i], a);
        if constexpr (ADD) {
            // eager semantics: widen, add in fp32, round once to the dtype
            float2 b[P];
            unpack_pairs<T, N>(rv[i], b);
#pragma unroll
            for (int j = 0; j < P; ++j) a[j] = __fadd2_rn(a[j], b[j]);
            xv[i] = pack_pairs<T, N>(a);
            unpack_pairs<T, N>(xv[i], a);  // the rounded sums
            const int idx = tid + i * tpr;
            if (active && idx < p.nvec) rr[idx] = xv[i];
        }
#pragma unroll
        for (int j = 0; j < P; ++j) {
            ssp[kSplit ? (i & 1) : 0] = __ffma2_rn(a[j], a[j], ssp[kSplit ? (i & 1) : 0]);
        }
    }
    const float2 s2 = kSplit ? __fadd2_rn(ssp[0], ssp[1]) : ssp[0];
    const float ss = row_sum(__fadd_rn(s2.x, s2.y), red);
    const float2 r2 = splat2(inv_rms(ss, p.invH, p.eps));
    const float2 delta2 = splat2(p.delta);

    char* orow = p.out + rsafe * out_row;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        if (!(active && idx < p.nvec)) continue;
        float2 sv[P], y[P];
        unpack_pairs<T, N>(xv[i], sv);
        if (wv != nullptr) {
            float2 w[P];
            unpack_pairs<T, N>(wr[i], w);
#pragma unroll
            for (int j = 0; j < P; ++j) y[j] = __fmul2_rn(__fmul2_rn(sv[j], r2), __fadd2_rn(w[j], delta2));
        } else {
#pragma unroll
            for (int j = 0; j < P; ++j) y[j] = __fmul2_rn(sv[j], r2);
        }
        if constexpr (FP8) {
            auto q8 = quantize_pairs<N>(y, p.inv);
            reinterpret_cast<decltype(q8)*>(orow)[idx] = q8;
        } else {
            reinterpret_cast<uint4*>(orow)[idx] = pack_pairs<T, N>(y);
        }
    }
}

// The row's sum of squares is accumulated in fp64: a thread here sums
// hidden / 256 terms (65,536 at the largest row), too many for an fp32
// running sum to stay within a few fp32 ulps.
template <typename T, bool FP8, bool ADD>
__global__ void __launch_bounds__(256) rows_generic_kernel(RowsP p) {
    __shared__ double red[8];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;

    pdl_wait();
    pdl_launch_dependents();

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const T* x = reinterpret_cast<const T*>(p.x) + row * p.hidden;
        T* res = ADD ? reinterpret_cast<T*>(p.res) + row * p.hidden : nullptr;
        double ss = 0.0;
        for (int i = threadIdx.x; i < p.hidden; i += blockDim.x) {
            float a = to_f(x[i]);
            if constexpr (ADD) {
                a = round_to<T>(__fadd_rn(a, to_f(res[i])));
                res[i] = from_f<T>(a);
            }
            ss = __fma_rn((double)a, (double)a, ss);
        }
        ss = group_sum<32>(ss);
        if (lane == 0) red[wib] = ss;
        __syncthreads();
        ss = 0.0;
        for (int k = 0; k < nw; ++k) ss = __dadd_rn(ss, red[k]);
        __syncthreads();
        const float r = inv_rms((float)ss, p.invH, p.eps);
        const T* w = reinterpret_cast<const T*>(p.w);
        for (int i = threadIdx.x; i < p.hidden; i += blockDim.x) {
            const float s = ADD ? to_f(res[i]) : to_f(x[i]);
            const float y = w ? __fmul_rn(__fmul_rn(s, r), __fadd_rn(to_f(w[i]), p.delta))
                              : __fmul_rn(s, r);
            if constexpr (FP8) {
                reinterpret_cast<uint8_t*>(p.out)[row * p.hidden + i] = quantize1(y, p.inv);
            } else {
                reinterpret_cast<T*>(p.out)[row * p.hidden + i] = from_f<T>(y);
            }
        }
    }
}

// One-read LayerNorm (FlashRT siglip_layernorm_1read): the row stays in
// registers for the mean, the variance of the centred values and the
// output, so x is read from HBM once.  y = (x - mu) r gamma + beta.  gamma
// and beta are loaded after the two reductions, so they hold no registers
// across them.
template <typename T, bool FP8, int V>
__global__ void __launch_bounds__(512) ln_vec_kernel(RowsP p) {
    constexpr int N = vec_elems<T>();
    __shared__ float red_mu[16], red_var[16];
    const int tid = threadIdx.x;
    const int tpr = blockDim.x;
    const int64_t row0 = (int64_t)blockIdx.x * blockDim.y;
    const int64_t row = row0 + threadIdx.y;
    const bool active = row < p.rows;
    const int64_t in_row = (int64_t)p.nvec * 16;
    const int64_t out_row = FP8 ? (int64_t)p.hidden : in_row;
    const uint4* gv = reinterpret_cast<const uint4*>(p.w);
    const uint4* bv = reinterpret_cast<const uint4*>(p.beta);

    if (tid == 0 && threadIdx.y == 0) {
        const int64_t r1 = row0 + blockDim.y < p.rows ? row0 + blockDim.y : p.rows;
        prefetch_l2(p.x, row0 * in_row, r1 * in_row);
    }
    pdl_wait();
    pdl_launch_dependents();

    const int64_t rsafe = active ? row : row0;
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + rsafe * in_row);
    uint4 xv[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        const bool ok = active && idx < p.nvec;
        xv[i] = ok ? __ldcs(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
    // running sums: the two lanes of a pair, and beyond 32 terms per thread
    // two pairs alternating by vector
    constexpr int P = N / 2;
    constexpr bool kSplit = V * N > 32;
    float2 sp[2] = {splat2(0.0f), splat2(0.0f)};
#pragma unroll
    for (int i = 0; i < V; ++i) {
        float2 a[P];
        unpack_pairs<T, N>(xv[i], a);
#pragma unroll
        for (int j = 0; j < P; ++j) {
            sp[kSplit ? (i & 1) : 0] = __fadd2_rn(sp[kSplit ? (i & 1) : 0], a[j]);
        }
    }
    const float2 s2 = kSplit ? __fadd2_rn(sp[0], sp[1]) : sp[0];
    const float mu = __fmul_rn(row_sum(__fadd_rn(s2.x, s2.y), red_mu), p.invH);
    const float2 nmu = splat2(-mu);  // x + (-mu) is x - mu exactly
    float2 sqp[2] = {splat2(0.0f), splat2(0.0f)};
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        if (!(active && idx < p.nvec)) continue;  // padding lanes add nothing
        float2 a[P];
        unpack_pairs<T, N>(xv[i], a);
#pragma unroll
        for (int j = 0; j < P; ++j) {
            const float2 d = __fadd2_rn(a[j], nmu);
            sqp[kSplit ? (i & 1) : 0] = __ffma2_rn(d, d, sqp[kSplit ? (i & 1) : 0]);
        }
    }
    const float2 q2 = kSplit ? __fadd2_rn(sqp[0], sqp[1]) : sqp[0];
    const float2 r2 = splat2(inv_rms(row_sum(__fadd_rn(q2.x, q2.y), red_var), p.invH, p.eps));
    // gamma and beta (L1/L2-resident), all issued before the output loop
    uint4 gr[V], br[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        const bool ok = active && idx < p.nvec;
        gr[i] = (ok && gv != nullptr) ? __ldg(gv + idx) : make_uint4(0u, 0u, 0u, 0u);
        br[i] = (ok && bv != nullptr) ? __ldg(bv + idx) : make_uint4(0u, 0u, 0u, 0u);
    }
    char* orow = p.out + rsafe * out_row;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const int idx = tid + i * tpr;
        if (!(active && idx < p.nvec)) continue;
        float2 a[P], gg[P], bb[P], y[P];
        unpack_pairs<T, N>(xv[i], a);
        if (gv != nullptr) unpack_pairs<T, N>(gr[i], gg);
        if (bv != nullptr) unpack_pairs<T, N>(br[i], bb);
#pragma unroll
        for (int j = 0; j < P; ++j) {
            // (x - mu) (r gamma) + beta: one product and one fma per pair
            const float2 d = __fadd2_rn(a[j], nmu);
            const float2 rg = gv != nullptr ? __fmul2_rn(r2, gg[j]) : r2;
            y[j] = bv != nullptr ? __ffma2_rn(d, rg, bb[j]) : __fmul2_rn(d, rg);
        }
        if constexpr (FP8) {
            auto q8 = quantize_pairs<N>(y, p.inv);
            reinterpret_cast<decltype(q8)*>(orow)[idx] = q8;
        } else {
            reinterpret_cast<uint4*>(orow)[idx] = pack_pairs<T, N>(y);
        }
    }
}

// LayerNorm with one warp per row, for rows of at most 256 16-byte vectors
// (bf16/fp16 width <= 2048, fp32 <= 1024).  Both reductions are warp
// shuffles, with no block barrier per row.  gamma and beta are staged once per
// CTA in shared memory, so the output loop reads them without global latency
// and they hold no registers across the reductions.  A lane holds
// V = ceil(vectors / 32) <= 8 vectors, so few registers are live and many
// rows are in flight per SM.  The elementwise steps run on fp32 pairs.
// Register budget, in CTAs of the 128 threads launched per SM: 8 (64
// registers) up to 4 vectors per lane, 7 (72) at 5 and 4 (128) beyond, the
// counts at which ptxas for sm_103a keeps the variants spill-free.  At 5
// vectors (width 1152) 7 CTAs per SM hold the 1024 CTAs of T = 4096 in one
// wave (1064 slots); a variant held to 6 (78 registers) measured 1.27x
// slower there.
template <int V>
constexpr int ln_warp_min_blocks() {
    return V <= 4 ? 8 : V == 5 ? 7 : 4;
}

template <typename T, bool FP8, int V>
__global__ void __launch_bounds__(128, ln_warp_min_blocks<V>()) ln_warp_kernel(RowsP p) {
    constexpr int N = vec_elems<T>();
    constexpr int P = N / 2;
    extern __shared__ __align__(16) uint4 ln_gb[];  // gamma [nvec], then beta [nvec]
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    const int64_t in_row = (int64_t)p.hidden * (int64_t)sizeof(T);
    const int64_t out_row = FP8 ? (int64_t)p.hidden : in_row;
    const uint4* gv = reinterpret_cast<const uint4*>(p.w);
    const uint4* bv = reinterpret_cast<const uint4*>(p.beta);

    if (threadIdx.x == 0) {
        const int64_t r0 = (int64_t)blockIdx.x * wpb;
        const int64_t r1 = r0 + wpb < p.rows ? r0 + wpb : p.rows;
        prefetch_l2(p.x, r0 * in_row, r1 * in_row);
        if (blockIdx.x == 0) {
            prefetch_l2(p.w, 0, in_row);
            prefetch_l2(p.beta, 0, in_row);
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    uint4* gs = ln_gb;
    uint4* bs = ln_gb + p.nvec;
    bool staged = false;
    // passes over wpb rows at a time (the same for the whole CTA, so the one
    // barrier below is reached by every warp)
    for (int64_t base = (int64_t)blockIdx.x * wpb; base < p.rows; base += (int64_t)gridDim.x * wpb) {
        const int64_t row = base + (threadIdx.x >> 5);
        const bool active = row < p.rows;
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (active ? row : base) * in_row);
        uint4 xv[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int idx = lane + 32 * i;
            xv[i] = (active && idx < p.nvec) ? __ldcs(xr + idx) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (!staged) {
            // gamma and beta into shared memory while the first rows are in
            // flight
            for (int i = threadIdx.x; i < p.nvec; i += blockDim.x) {
                if (gv != nullptr) gs[i] = __ldg(gv + i);
                if (bv != nullptr) bs[i] = __ldg(bv + i);
            }
            __syncthreads();
            staged = true;
        }
        // running sums: the two lanes of a pair, and beyond 32 terms per
        // thread two pairs alternating by vector
        constexpr bool kSplit = V * N > 32;
        float2 sp[2] = {splat2(0.0f), splat2(0.0f)};
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float2 a[P];
            unpack_pairs<T, N>(xv[i], a);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                sp[kSplit ? (i & 1) : 0] = __fadd2_rn(sp[kSplit ? (i & 1) : 0], a[j]);
            }
        }
        const float2 s2 = kSplit ? __fadd2_rn(sp[0], sp[1]) : sp[0];
        const float mu = __fmul_rn(group_sum<32>(__fadd_rn(s2.x, s2.y)), p.invH);
        const float2 nmu = splat2(-mu);  // x + (-mu) is x - mu exactly
        float2 sqp[2] = {splat2(0.0f), splat2(0.0f)};
#pragma unroll
        for (int i = 0; i < V; ++i) {
            if (lane + 32 * i >= p.nvec) continue;  // padding lanes add nothing
            float2 a[P];
            unpack_pairs<T, N>(xv[i], a);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                const float2 d = __fadd2_rn(a[j], nmu);
                sqp[kSplit ? (i & 1) : 0] = __ffma2_rn(d, d, sqp[kSplit ? (i & 1) : 0]);
            }
        }
        const float2 q2 = kSplit ? __fadd2_rn(sqp[0], sqp[1]) : sqp[0];
        const float r = inv_rms(group_sum<32>(__fadd_rn(q2.x, q2.y)), p.invH, p.eps);
        if (!active) continue;
        const float2 r2 = splat2(r);
        char* orow = p.out + row * out_row;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int idx = lane + 32 * i;
            if (idx >= p.nvec) continue;
            float2 a[P], gg[P], bb[P], y[P];
            unpack_pairs<T, N>(xv[i], a);
            if (gv != nullptr) unpack_pairs<T, N>(gs[idx], gg);
            if (bv != nullptr) unpack_pairs<T, N>(bs[idx], bb);
#pragma unroll
            for (int j = 0; j < P; ++j) {
                // (x - mu) (r gamma) + beta: one product and one fma per pair
                const float2 d = __fadd2_rn(a[j], nmu);
                const float2 rg = gv != nullptr ? __fmul2_rn(r2, gg[j]) : r2;
                y[j] = bv != nullptr ? __ffma2_rn(d, rg, bb[j]) : __fmul2_rn(d, rg);
            }
            if constexpr (FP8) {
                auto q8 = quantize_pairs<N>(y, p.inv);
                reinterpret_cast<decltype(q8)*>(orow)[idx] = q8;
            } else {
                reinterpret_cast<uint4*>(orow)[idx] = pack_pairs<T, N>(y);
            }
        }
    }
}

// Any size or alignment: one CTA per row, three passes (the second and third
// hit L1/L2).  Both reductions accumulate in fp64, as in the scalar RMSNorm
// kernel.
template <typename T, bool FP8>
__global__ void __launch_bounds__(256) ln_generic_kernel(RowsP p) {
    __shared__ double red[8];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    auto block_sum = [&](double v) {
        v = group_sum<32>(v);
        if (lane == 0) red[wib] = v;
        __syncthreads();
        v = 0.0;
        for (int k = 0; k < nw; ++k) v = __dadd_rn(v, red[k]);
        __syncthreads();
        return v;
    };

    pdl_wait();
    pdl_launch_dependents();

    const T* gm = reinterpret_cast<const T*>(p.w);
    const T* bt = reinterpret_cast<const T*>(p.beta);
    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        const T* x = reinterpret_cast<const T*>(p.x) + row * p.hidden;
        double sum = 0.0;
        for (int i = threadIdx.x; i < p.hidden; i += blockDim.x) {
            sum = __dadd_rn(sum, (double)to_f(x[i]));
        }
        const float mu = (float)(block_sum(sum) / (double)p.hidden);
        double sq = 0.0;
        for (int i = threadIdx.x; i < p.hidden; i += blockDim.x) {
            const float d = __fsub_rn(to_f(x[i]), mu);
            sq = __fma_rn((double)d, (double)d, sq);
        }
        const float r = inv_rms((float)block_sum(sq), p.invH, p.eps);
        for (int i = threadIdx.x; i < p.hidden; i += blockDim.x) {
            const float d = __fsub_rn(to_f(x[i]), mu);
            const float rg = gm != nullptr ? __fmul_rn(r, to_f(gm[i])) : r;
            const float v = bt != nullptr ? __fmaf_rn(d, rg, to_f(bt[i])) : __fmul_rn(d, rg);
            if constexpr (FP8) {
                reinterpret_cast<uint8_t*>(p.out)[row * p.hidden + i] = quantize1(v, p.inv);
            } else {
                reinterpret_cast<T*>(p.out)[row * p.hidden + i] = from_f<T>(v);
            }
        }
    }
}

// Launch shape of the vector kernels.
struct VecShape {
    int nvec;  // 16-byte vectors per row
    int W;     // warps per row (blockDim.x = 32 W)
    int R;     // rows per CTA (blockDim.y)
    int V;     // vectors per thread (template argument)
};

// The vector shape of a call, or false when the row needs the generic kernel
// (length or alignment not a multiple of 16 bytes, more than 16 x 32 x 8
// vectors per row, or more CTAs than a one-shot grid holds).
template <typename T, bool FP8>
bool vec_shape(const RowsArgs& a, int sms, VecShape& v) {
    constexpr int N = vec_elems<T>();
    auto aligned = [](const void* ptr, uintptr_t n) {
        return ptr == nullptr || (reinterpret_cast<uintptr_t>(ptr) % n) == 0;
    };
    const bool vec_ok = (a.hidden * (int64_t)sizeof(T)) % 16 == 0 && aligned(a.x, 16) &&
                        aligned(a.residual, 16) && aligned(a.w, 16) && aligned(a.beta, 16) &&
                        aligned(a.out, FP8 ? N : 16);
    const int64_t nvec = a.hidden / N;
    if (!vec_ok || nvec > 16 * 32 * 8) return false;
    // target vectors per thread (measured on GB300: 1 for few rows, 2 for
    // many; more per thread lowers occupancy and loses bandwidth)
    int vt = a.rows >= 2 * sms ? 2 : 1;
    // plain RMSNorm with the FP8 epilogue (one input stream, one-byte
    // outputs): four vectors per thread once there are many rows.  Measured
    // on GB300 at width 2048: 5% faster at T = 1024, 16% at T = 4096 than
    // two; with a bf16 output two stay faster (by 6% at T = 4096)
    if (FP8 && !a.residual && !a.layernorm && a.rows >= 4 * sms) vt = 4;
    int W = (int)((nvec + 32 * vt - 1) / (32 * vt));
    if (W > 16) W = 16;
    const int64_t per = (nvec + 32 * W - 1) / (32 * W);
    v.V = per <= 1 ? 1 : per <= 2 ? 2 : per <= 4 ? 4 : 8;
    v.W = W;
    v.R = 256 / (32 * W) > 1 ? 256 / (32 * W) : 1;
    v.nvec = (int)nvec;
    return (a.rows + v.R - 1) / v.R <= (int64_t)INT32_MAX;
}

template <typename T, bool FP8, bool ADD>
cudaError_t launch_typed(const RowsArgs& a, RowsP& p, cudaStream_t s) {
    const int sms = sm_count();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;

    VecShape v;
    const bool vec = vec_shape<T, FP8>(a, sms, v);
    if (vec) p.nvec = v.nvec;
    // LayerNorm: one warp per row once there are many rows.  Measured
    // crossover on GB300: between T = 768 and 1024 at width 1152 (5 vectors
    // per lane; the CTA-per-row form 4.5% faster at 768, 15% slower at 1024),
    // T = 1536 at width 2048 (8 vectors per lane, fewer CTAs per SM)
    const int64_t lanes_vecs = ((int64_t)a.hidden / vec_elems<T>() + 31) / 32;
    const bool ln_warp = a.rows >= (lanes_vecs <= 5 ? 6 : 10) * (int64_t)sms;
    if (vec && a.layernorm && v.nvec <= 256 && ln_warp) {
        // 4 rows per CTA: finer CTAs balance the last wave (measured on
        // GB300: 1.35x faster than 8 rows per CTA at T = 4096, width 1152)
        const int threads = 128;
        const int64_t rpb = threads / 32;
        int64_t blocks = (a.rows + rpb - 1) / rpb;
        const int64_t cap = (int64_t)sms * 64;
        if (blocks > cap) blocks = cap;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = (size_t)2 * v.nvec * 16;
        switch ((v.nvec + 31) / 32) {
            case 1: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 1>, p);
            case 2: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 2>, p);
            case 3: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 3>, p);
            case 4: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 4>, p);
            case 5: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 5>, p);
            case 6: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 6>, p);
            case 7: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 7>, p);
            default: return cudaLaunchKernelEx(&cfg, ln_warp_kernel<T, FP8, 8>, p);
        }
    }
    if (vec) {
        // one-shot grid: one CTA per R rows
        cfg.gridDim = dim3((unsigned)((a.rows + v.R - 1) / v.R));
        cfg.blockDim = dim3(32 * v.W, v.R);
        if (a.layernorm) {
            switch (v.V) {
                case 1: return cudaLaunchKernelEx(&cfg, ln_vec_kernel<T, FP8, 1>, p);
                case 2: return cudaLaunchKernelEx(&cfg, ln_vec_kernel<T, FP8, 2>, p);
                case 4: return cudaLaunchKernelEx(&cfg, ln_vec_kernel<T, FP8, 4>, p);
                default: return cudaLaunchKernelEx(&cfg, ln_vec_kernel<T, FP8, 8>, p);
            }
        }
        switch (v.V) {
            case 1: return cudaLaunchKernelEx(&cfg, rows_vec_kernel<T, FP8, ADD, 1>, p);
            case 2: return cudaLaunchKernelEx(&cfg, rows_vec_kernel<T, FP8, ADD, 2>, p);
            case 4: return cudaLaunchKernelEx(&cfg, rows_vec_kernel<T, FP8, ADD, 4>, p);
            default: return cudaLaunchKernelEx(&cfg, rows_vec_kernel<T, FP8, ADD, 8>, p);
        }
    }
    int64_t blocks = a.rows;
    const int64_t cap = (int64_t)sms * 16;
    if (blocks > cap) blocks = cap;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    if (a.layernorm) return cudaLaunchKernelEx(&cfg, ln_generic_kernel<T, FP8>, p);
    return cudaLaunchKernelEx(&cfg, rows_generic_kernel<T, FP8, ADD>, p);
}

template <typename T>
cudaError_t launch_dt(const RowsArgs& a, RowsP& p, cudaStream_t s) {
    const bool fp8 = a.out_dt == kFP8;
    const bool add = a.residual != nullptr;
    if (fp8) return add ? launch_typed<T, true, true>(a, p, s) : launch_typed<T, true, false>(a, p, s);
    return add ? launch_typed<T, false, true>(a, p, s) : launch_typed<T, false, false>(a, p, s);
    // (LayerNorm takes the ADD = false instantiation of launch_typed)
}

}  // namespace

cudaError_t launch_rows(const RowsArgs& a, cudaStream_t s) {
    RowsP p;
    p.x = static_cast<const char*>(a.x);
    p.res = static_cast<char*>(a.residual);
    p.w = static_cast<const char*>(a.w);
    p.beta = static_cast<const char*>(a.beta);
    p.out = static_cast<char*>(a.out);
    p.rows = a.rows;
    p.hidden = (int)a.hidden;
    p.nvec = 0;
    p.eps = a.eps;
    p.delta = (float)a.weight_offset;
    p.inv = a.inv_scale;
    p.invH = 1.0f / (float)a.hidden;
    switch (a.dt) {
        case kF32: return launch_dt<float>(a, p, s);
        case kF16: return launch_dt<__half>(a, p, s);
        default: return launch_dt<__nv_bfloat16>(a, p, s);
    }
}

}  // namespace edge
