// launch.h -- internal interface between the C ABI layer and the kernels.
// Arguments arrive here validated; each launcher picks a kernel and launch
// shape for its op and enqueues it on the caller's stream.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace edge {

enum Dt { kF32 = 0, kF16 = 1, kBF16 = 2, kFP8 = 3 };

struct QKArgs {
    const void* q;
    const void* k;
    void* q_out;
    void* k_out;
    const void* wq;          // nullable
    const void* wk;          // nullable
    const int64_t* pos;      // nullable when no rotation can happen
    const float* cos;
    const float* sin;
    int64_t tokens;
    int64_t cache_len;
    int q_heads, k_heads, head_dim, rotary_dim, layout;
    int dt, out_dt;
    float eps, inv_scale;
    int weight_offset;
    int mode;                // kModeNorm (1) | kModeUnrounded (2), qk_common.cuh
};

struct RowsArgs {
    const void* x;
    void* residual;          // nullptr: plain RMSNorm
    const void* w;           // nullable (LayerNorm: gamma)
    const void* beta;        // LayerNorm only, nullable
    int layernorm;           // 1: LayerNorm (no residual)
    void* out;
    int64_t rows;
    int64_t hidden;
    int dt, out_dt;
    float eps, inv_scale;
    int weight_offset;
};

struct GluArgs {
    const void* gate_up;
    void* out;
    int64_t rows;
    int64_t d;
    int dt, out_dt, act;
    float inv_scale;
};

// Launch-shape limits of the paths, checked by the ABI layer.
constexpr int64_t kMaxQKHeadDim = 2048;       // generic prologue path (smem per warp)
constexpr int64_t kMaxHidden = int64_t(1) << 24;  // row length, exact as fp32
constexpr int64_t kMaxUnits = (int64_t(1) << 31) - 1;

cudaError_t launch_qk(const QKArgs& a, cudaStream_t s);
cudaError_t launch_rows(const RowsArgs& a, cudaStream_t s);
cudaError_t launch_glu(const GluArgs& a, cudaStream_t s);

struct QKVArgs {
    const void* qkv;
    void* q_out;
    void* k_cache;
    void* v_cache;
    const void* wq;          // nullable
    const void* wk;          // nullable
    const int64_t* pos;
    const float* cos;
    const float* sin;
    const int64_t* slots;
    int64_t tokens, cache_len, num_slots;
    int q_heads, kv_heads, head_dim, rotary_dim, layout, dt;
    int normalize, weight_offset;
    float eps;
};
// *handled is false when the geometry or alignment has no vector path.
cudaError_t launch_qkv_cache(const QKVArgs& a, cudaStream_t s, bool* handled);

struct QuantArgs {
    const void* x;
    void* out;
    int64_t n;
    int dt;
    float inv_scale;
};
cudaError_t launch_quant(const QuantArgs& a, cudaStream_t s);

// The yardstick copy (copy.cu): bytes from src to dst, validated.
cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// CTAs of kernel `fn` resident per SM at `threads` threads and no dynamic
// shared memory (the occupancy calculator, cached per kernel and device).
int resident_ctas(const void* fn, int threads);

// Programmatic dependent launch for all ops (on unless EDGE_OPS_PDL=0 in the
// environment, read once per process).  Every kernel executes
// griddepcontrol.wait before its first global load whose value it uses, so
// it is always safe as a dependent; it triggers its own dependents at its
// start.
bool pdl_enabled();

}  // namespace edge
