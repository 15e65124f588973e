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


// Threads-per-head path for many heads (qk_quad.cu).  *handled is false when
// the geometry is outside its instantiations; the caller then takes the
// lane-group path.
template <typename T, bool FP8>
cudaError_t launch_qk_quad(const QKArgs& a, const QKP& p, cudaLaunchConfig_t cfg, bool* handled);

// Whether the threads-per-head path is the better choice for this call.
bool qk_quad_preferred(const QKArgs& a, int sms);

}  // namespace edge
