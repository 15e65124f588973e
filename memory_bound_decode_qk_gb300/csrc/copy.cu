// copy.cu -- a plain device copy in the launch form of the seam kernels (sm_103a).
//
// Not one of the operators: the yardstick the measurements set them against.
// A seam op at decode or mid widths moves a few MB, which HBM alone would move
// in well under a microsecond, so launch, ramp and drain decide its time.  This
// kernel moves the same number of bytes with the same launch form as the ops:
//   - a one-shot grid of 256-thread CTAs over 16-byte vectors, each thread
//     loading V vectors before its first store;
//   - one thread per CTA prefetching the CTA's source span into L2 before the
//     dependent-launch wait;
//   - programmatic dependent launch (wait, then trigger).
// Its time at an op's byte count is the time of a kernel that does nothing but
// move those bytes, which is what "the op reaches x% of the achievable" means.
// The bytes past the last whole vector, and misaligned buffers, take a byte
// loop.
#include "edge_common.cuh"
#include "launch.h"

namespace edge {
namespace {

template <int V>
__global__ void __launch_bounds__(256) copy_kernel(const char* src, char* dst, int64_t nvec,
                                                   int64_t bytes) {
    const int64_t span = (int64_t)blockDim.x * V;
    const int64_t v0 = (int64_t)blockIdx.x * span;
    if (threadIdx.x == 0 && v0 < nvec) {
        const int64_t v1 = v0 + span < nvec ? v0 + span : nvec;
        prefetch_l2(src, 16 * v0, 16 * v1);
    }
    pdl_wait();
    pdl_launch_dependents();
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    const int64_t stride = (int64_t)gridDim.x * span;
    for (int64_t b = v0 + threadIdx.x; b < nvec; b += stride) {
        uint4 v[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = b + (int64_t)k * blockDim.x;
            v[k] = i < nvec ? __ldcs(s + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int64_t i = b + (int64_t)k * blockDim.x;
            if (i < nvec) d[i] = v[k];
        }
    }
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = 16 * nvec + tid; i < bytes; i += (int64_t)gridDim.x * blockDim.x) {
        dst[i] = src[i];
    }
}

}  // namespace

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
    const bool vec = (reinterpret_cast<uintptr_t>(dst) % 16) == 0 &&
                     (reinterpret_cast<uintptr_t>(src) % 16) == 0;
    const int64_t nvec = vec ? bytes / 16 : 0;
    // two vectors per thread from 1 MB of source, one below (measured on
    // GB300 between 64 KB and 42 MB moved, in back-to-back dependent launches)
    const int V = nvec >= (int64_t)1 << 16 ? 2 : 1;
    const int threads = 256;
    const int64_t work = nvec > 0 ? (nvec + V - 1) / V : bytes;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 64;
    if (blocks > cap) blocks = cap;  // a grid-stride pass beyond 64 CTAs per SM
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    const char* sp = static_cast<const char*>(src);
    char* dp = static_cast<char*>(dst);
    if (V == 2) return cudaLaunchKernelEx(&cfg, copy_kernel<2>, sp, dp, nvec, bytes);
    return cudaLaunchKernelEx(&cfg, copy_kernel<1>, sp, dp, nvec, bytes);
}

}  // namespace edge
