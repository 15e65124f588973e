/*
 * edge_ops.h -- C ABI of the GB300 fused decode-seam operator library
 * (libedge_ops.so, sm_103a).
 *
 * Four operators from the fused decode seams of small transformer decoders:
 *   edge_qk_norm_rope  per-head QK-RMSNorm + rotary embedding prologue
 *   edge_add_rmsnorm   residual add followed by RMSNorm of the rounded sum
 *   edge_rmsnorm       RMSNorm, with or without a weight
 *   edge_glu_act       SiLU / tanh-GELU gated activation of a merged gate+up
 * Each op can write a static-scale FP8 E4M3 output instead of the activation
 * dtype.
 *
 * Sources, by page and section:
 *   "thox-edge-ops v2: fused decode kernels for small models on THOX edge
 *     hardware": section 3 (tensor contract; R1 numerics; R2 conventions;
 *     R5 safety), section 5.1 (operators), section 5.4 (fused QK-norm+RoPE),
 *     section 5.5 (validation before pointer arithmetic).
 *   ninfer pull request "Register the text profile of ops::rmsnorm_rope ...":
 *     "Implementation" (out-of-place partial-rotary text profile) and the
 *     review (pass eps and theta, keep the shape dispatch inside the op).
 *   FlashRT "optimization-details": the static-scale FP8 fused kernels, the
 *     static calibration and the no-weight RMSNorm.
 *
 * Common contract (all entry points):
 *   - Every tensor pointer is a caller-owned CUDA device pointer to a dense,
 *     row-major (contiguous) array.  The library allocates nothing, caches
 *     no tensor, never synchronizes the device or the stream, and copies
 *     nothing between host and device.  Every call can be captured into a
 *     CUDA graph.
 *   - `stream` is a cudaStream_t, or NULL for the legacy default stream.
 *     The kernel is enqueued on it, and the call returns once it is enqueued.
 *   - `dt` is the activation dtype: EDGE_F32, EDGE_F16 or EDGE_BF16.  Norm
 *     weights have dtype `dt`.  The output dtype `out_dt` is either `dt` or
 *     EDGE_FP8_E4M3.
 *   - Arithmetic is fp32 with one rounding of each output, to nearest even
 *     (R1).  With an FP8 output, the fp32 result y is multiplied by
 *     `inv_scale` in fp32 and converted to E4M3 with saturation to +-448.
 *     Here inv_scale = 1 / scale, and scale = amax / 448 comes from a
 *     calibration pass.  `inv_scale` is ignored unless out_dt is FP8.
 *   - Validation happens before any pointer arithmetic or launch.  An
 *     invalid call launches nothing and returns a nonzero edge_status.  A
 *     call with zero rows or tokens returns EDGE_OK and launches nothing.
 *   - Pointers must be aligned to their element size (EDGE_ERR_ALIGN
 *     otherwise).  16-byte aligned tensors whose rows are multiples of 16
 *     bytes take the vectorized path; other valid layouts take a scalar GPU
 *     path.  There is never a CPU fallback.
 *   - An output may alias its input exactly (in place) where stated.  Any
 *     other overlap between a written buffer and another buffer is rejected
 *     with EDGE_ERR_ALIAS.  An FP8 output must not alias an input.
 *   - A launch failure returns EDGE_ERR_CUDA.  edge_last_cuda_error() then
 *     gives the cudaError_t of the calling thread's last failure.
 */
#ifndef EDGE_OPS_H
#define EDGE_OPS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EDGE_F32 = 0,
    EDGE_F16 = 1,
    EDGE_BF16 = 2,
    EDGE_FP8_E4M3 = 3 /* output only: OCP E4M3 "fn", saturating */
} edge_dtype;

typedef enum {
    EDGE_OK = 0,
    EDGE_ERR_NULL = 1,        /* a required pointer is NULL */
    EDGE_ERR_DTYPE = 2,       /* unknown dtype, or out_dt not dt / FP8 */
    EDGE_ERR_SHAPE = 3,       /* negative or inconsistent sizes */
    EDGE_ERR_ALIGN = 4,       /* a pointer not aligned to its element size */
    EDGE_ERR_ALIAS = 5,       /* a written buffer overlaps another buffer */
    EDGE_ERR_UNSUPPORTED = 6, /* valid but beyond this build's limits */
    EDGE_ERR_CUDA = 7,        /* the launch failed (see edge_last_cuda_error) */
    EDGE_ERR_VALUE = 8        /* bad scalar: eps, inv_scale, flag or enum */
} edge_status;

typedef enum {
    EDGE_ROPE_ROTATE_HALF = 0, /* pairs (j, j + rotary_dim/2), GPT-NeoX */
    EDGE_ROPE_INTERLEAVED = 1  /* pairs (2j, 2j + 1), GPT-J */
} edge_rope_layout;

typedef enum {
    EDGE_ACT_SILU = 0,     /* silu(g) = g / (1 + e^-g) */
    EDGE_ACT_GELU_TANH = 1 /* 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) */
} edge_act;

/*
 * RMSNorm ("thox-edge-ops v2", section 5.1; FlashRT no-weight RMSNorm).
 *
 *   out[t, i] = x[t, i] * r_t * (w[i] + weight_offset),
 *   r_t = 1 / sqrt(mean_i(x[t, i]^2) + eps).
 *
 * x:    [rows, hidden] of dt.
 * w:    [hidden] of dt, or NULL for the no-weight form out = x * r.
 *       weight_offset 0 applies w directly (Llama).  weight_offset 1
 *       applies 1 + w in fp32 (Gemma, zero-centred weight).
 * out:  [rows, hidden] of out_dt.  out == x is allowed when out_dt == dt.
 * eps:  finite and >= 0; it sits inside the root.
 * Errors: NULL x/out; rows < 0 or hidden <= 0; eps or weight_offset invalid;
 * partial overlap.
 */
edge_status edge_rmsnorm(void* out, edge_dtype out_dt, const void* x, const void* w,
                         edge_dtype dt, int64_t rows, int64_t hidden, float eps,
                         int weight_offset, float inv_scale, void* stream);

/*
 * Fused residual-add RMSNorm ("thox-edge-ops v2", R1 and sections 5.1 and
 * 5.2; FlashRT residual_add_rms_norm_fp8_static).
 *
 *   residual[t, i] <- round_dt(fp32(x[t, i]) + fp32(residual[t, i]))
 *   out[t, i]       = RMSNorm(residual[t, :])[i]
 *
 * The sum is widened, added in fp32 and rounded once to dt.  The result is
 * bit-identical to an eager add of the two tensors.  The norm (same
 * arguments as edge_rmsnorm) is taken of the rounded sum.
 * x:        [rows, hidden] of dt (read).
 * residual: [rows, hidden] of dt (read, then overwritten with the sum).
 * out:      [rows, hidden] of out_dt.  out == x is allowed when out_dt == dt.
 *           out must not overlap residual.
 */
edge_status edge_add_rmsnorm(void* out, edge_dtype out_dt, const void* x, void* residual,
                             const void* w, edge_dtype dt, int64_t rows, int64_t hidden,
                             float eps, int weight_offset, float inv_scale, void* stream);

/*
 * Gated activation of a merged gate+up projection ("thox-edge-ops v2",
 * section 5.1; FlashRT gate_geglu_merged_fp8).
 *
 *   out[t, i] = act(gate_up[t, i]) * gate_up[t, d + i],  0 <= i < d
 *
 * The gate is the first half of each row and the up projection the second.
 * gate_up: [rows, 2*d] of dt.   out: [rows, d] of out_dt (no overlap).
 * act: EDGE_ACT_SILU or EDGE_ACT_GELU_TANH.
 */
edge_status edge_glu_act(void* out, edge_dtype out_dt, const void* gate_up, edge_dtype dt,
                         int64_t rows, int64_t d, edge_act act, float inv_scale, void* stream);

/*
 * Fused per-head QK-RMSNorm + RoPE prologue ("thox-edge-ops v2", sections
 * 5.1 and 5.4; ninfer text profile, "Implementation").
 *
 * For every token t and every head h of q (weight wq) and of k (weight wk):
 *   m = round_dt(RMSNorm(head) with the head's weight)   (as edge_rmsnorm)
 *   if 0 <= positions[t] < cache_len, rotate the first rotary_dim channels
 *   of m.  For pair j < rotary_dim/2 with members (a, b), c = cos[p, j] and
 *   s = sin[p, j]:
 *        a' = a c - b s,   b' = b c + a s   (fp32, then one rounding)
 *   Channels at or past rotary_dim carry m.  A token whose position is
 *   negative or >= cache_len is normalized but not rotated, and no cache row
 *   at that position is read (R5), so no device synchronization is needed:
 *   every cache read lies inside [0, cache_len).
 *
 * q, k:        [tokens, q_heads, head_dim] and [tokens, k_heads, head_dim]
 *              of dt.  This is the innermost-first [head_dim, heads, tokens]
 *              of the ninfer profile.
 * q_out,k_out: same shapes, of out_dt.  q_out == q and k_out == k are allowed
 *              (in place) when out_dt == dt.
 * wq, wk:      [head_dim] of dt each, or NULL for unit weight.
 * rotary_dim:  even, 0 <= rotary_dim <= head_dim (0: no rotation).
 * layout:      EDGE_ROPE_ROTATE_HALF or EDGE_ROPE_INTERLEAVED.
 * positions:   [tokens] int64, device.  It may be NULL only if rotary_dim == 0
 *              or cache_len == 0.
 * cos, sin:    [cache_len, rotary_dim/2] fp32, device.  Row p holds the
 *              angles of position p, so theta is the caller's.  They may be
 *              NULL only if rotary_dim == 0 or cache_len == 0.
 * The FP8 epilogue quantizes the rotated value and the rounded m of the
 * channels that do not rotate.
 */
edge_status edge_qk_norm_rope(void* q_out, void* k_out, edge_dtype out_dt, const void* q,
                              const void* k, const void* wq, const void* wk, edge_dtype dt,
                              int64_t tokens, int32_t q_heads, int32_t k_heads, int32_t head_dim,
                              int32_t rotary_dim, edge_rope_layout layout,
                              const int64_t* positions, const float* cos, const float* sin,
                              int64_t cache_len, float eps, int weight_offset, float inv_scale,
                              void* stream);

/*
 * One-read LayerNorm (FlashRT "optimization-details": siglip_layernorm_1read,
 * a single pass over a register-cached row instead of three).
 *
 *   out[t, i] = (x[t, i] - mu_t) / sqrt(var_t + eps) * gamma[i] + beta[i]
 *   mu_t = mean_i x[t, i],  var_t = mean_i (x[t, i] - mu_t)^2  (biased)
 *
 * x: [rows, hidden] of dt.  gamma, beta: [hidden] of dt, each nullable (1, 0).
 * out: [rows, hidden] of out_dt; out == x is allowed when out_dt == dt.
 * fp32 arithmetic, one rounding (or the FP8 epilogue).
 */
edge_status edge_layernorm(void* out, edge_dtype out_dt, const void* x, const void* gamma,
                           const void* beta, edge_dtype dt, int64_t rows, int64_t hidden,
                           float eps, float inv_scale, void* stream);

/*
 * Standalone static-scale FP8 quantization (FlashRT "optimization-details":
 * quantize_fp8_static).  out[i] = E4M3(fl32(x[i]) * inv_scale), to nearest
 * even with saturation to +-448.  x: n elements of dt.  out: n bytes, which
 * must not overlap x.  inv_scale must be finite and > 0.
 */
edge_status edge_quantize_fp8(void* out, const void* x, edge_dtype dt, int64_t n, float inv_scale,
                              void* stream);

/*
 * Fused QKV split + QK-norm + RoPE + KV-cache write (FlashRT
 * "optimization-details": qkv_split_rope_kvcache; "thox-edge-ops v2",
 * roadmap item 4: a KV write fused into the prologue).
 *
 * qkv:   [tokens, (q_heads + 2 kv_heads) head_dim] of dt.  Row t holds q_heads
 *        query heads, then kv_heads key heads, then kv_heads value heads
 *        (the output of a fused QKV projection).
 * q_out: [tokens, q_heads, head_dim] of dt: the query heads after the prologue
 *        of edge_qk_norm_rope (per-head RMSNorm when normalize = 1, rounded to
 *        dt; the rotation of the first rotary_dim channels by cos/sin row
 *        positions[t]).
 * k_cache, v_cache: [num_slots, kv_heads, head_dim] of dt.  Row slots[t]
 *        receives the key heads of token t after the same prologue, and the
 *        value heads unchanged.  A token whose slot is negative or
 *        >= num_slots writes no cache row, so the cache is never written out
 *        of bounds; the other rows are left untouched.  When two tokens name
 *        the same slot, which token's row remains there is unspecified.
 * slots: [tokens] int64, device.  Caches and slots may be NULL when
 *        kv_heads == 0 or num_slots == 0.
 * slots == NULL with num_slots == 0 writes no cache row at all (the query
 * heads are still produced).
 * Output dtype is dt (no FP8 epilogue).  Outputs must not overlap each other
 * or any input.  Element-aligned tensors of any head size up to 2048 are
 * served: a vector path when head_dim * size(dt) is a power-of-two multiple
 * of 16 up to 512 bytes, the tensors are 16-byte aligned and the rotary width
 * suits 16-byte vectors, else a scalar path.  EDGE_ERR_UNSUPPORTED: head_dim
 * above 2048, or tokens * (q_heads + 2 kv_heads) above 2^31 - 1.
 */
edge_status edge_qkv_rope_cache(void* q_out, void* k_cache, void* v_cache, const void* qkv,
                                const void* wq, const void* wk, edge_dtype dt, int64_t tokens,
                                int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                                int32_t rotary_dim, edge_rope_layout layout,
                                const int64_t* positions, const float* cos, const float* sin,
                                int64_t cache_len, const int64_t* slots, int64_t num_slots,
                                float eps, int weight_offset, int normalize, void* stream);

/* Flags of edge_qk_norm_rope_ex. */
enum {
    /* Rotate the fp32 normalized value and round once after the rotation,
     * instead of rotating its rounding to dt.  This is the variant the
     * ninfer review asks for (item 1).  Channels that do not rotate are
     * unchanged (they carry round_dt of the normalized value either way). */
    EDGE_QK_ROTATE_UNROUNDED = 1
};

/*
 * edge_qk_norm_rope with option flags (EDGE_QK_* above; 0 gives exactly
 * edge_qk_norm_rope).  Unknown flags return EDGE_ERR_VALUE.
 */
edge_status edge_qk_norm_rope_ex(void* q_out, void* k_out, edge_dtype out_dt, const void* q,
                                 const void* k, const void* wq, const void* wk, edge_dtype dt,
                                 int64_t tokens, int32_t q_heads, int32_t k_heads,
                                 int32_t head_dim, int32_t rotary_dim, edge_rope_layout layout,
                                 const int64_t* positions, const float* cos, const float* sin,
                                 int64_t cache_len, float eps, int weight_offset, float inv_scale,
                                 uint32_t flags, void* stream);

/*
 * Standalone rotary embedding ("thox-edge-ops v2", section 5.1, the rotary
 * operator: query and key in one launch).  For every head of q and k of token
 * t with 0 <= positions[t] < cache_len, pair j < rotary_dim/2 (rotate-half or
 * interleaved, as in edge_qk_norm_rope) becomes a' = a c - b s, b' = b c + a s
 * in fp32, rounded once (or the FP8 epilogue).  Other channels, and every
 * channel of a token outside the cache, are copied unchanged.  Same layout,
 * aliasing and error rules as edge_qk_norm_rope, with no weights and no eps.
 */
edge_status edge_rope(void* q_out, void* k_out, edge_dtype out_dt, const void* q, const void* k,
                      edge_dtype dt, int64_t tokens, int32_t q_heads, int32_t k_heads,
                      int32_t head_dim, int32_t rotary_dim, edge_rope_layout layout,
                      const int64_t* positions, const float* cos, const float* sin,
                      int64_t cache_len, float inv_scale, void* stream);

/*
 * Plain device copy of `bytes` bytes from src to dst, in the launch form of the
 * operators above (a one-shot grid of 16-byte vectors, each CTA's source span
 * prefetched into L2 before the dependent-launch wait).  It computes nothing:
 * it is the yardstick the measurements set each operator against, the time a
 * kernel of that form needs to move the same number of bytes.  No page defines
 * it.  dst and src are device pointers of any alignment (16-byte aligned ones
 * take the vector path); the ranges must not overlap (EDGE_ERR_ALIAS).
 * bytes < 0: EDGE_ERR_SHAPE; bytes == 0 launches nothing.
 */
edge_status edge_copy(void* dst, const void* src, int64_t bytes, void* stream);

/* A static, NUL-terminated description of a status code. */
const char* edge_status_str(edge_status status);

/* The cudaError_t of the calling thread's last EDGE_ERR_CUDA (0 if none). */
int edge_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int edge_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EDGE_OPS_H */
