// edge_ops.cu -- the C ABI of libedge_ops.so: validation, then dispatch.
//
// Every entry point validates its arguments completely before any pointer
// arithmetic or launch ("thox-edge-ops v2", section 5.5): dtypes, NULL
// pointers, sizes, scalars, alignment, and overlap between written and read
// buffers.  An invalid call launches nothing and returns an edge_status.  The
// launchers in qk_norm_rope.cu, rows.cu and glu.cu then choose the kernel and
// launch shape.  Nothing here allocates, synchronizes or copies.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <atomic>
#include <mutex>

#include "../../include/edge_ops.h"
#include "launch.h"

namespace edge {

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = 148;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int resident_ctas(const void* fn, int threads) {
    struct Entry {
        const void* fn;
        int threads, dev, n;
    };
    static std::mutex mu;
    static Entry table[128];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
        if (table[i].fn == fn && table[i].threads == threads && table[i].dev == dev) {
            return table[i].n;
        }
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
    }
    if (n < 1) n = 1;
    if (used < 128) table[used++] = Entry{fn, threads, dev, n};
    return n;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("EDGE_OPS_PDL");
        return !(v != nullptr && v[0] == '0');
    }();
    return on;
}

}  // namespace edge

namespace {

thread_local int g_last_cuda_error = 0;

bool act_dtype(edge_dtype dt) { return dt == EDGE_F32 || dt == EDGE_F16 || dt == EDGE_BF16; }

int64_t esize(edge_dtype dt) { return dt == EDGE_F32 ? 4 : (dt == EDGE_FP8_E4M3 ? 1 : 2); }

bool aligned(const void* p, int64_t n) {
    return p == nullptr || (reinterpret_cast<uintptr_t>(p) % (uintptr_t)n) == 0;
}

// Byte range [p, p + n) of a buffer; empty ranges never overlap.
struct Span {
    uintptr_t lo, hi;
};

Span span(const void* p, int64_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, p == nullptr ? lo : lo + (uintptr_t)bytes};
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// A written buffer may coincide with one input exactly (in place), else must not overlap it.
bool bad_alias(Span out, Span in, bool exact_ok) {
    if (!overlap(out, in)) return false;
    return !(exact_ok && out.lo == in.lo && out.hi == in.hi);
}

bool finite_nonneg(float v) { return std::isfinite(v) && v >= 0.0f; }

// rows * cols * bytes without overflow; false if it would exceed int64.
bool checked_bytes(int64_t rows, int64_t cols, int64_t bytes, int64_t* out) {
    if (rows < 0 || cols < 0) return false;
    if (cols != 0 && rows > INT64_MAX / cols) return false;
    const int64_t n = rows * cols;
    if (bytes != 0 && n > INT64_MAX / bytes) return false;
    *out = n * bytes;
    return true;
}

edge_status finish(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return EDGE_ERR_CUDA;
    }
    return EDGE_OK;
}

edge_status check_out_dt(edge_dtype out_dt, edge_dtype dt) {
    if (!act_dtype(dt)) return EDGE_ERR_DTYPE;
    if (out_dt != dt && out_dt != EDGE_FP8_E4M3) return EDGE_ERR_DTYPE;
    return EDGE_OK;
}

edge_status check_scale(edge_dtype out_dt, float inv_scale) {
    if (out_dt == EDGE_FP8_E4M3 && !(std::isfinite(inv_scale) && inv_scale > 0.0f)) {
        return EDGE_ERR_VALUE;
    }
    return EDGE_OK;
}

edge_status rows_entry(void* out, edge_dtype out_dt, const void* x, void* residual, bool fused,
                       const void* w, edge_dtype dt, int64_t rows, int64_t hidden, float eps,
                       int weight_offset, float inv_scale, void* stream) {
    edge_status st = check_out_dt(out_dt, dt);
    if (st != EDGE_OK) return st;
    if (x == nullptr || out == nullptr || (fused && residual == nullptr)) return EDGE_ERR_NULL;
    if (rows < 0 || hidden <= 0) return EDGE_ERR_SHAPE;
    if (!finite_nonneg(eps) || (weight_offset != 0 && weight_offset != 1)) return EDGE_ERR_VALUE;
    if ((st = check_scale(out_dt, inv_scale)) != EDGE_OK) return st;
    int64_t in_bytes = 0, out_bytes = 0;
    if (!checked_bytes(rows, hidden, esize(dt), &in_bytes) ||
        !checked_bytes(rows, hidden, esize(out_dt), &out_bytes)) {
        return EDGE_ERR_SHAPE;
    }
    if (hidden > edge::kMaxHidden) return EDGE_ERR_UNSUPPORTED;
    const int64_t es = esize(dt);
    if (!aligned(x, es) || !aligned(residual, es) || !aligned(w, es) || !aligned(out, esize(out_dt))) {
        return EDGE_ERR_ALIGN;
    }
    const Span so = span(out, out_bytes), sx = span(x, in_bytes), sw = span(w, hidden * es);
    const Span sr = span(fused ? residual : nullptr, in_bytes);
    const bool same_dt = out_dt == dt;
    if (bad_alias(so, sx, same_dt) || overlap(so, sw) || overlap(so, sr)) return EDGE_ERR_ALIAS;
    if (fused && (overlap(sr, sx) || overlap(sr, sw))) return EDGE_ERR_ALIAS;
    if (rows == 0) return EDGE_OK;

    edge::RowsArgs a;
    a.x = x;
    a.residual = fused ? residual : nullptr;
    a.w = w;
    a.beta = nullptr;
    a.layernorm = 0;
    a.out = out;
    a.rows = rows;
    a.hidden = hidden;
    a.dt = (int)dt;
    a.out_dt = (int)out_dt;
    a.eps = eps;
    a.inv_scale = inv_scale;
    a.weight_offset = weight_offset;
    return finish(edge::launch_rows(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

namespace {

static edge_status qk_entry(void* q_out, void* k_out, edge_dtype out_dt, const void* q,
                            const void* k, const void* wq, const void* wk, edge_dtype dt,
                            int64_t tokens, int32_t q_heads, int32_t k_heads, int32_t head_dim,
                            int32_t rotary_dim, edge_rope_layout layout, const int64_t* positions,
                            const float* cos, const float* sin, int64_t cache_len, float eps,
                            int weight_offset, float inv_scale, int mode, void* stream) {
    edge_status st = check_out_dt(out_dt, dt);
    if (st != EDGE_OK) return st;
    if (q == nullptr || q_out == nullptr) return EDGE_ERR_NULL;
    if (k_heads > 0 && (k == nullptr || k_out == nullptr)) return EDGE_ERR_NULL;
    if (tokens < 0 || q_heads < 1 || k_heads < 0 || head_dim < 1 || cache_len < 0) {
        return EDGE_ERR_SHAPE;
    }
    if (rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return EDGE_ERR_SHAPE;
    if (layout != EDGE_ROPE_ROTATE_HALF && layout != EDGE_ROPE_INTERLEAVED) return EDGE_ERR_VALUE;
    if (!finite_nonneg(eps) || (weight_offset != 0 && weight_offset != 1)) return EDGE_ERR_VALUE;
    if ((st = check_scale(out_dt, inv_scale)) != EDGE_OK) return st;
    const bool may_rotate = rotary_dim > 0 && cache_len > 0;
    if (may_rotate && (positions == nullptr || cos == nullptr || sin == nullptr)) {
        return EDGE_ERR_NULL;
    }
    const int64_t es = esize(dt), eo = esize(out_dt);
    int64_t qb = 0, kb = 0, qob = 0, kob = 0, cb = 0;
    if (!checked_bytes(tokens, (int64_t)q_heads * head_dim, es, &qb) ||
        !checked_bytes(tokens, (int64_t)k_heads * head_dim, es, &kb) ||
        !checked_bytes(tokens, (int64_t)q_heads * head_dim, eo, &qob) ||
        !checked_bytes(tokens, (int64_t)k_heads * head_dim, eo, &kob) ||
        !checked_bytes(cache_len, rotary_dim / 2, 4, &cb)) {
        return EDGE_ERR_SHAPE;
    }
    if (head_dim > edge::kMaxQKHeadDim) return EDGE_ERR_UNSUPPORTED;
    if (tokens > edge::kMaxUnits / ((int64_t)q_heads + k_heads)) return EDGE_ERR_UNSUPPORTED;
    if (!aligned(q, es) || !aligned(k, es) || !aligned(wq, es) || !aligned(wk, es) ||
        !aligned(q_out, eo) || !aligned(k_out, eo) || !aligned(positions, 8) || !aligned(cos, 4) ||
        !aligned(sin, 4)) {
        return EDGE_ERR_ALIGN;
    }
    const bool same_dt = out_dt == dt;
    const Span sq = span(q, qb), sk = span(k_heads ? k : nullptr, kb);
    const Span sqo = span(q_out, qob), sko = span(k_heads ? k_out : nullptr, kob);
    const Span ro[] = {span(wq, head_dim * es), span(wk, head_dim * es),
                       span(may_rotate ? positions : nullptr, tokens * 8),
                       span(may_rotate ? cos : nullptr, cb), span(may_rotate ? sin : nullptr, cb)};
    if (bad_alias(sqo, sq, same_dt) || bad_alias(sko, sk, same_dt) || overlap(sqo, sk) ||
        overlap(sko, sq) || overlap(sqo, sko)) {
        return EDGE_ERR_ALIAS;
    }
    for (const Span& r : ro) {
        if (overlap(sqo, r) || overlap(sko, r)) return EDGE_ERR_ALIAS;
    }
    if (tokens == 0) return EDGE_OK;

    edge::QKArgs a;
    a.q = q;
    a.k = k_heads ? k : nullptr;
    a.q_out = q_out;
    a.k_out = k_heads ? k_out : nullptr;
    a.wq = wq;
    a.wk = wk;
    a.pos = may_rotate ? positions : nullptr;
    a.cos = may_rotate ? cos : nullptr;
    a.sin = may_rotate ? sin : nullptr;
    a.tokens = tokens;
    a.cache_len = cache_len;
    a.q_heads = q_heads;
    a.k_heads = k_heads;
    a.head_dim = head_dim;
    a.rotary_dim = rotary_dim;
    a.layout = (int)layout;
    a.dt = (int)dt;
    a.out_dt = (int)out_dt;
    a.eps = eps;
    a.inv_scale = inv_scale;
    a.weight_offset = weight_offset;
    a.mode = mode;
    return finish(edge::launch_qk(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

edge_status edge_rmsnorm(void* out, edge_dtype out_dt, const void* x, const void* w, edge_dtype dt,
                         int64_t rows, int64_t hidden, float eps, int weight_offset,
                         float inv_scale, void* stream) {
    return rows_entry(out, out_dt, x, nullptr, false, w, dt, rows, hidden, eps, weight_offset,
                      inv_scale, stream);
}

edge_status edge_add_rmsnorm(void* out, edge_dtype out_dt, const void* x, void* residual,
                             const void* w, edge_dtype dt, int64_t rows, int64_t hidden, float eps,
                             int weight_offset, float inv_scale, void* stream) {
    return rows_entry(out, out_dt, x, residual, true, w, dt, rows, hidden, eps, weight_offset,
                      inv_scale, stream);
}

edge_status edge_qkv_rope_cache(void* q_out, void* k_cache, void* v_cache, const void* qkv,
                                const void* wq, const void* wk, edge_dtype dt, int64_t tokens,
                                int32_t q_heads, int32_t kv_heads, int32_t head_dim,
                                int32_t rotary_dim, edge_rope_layout layout,
                                const int64_t* positions, const float* cos, const float* sin,
                                int64_t cache_len, const int64_t* slots, int64_t num_slots,
                                float eps, int weight_offset, int normalize, void* stream) {
    if (!act_dtype(dt)) return EDGE_ERR_DTYPE;
    if (qkv == nullptr || q_out == nullptr) return EDGE_ERR_NULL;
    const bool writes_cache = kv_heads > 0 && num_slots > 0;
    if (writes_cache && (k_cache == nullptr || v_cache == nullptr || slots == nullptr)) {
        return EDGE_ERR_NULL;
    }
    if (tokens < 0 || q_heads < 1 || kv_heads < 0 || head_dim < 1 || cache_len < 0 ||
        num_slots < 0) {
        return EDGE_ERR_SHAPE;
    }
    if (rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return EDGE_ERR_SHAPE;
    if (layout != EDGE_ROPE_ROTATE_HALF && layout != EDGE_ROPE_INTERLEAVED) return EDGE_ERR_VALUE;
    if (!finite_nonneg(eps) || (weight_offset != 0 && weight_offset != 1) ||
        (normalize != 0 && normalize != 1)) {
        return EDGE_ERR_VALUE;
    }
    const bool may_rotate = rotary_dim > 0 && cache_len > 0;
    if (may_rotate && (positions == nullptr || cos == nullptr || sin == nullptr)) {
        return EDGE_ERR_NULL;
    }
    const int64_t es = esize(dt);
    const int64_t heads_row = (int64_t)q_heads + 2 * (int64_t)kv_heads;
    int64_t in_b = 0, q_b = 0, c_b = 0, cs_b = 0;
    if (!checked_bytes(tokens, heads_row * head_dim, es, &in_b) ||
        !checked_bytes(tokens, (int64_t)q_heads * head_dim, es, &q_b) ||
        !checked_bytes(num_slots, (int64_t)kv_heads * head_dim, es, &c_b) ||
        !checked_bytes(cache_len, rotary_dim / 2, 4, &cs_b)) {
        return EDGE_ERR_SHAPE;
    }
    if (head_dim > edge::kMaxQKHeadDim) return EDGE_ERR_UNSUPPORTED;
    if (tokens > edge::kMaxUnits / heads_row) return EDGE_ERR_UNSUPPORTED;
    if (!aligned(qkv, es) || !aligned(q_out, es) || !aligned(k_cache, es) ||
        !aligned(v_cache, es) || !aligned(wq, es) || !aligned(wk, es) || !aligned(positions, 8) ||
        !aligned(slots, 8) || !aligned(cos, 4) || !aligned(sin, 4)) {
        return EDGE_ERR_ALIGN;
    }
    const Span sq = span(q_out, q_b);
    const Span sk = span(writes_cache ? k_cache : nullptr, c_b);
    const Span sv = span(writes_cache ? v_cache : nullptr, c_b);
    const Span ro[] = {span(qkv, in_b), span(wq, head_dim * es), span(wk, head_dim * es),
                       span(may_rotate ? positions : nullptr, tokens * 8),
                       span(may_rotate ? cos : nullptr, cs_b), span(may_rotate ? sin : nullptr, cs_b),
                       span(writes_cache ? slots : nullptr, tokens * 8)};
    if (overlap(sq, sk) || overlap(sq, sv) || overlap(sk, sv)) return EDGE_ERR_ALIAS;
    for (const Span& r : ro) {
        if (overlap(sq, r) || overlap(sk, r) || overlap(sv, r)) return EDGE_ERR_ALIAS;
    }
    if (tokens == 0) return EDGE_OK;
    edge::QKVArgs a;
    a.qkv = qkv;
    a.q_out = q_out;
    a.k_cache = writes_cache ? k_cache : nullptr;
    a.v_cache = writes_cache ? v_cache : nullptr;
    a.wq = wq;
    a.wk = wk;
    a.pos = may_rotate ? positions : nullptr;
    a.cos = may_rotate ? cos : nullptr;
    a.sin = may_rotate ? sin : nullptr;
    a.slots = writes_cache ? slots : nullptr;
    a.tokens = tokens;
    a.cache_len = cache_len;
    a.num_slots = writes_cache ? num_slots : 0;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.head_dim = head_dim;
    a.rotary_dim = rotary_dim;
    a.layout = (int)layout;
    a.dt = (int)dt;
    a.normalize = normalize;
    a.weight_offset = weight_offset;
    a.eps = eps;
    bool handled = false;
    cudaError_t e = edge::launch_qkv_cache(a, static_cast<cudaStream_t>(stream), &handled);
    if (e == cudaSuccess && !handled) return EDGE_ERR_UNSUPPORTED;
    return finish(e);
}

edge_status edge_layernorm(void* out, edge_dtype out_dt, const void* x, const void* gamma,
                           const void* beta, edge_dtype dt, int64_t rows, int64_t hidden,
                           float eps, float inv_scale, void* stream) {
    edge_status st = check_out_dt(out_dt, dt);
    if (st != EDGE_OK) return st;
    if (x == nullptr || out == nullptr) return EDGE_ERR_NULL;
    if (rows < 0 || hidden <= 0) return EDGE_ERR_SHAPE;
    if (!finite_nonneg(eps)) return EDGE_ERR_VALUE;
    if ((st = check_scale(out_dt, inv_scale)) != EDGE_OK) return st;
    int64_t in_bytes = 0, out_bytes = 0;
    if (!checked_bytes(rows, hidden, esize(dt), &in_bytes) ||
        !checked_bytes(rows, hidden, esize(out_dt), &out_bytes)) {
        return EDGE_ERR_SHAPE;
    }
    if (hidden > edge::kMaxHidden) return EDGE_ERR_UNSUPPORTED;
    const int64_t es = esize(dt);
    if (!aligned(x, es) || !aligned(gamma, es) || !aligned(beta, es) ||
        !aligned(out, esize(out_dt))) {
        return EDGE_ERR_ALIGN;
    }
    const Span so = span(out, out_bytes);
    if (bad_alias(so, span(x, in_bytes), out_dt == dt) || overlap(so, span(gamma, hidden * es)) ||
        overlap(so, span(beta, hidden * es))) {
        return EDGE_ERR_ALIAS;
    }
    if (rows == 0) return EDGE_OK;
    edge::RowsArgs a;
    a.x = x;
    a.residual = nullptr;
    a.w = gamma;
    a.beta = beta;
    a.layernorm = 1;
    a.out = out;
    a.rows = rows;
    a.hidden = hidden;
    a.dt = (int)dt;
    a.out_dt = (int)out_dt;
    a.eps = eps;
    a.inv_scale = inv_scale;
    a.weight_offset = 0;
    return finish(edge::launch_rows(a, static_cast<cudaStream_t>(stream)));
}

edge_status edge_quantize_fp8(void* out, const void* x, edge_dtype dt, int64_t n, float inv_scale,
                              void* stream) {
    if (!act_dtype(dt)) return EDGE_ERR_DTYPE;
    if (out == nullptr || x == nullptr) return EDGE_ERR_NULL;
    if (n < 0) return EDGE_ERR_SHAPE;
    if (!(std::isfinite(inv_scale) && inv_scale > 0.0f)) return EDGE_ERR_VALUE;
    int64_t in_bytes = 0;
    if (!checked_bytes(n, 1, esize(dt), &in_bytes)) return EDGE_ERR_SHAPE;
    if (n > edge::kMaxUnits * 8) return EDGE_ERR_UNSUPPORTED;
    if (!aligned(x, esize(dt))) return EDGE_ERR_ALIGN;
    if (overlap(span(out, n), span(x, in_bytes))) return EDGE_ERR_ALIAS;
    if (n == 0) return EDGE_OK;
    edge::QuantArgs a;
    a.x = x;
    a.out = out;
    a.n = n;
    a.dt = (int)dt;
    a.inv_scale = inv_scale;
    return finish(edge::launch_quant(a, static_cast<cudaStream_t>(stream)));
}

edge_status edge_glu_act(void* out, edge_dtype out_dt, const void* gate_up, edge_dtype dt,
                         int64_t rows, int64_t d, edge_act act, float inv_scale, void* stream) {
    edge_status st = check_out_dt(out_dt, dt);
    if (st != EDGE_OK) return st;
    if (out == nullptr || gate_up == nullptr) return EDGE_ERR_NULL;
    if (rows < 0 || d <= 0) return EDGE_ERR_SHAPE;
    if (act != EDGE_ACT_SILU && act != EDGE_ACT_GELU_TANH) return EDGE_ERR_VALUE;
    if ((st = check_scale(out_dt, inv_scale)) != EDGE_OK) return st;
    int64_t in_bytes = 0, out_bytes = 0;
    if (d > INT64_MAX / 2 || !checked_bytes(rows, 2 * d, esize(dt), &in_bytes) ||
        !checked_bytes(rows, d, esize(out_dt), &out_bytes)) {
        return EDGE_ERR_SHAPE;
    }
    if (!aligned(gate_up, esize(dt)) || !aligned(out, esize(out_dt))) return EDGE_ERR_ALIGN;
    if (overlap(span(out, out_bytes), span(gate_up, in_bytes))) return EDGE_ERR_ALIAS;
    if (rows == 0) return EDGE_OK;

    edge::GluArgs a;
    a.gate_up = gate_up;
    a.out = out;
    a.rows = rows;
    a.d = d;
    a.dt = (int)dt;
    a.out_dt = (int)out_dt;
    a.act = (int)act;
    a.inv_scale = inv_scale;
    return finish(edge::launch_glu(a, static_cast<cudaStream_t>(stream)));
}

edge_status edge_qk_norm_rope(void* q_out, void* k_out, edge_dtype out_dt, const void* q,
                              const void* k, const void* wq, const void* wk, edge_dtype dt,
                              int64_t tokens, int32_t q_heads, int32_t k_heads, int32_t head_dim,
                              int32_t rotary_dim, edge_rope_layout layout,
                              const int64_t* positions, const float* cos, const float* sin,
                              int64_t cache_len, float eps, int weight_offset, float inv_scale,
                              void* stream) {
    return qk_entry(q_out, k_out, out_dt, q, k, wq, wk, dt, tokens, q_heads, k_heads, head_dim,
                    rotary_dim, layout, positions, cos, sin, cache_len, eps, weight_offset,
                    inv_scale, 1 /* normalize */, stream);
}

edge_status edge_qk_norm_rope_ex(void* q_out, void* k_out, edge_dtype out_dt, const void* q,
                                 const void* k, const void* wq, const void* wk, edge_dtype dt,
                                 int64_t tokens, int32_t q_heads, int32_t k_heads,
                                 int32_t head_dim, int32_t rotary_dim, edge_rope_layout layout,
                                 const int64_t* positions, const float* cos, const float* sin,
                                 int64_t cache_len, float eps, int weight_offset, float inv_scale,
                                 uint32_t flags, void* stream) {
    if ((flags & ~(uint32_t)EDGE_QK_ROTATE_UNROUNDED) != 0) return EDGE_ERR_VALUE;
    const int mode = 1 | ((flags & EDGE_QK_ROTATE_UNROUNDED) ? 2 : 0);
    return qk_entry(q_out, k_out, out_dt, q, k, wq, wk, dt, tokens, q_heads, k_heads, head_dim,
                    rotary_dim, layout, positions, cos, sin, cache_len, eps, weight_offset,
                    inv_scale, mode, stream);
}

edge_status edge_rope(void* q_out, void* k_out, edge_dtype out_dt, const void* q, const void* k,
                      edge_dtype dt, int64_t tokens, int32_t q_heads, int32_t k_heads,
                      int32_t head_dim, int32_t rotary_dim, edge_rope_layout layout,
                      const int64_t* positions, const float* cos, const float* sin,
                      int64_t cache_len, float inv_scale, void* stream) {
    return qk_entry(q_out, k_out, out_dt, q, k, nullptr, nullptr, dt, tokens, q_heads, k_heads,
                    head_dim, rotary_dim, layout, positions, cos, sin, cache_len, 0.0f, 0,
                    inv_scale, 0 /* rotate only */, stream);
}

edge_status edge_copy(void* dst, const void* src, int64_t bytes, void* stream) {
    if (dst == nullptr || src == nullptr) return EDGE_ERR_NULL;
    if (bytes < 0) return EDGE_ERR_SHAPE;
    if (overlap(span(dst, bytes), span(src, bytes))) return EDGE_ERR_ALIAS;
    if (bytes == 0) return EDGE_OK;
    return finish(edge::launch_copy(dst, src, bytes, static_cast<cudaStream_t>(stream)));
}

const char* edge_status_str(edge_status status) {
    switch (status) {
        case EDGE_OK: return "ok";
        case EDGE_ERR_NULL: return "a required pointer is NULL";
        case EDGE_ERR_DTYPE: return "unsupported dtype combination";
        case EDGE_ERR_SHAPE: return "invalid or inconsistent sizes";
        case EDGE_ERR_ALIGN: return "pointer not aligned to its element size";
        case EDGE_ERR_ALIAS: return "a written buffer overlaps another buffer";
        case EDGE_ERR_UNSUPPORTED: return "valid call beyond this build's limits";
        case EDGE_ERR_CUDA: return "CUDA launch failed";
        case EDGE_ERR_VALUE: return "invalid scalar argument";
        default: return "unknown status";
    }
}

int edge_last_cuda_error(void) { return g_last_cuda_error; }

int edge_version(void) { return 100; }

}  // extern "C"
