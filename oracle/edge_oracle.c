/*
 * edge_oracle.c -- CPU oracle for the fused decode-seam operators.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * definition of what the GPU library computes, written as scalar fp64 loops.
 * It shares no code, header, table or constant with the CUDA path and is
 * never linked into it.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Sources (web pages, cited by title and section):
 *   [TEO]  "thox-edge-ops v2: fused decode kernels for small models on THOX
 *          edge hardware": section 3 (requirements R1 numerics, R5 safety),
 *          section 5.1 (operators), section 5.4 (fused QK-norm and RoPE).
 *   [NIN]  ninfer pull request "Register the text profile of
 *          ops::rmsnorm_rope and route the two full-attention call sites to
 *          it": "Implementation" (the text profile) and "Output" (the strength
 *          control).
 *   [FRT]  FlashRT "optimization-details" (Pi0.5 on Jetson AGX Thor): the
 *          fused static-scale FP8 kernels, static calibration, and the
 *          no-weight RMSNorm.
 *
 * The displayed equations of [TEO] section 5.1 are missing from the page
 * text.  Each operator below is the standard form that the surrounding prose
 * names: RMSNorm (Zhang and Sennrich), the RoFormer pair rotation, and the
 * SiLU and tanh-GELU gated linear units.
 *
 * Number formats are decoded and rounded from their definitions: IEEE 754
 * binary32 and binary16, bfloat16 (binary32 with 8 significand bits), and the
 * OCP 8-bit E4M3 "fn" format (bias 7, no infinities, S.1111.111 is NaN,
 * largest finite 448).  Every rounding is to nearest, ties to even.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no -ffast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_PI 3.14159265358979323846264338327950288

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 };
enum { OR_ROTATE_HALF = 0, OR_INTERLEAVED = 1 };
enum { OR_SILU = 0, OR_GELU_TANH = 1 };

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

typedef struct {
    int ebits;    /* exponent field width */
    int mbits;    /* stored significand bits */
    int bias;
    int has_inf;  /* IEEE-style infinities (E4M3 "fn" has none) */
    int sat;      /* overflow saturates to the largest finite value */
} fmt_desc;

static const fmt_desc FMTS[4] = {
    {8, 23, 127, 1, 0}, /* binary32 */
    {5, 10, 15, 1, 0},  /* binary16 */
    {8, 7, 127, 1, 0},  /* bfloat16 */
    {4, 3, 7, 0, 1},    /* E4M3 fn, converted with saturation to +-448 */
};

static int fmt_ok(int f) { return f >= 0 && f <= 3; }

static int fmt_bytes(int f) { return f == OR_F32 ? 4 : (f == OR_E4M3 ? 1 : 2); }

/* Largest finite value: all-ones significand at the top exponent, except
 * E4M3 fn, whose all-ones pattern at the top exponent is NaN. */
static double fmt_max(int f)
{
    const fmt_desc* d = &FMTS[f];
    int emax = (1 << d->ebits) - 2 - d->bias;
    double frac = 2.0 - ldexp(1.0, -d->mbits);
    if (!d->has_inf) {
        emax += 1;
        frac -= ldexp(1.0, -d->mbits);
    }
    return ldexp(frac, emax);
}

/* Round v to format f, to nearest with ties to even.  Returns the rounded
 * value as a double (every value of the four formats is a double). */
double oracle_round(double v, int f)
{
    const fmt_desc* d = &FMTS[f];
    if (isnan(v)) return v;
    double maxf = fmt_max(f);
    if (isinf(v)) return d->sat ? copysign(maxf, v) : v;
    if (v == 0.0) return v;
    double a = fabs(v);
    int e;
    (void)frexp(a, &e);       /* a = m * 2^e with m in [0.5, 1) */
    int E = e - 1;            /* 2^E <= a < 2^(E+1) */
    int emin = 1 - d->bias;   /* exponent of the smallest normal */
    if (E < emin) E = emin;   /* subnormals share the smallest normal spacing */
    double q = ldexp(1.0, E - d->mbits); /* spacing of representable values */
    double r = rint(a / q) * q;          /* a/q is exact; rint ties to even */
    if (r > maxf) r = d->sat ? maxf : INFINITY;
    return copysign(r, v);
}

/* Bit pattern of a value that is exactly representable in format f. */
uint32_t oracle_bits(double r, int f)
{
    if (f == OR_F32) {
        float x = (float)r;
        uint32_t b;
        memcpy(&b, &x, 4);
        return b;
    }
    const fmt_desc* d = &FMTS[f];
    uint32_t sign = signbit(r) ? 1u : 0u;
    uint32_t emask = (1u << d->ebits) - 1u;
    uint32_t body;
    if (isnan(r)) {
        body = d->has_inf ? ((emask << d->mbits) | (1u << (d->mbits - 1)))
                          : ((emask << d->mbits) | ((1u << d->mbits) - 1u));
    } else if (isinf(r)) {
        body = emask << d->mbits;
    } else if (r == 0.0) {
        body = 0;
    } else {
        double a = fabs(r);
        int e;
        (void)frexp(a, &e);
        int E = e - 1;
        int emin = 1 - d->bias;
        if (E < emin) {
            body = (uint32_t)(a / ldexp(1.0, emin - d->mbits));
        } else {
            double frac = a / ldexp(1.0, E) - 1.0;
            body = ((uint32_t)(E + d->bias) << d->mbits) |
                   (uint32_t)(frac * ldexp(1.0, d->mbits));
        }
    }
    return (sign << (d->ebits + d->mbits)) | body;
}

/* Value of bit pattern b in format f. */
double oracle_value(uint32_t b, int f)
{
    if (f == OR_F32) {
        float x;
        memcpy(&x, &b, 4);
        return (double)x;
    }
    const fmt_desc* d = &FMTS[f];
    uint32_t sign = (b >> (d->ebits + d->mbits)) & 1u;
    uint32_t emask = (1u << d->ebits) - 1u;
    uint32_t E = (b >> d->mbits) & emask;
    uint32_t m = b & ((1u << d->mbits) - 1u);
    double v;
    if (d->has_inf && E == emask) {
        v = m ? NAN : INFINITY;
    } else if (!d->has_inf && E == emask && m == (1u << d->mbits) - 1u) {
        v = NAN;
    } else if (E == 0) {
        v = ldexp((double)m, 1 - d->bias - d->mbits);
    } else {
        v = ldexp(1.0 + ldexp((double)m, -d->mbits), (int)E - d->bias);
    }
    return sign ? -v : v;
}

static double load(const void* p, int f, int64_t i)
{
    const unsigned char* c = (const unsigned char*)p;
    uint32_t b = 0;
    switch (fmt_bytes(f)) {
    case 4: memcpy(&b, c + 4 * i, 4); break;
    case 2: { uint16_t h; memcpy(&h, c + 2 * i, 2); b = h; } break;
    default: b = c[i]; break;
    }
    return oracle_value(b, f);
}

static void store(void* p, int f, int64_t i, uint32_t b)
{
    unsigned char* c = (unsigned char*)p;
    switch (fmt_bytes(f)) {
    case 4: memcpy(c + 4 * i, &b, 4); break;
    case 2: { uint16_t h = (uint16_t)b; memcpy(c + 2 * i, &h, 2); } break;
    default: c[i] = (unsigned char)b; break;
    }
}

/* Output of one element.  For an activation-dtype output the exact value y
 * is rounded once.  For the FP8 epilogue ([FRT], fused static-scale FP8
 * kernels) the fp32 result is multiplied by the precomputed inverse scale in
 * fp32 and converted to E4M3 with saturation: the code decision is taken in
 * the same single precision as on the GPU. */
static uint32_t emit(double y, int out_fmt, float inv_scale)
{
    if (out_fmt == OR_E4M3) {
        volatile float y32 = (float)y;
        volatile float q = y32 * inv_scale;
        return oracle_bits(oracle_round((double)q, OR_E4M3), OR_E4M3);
    }
    return oracle_bits(oracle_round(y, out_fmt), out_fmt);
}

/* ------------------------------------------------------------------ */
/* Array helpers (for the tests' acceptance checks)                    */
/* ------------------------------------------------------------------ */

void oracle_decode_array(const void* src, int f, int64_t n, double* dst)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = load(src, f, i);
}

/* out = bits of round(src) in format f (plain rounding, no scale). */
void oracle_encode_array(const double* src, int64_t n, int f, void* dst)
{
    for (int64_t i = 0; i < n; ++i) store(dst, f, i, oracle_bits(oracle_round(src[i], f), f));
}

/* out = what the FP8 epilogue emits for the exact values src. */
void oracle_quantize_array(const double* src, int64_t n, float inv_scale, void* dst)
{
    for (int64_t i = 0; i < n; ++i) store(dst, OR_E4M3, i, emit(src[i], OR_E4M3, inv_scale));
}

/* ------------------------------------------------------------------ */
/* RMSNorm ([TEO] section 5.1, Zhang and Sennrich)                     */
/* ------------------------------------------------------------------ */

/* y_i = x_i * r * (w_i + delta), r = 1 / sqrt(mean(x^2) + eps).
 * delta = 0 applies the stored weight directly (Llama); delta = 1 applies
 * 1 + w (Gemma, zero-centred weight).  With no weight ([FRT], weight folded
 * into the next GEMM) y_i = x_i * r.  eps sits inside the root. */
static void rms_row(const double* x, const double* w, int delta, int64_t n, double eps,
                    double* y)
{
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; ++i) y[i] = w ? x[i] * r * (w[i] + (double)delta) : x[i] * r;
}

static int common_ok(int out_fmt, int f, int64_t rows, int64_t n, int weight_offset)
{
    if (!fmt_ok(f) || f == OR_E4M3 || !fmt_ok(out_fmt)) return 0;
    if (out_fmt != f && out_fmt != OR_E4M3) return 0;
    if (rows < 0 || n < 0) return 0;
    if (weight_offset != 0 && weight_offset != 1) return 0;
    return 1;
}

/* out[rows, hidden] = RMSNorm(x) in out_fmt; pre (nullable) receives the exact
 * value before the output rounding. */
int oracle_rmsnorm(void* out, int out_fmt, double* pre, const void* x, const void* w, int f,
                   int64_t rows, int64_t hidden, float eps, int weight_offset, float inv_scale)
{
    if (!common_ok(out_fmt, f, rows, hidden, weight_offset)) return 1;
    double* xr = malloc(sizeof(double) * (size_t)(hidden + 1));
    double* wr = malloc(sizeof(double) * (size_t)(hidden + 1));
    double* yr = malloc(sizeof(double) * (size_t)(hidden + 1));
    if (!xr || !wr || !yr) { free(xr); free(wr); free(yr); return 2; }
    if (w) for (int64_t i = 0; i < hidden; ++i) wr[i] = load(w, f, i);
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t i = 0; i < hidden; ++i) xr[i] = load(x, f, t * hidden + i);
        rms_row(xr, w ? wr : NULL, weight_offset, hidden, (double)eps, yr);
        for (int64_t i = 0; i < hidden; ++i) {
            store(out, out_fmt, t * hidden + i, emit(yr[i], out_fmt, inv_scale));
            if (pre) pre[t * hidden + i] = yr[i];
        }
    }
    free(xr); free(wr); free(yr);
    return 0;
}

/* Fused residual step ([TEO] R1 and section 5.2): the residual stream becomes
 * round(x + r), where the sum is taken the way an eager framework adds two
 * tensors of this dtype (widen both to binary32, add in binary32, round once
 * to the dtype), so it is bit-identical to eager addition; the norm is then
 * taken of that rounded sum.  residual_out may equal residual. */
int oracle_add_rmsnorm(void* out, int out_fmt, double* pre, void* residual_out, const void* x,
                       const void* residual, const void* w, int f, int64_t rows, int64_t hidden,
                       float eps, int weight_offset, float inv_scale)
{
    if (!common_ok(out_fmt, f, rows, hidden, weight_offset)) return 1;
    double* sr = malloc(sizeof(double) * (size_t)(hidden + 1));
    double* wr = malloc(sizeof(double) * (size_t)(hidden + 1));
    double* yr = malloc(sizeof(double) * (size_t)(hidden + 1));
    if (!sr || !wr || !yr) { free(sr); free(wr); free(yr); return 2; }
    if (w) for (int64_t i = 0; i < hidden; ++i) wr[i] = load(w, f, i);
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t i = 0; i < hidden; ++i) {
            volatile float a = (float)load(x, f, t * hidden + i);
            volatile float b = (float)load(residual, f, t * hidden + i);
            volatile float s32 = a + b;
            double s = oracle_round((double)s32, f);
            store(residual_out, f, t * hidden + i, oracle_bits(s, f));
            sr[i] = s;
        }
        rms_row(sr, w ? wr : NULL, weight_offset, hidden, (double)eps, yr);
        for (int64_t i = 0; i < hidden; ++i) {
            store(out, out_fmt, t * hidden + i, emit(yr[i], out_fmt, inv_scale));
            if (pre) pre[t * hidden + i] = yr[i];
        }
    }
    free(sr); free(wr); free(yr);
    return 0;
}

/* ------------------------------------------------------------------ */
/* LayerNorm ([FRT] siglip_layernorm_1read; Ba, Kiros and Hinton)      */
/* ------------------------------------------------------------------ */

/* y_i = (x_i - mu) / sqrt(var + eps) * gamma_i + beta_i with mu the row mean
 * and var = mean((x - mu)^2) (biased).  gamma / beta may be absent (1 / 0).
 * mag (nullable) receives the error scale of each output, the magnitudes of
 * the terms whose roundings enter it: (|x_i| + |mu| + mean|x|) r |gamma_i| +
 * |beta_i| (a float sum of the row errs in proportion to mean|x|). */
int oracle_layernorm(void* out, int out_fmt, double* pre, double* mag, const void* x,
                     const void* gamma, const void* beta, int f, int64_t rows, int64_t hidden,
                     float eps, float inv_scale)
{
    if (!common_ok(out_fmt, f, rows, hidden, 0)) return 1;
    double* xr = malloc(sizeof(double) * (size_t)(hidden + 1));
    if (!xr) return 2;
    for (int64_t t = 0; t < rows; ++t) {
        double mu = 0.0, mean_abs = 0.0;
        for (int64_t i = 0; i < hidden; ++i) {
            xr[i] = load(x, f, t * hidden + i);
            mu += xr[i];
            mean_abs += fabs(xr[i]);
        }
        mu /= (double)hidden;
        mean_abs /= (double)hidden;
        double var = 0.0;
        for (int64_t i = 0; i < hidden; ++i) var += (xr[i] - mu) * (xr[i] - mu);
        var /= (double)hidden;
        double r = 1.0 / sqrt(var + (double)eps);
        for (int64_t i = 0; i < hidden; ++i) {
            double g = gamma ? load(gamma, f, i) : 1.0;
            double b = beta ? load(beta, f, i) : 0.0;
            double y = (xr[i] - mu) * r * g + b;
            store(out, out_fmt, t * hidden + i, emit(y, out_fmt, inv_scale));
            if (pre) pre[t * hidden + i] = y;
            if (mag) mag[t * hidden + i] = (fabs(xr[i]) + fabs(mu) + mean_abs) * r * fabs(g) + fabs(b);
        }
    }
    free(xr);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Static FP8 quantization ([FRT] quantize_fp8_static)                 */
/* ------------------------------------------------------------------ */

/* out_i = E4M3(fl32(x_i) * inv_scale) with the epilogue's fp32 decision and
 * saturation: the standalone form of the fused static-scale epilogue. */
int oracle_quantize_static(void* out, const void* x, int f, int64_t n, float inv_scale)
{
    if (!fmt_ok(f) || f == OR_E4M3 || n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) store(out, OR_E4M3, i, emit(load(x, f, i), OR_E4M3, inv_scale));
    return 0;
}

/* ------------------------------------------------------------------ */
/* Gated activations ([TEO] section 5.1; Shazeer GLU variants)         */
/* ------------------------------------------------------------------ */

/* silu(g) = g / (1 + e^-g). */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* gelu_tanh(g) = 0.5 g (1 + tanh(z)), z = sqrt(2/pi) (g + 0.044715 g^3)
 * (Hendrycks and Gimpel, tanh approximation).  Evaluated through the exact
 * identity 0.5 (1 + tanh z) = 1 / (1 + e^(-2z)), which avoids the
 * cancellation of 1 + tanh z for large negative z; the tests check the
 * identity against the tanh form where that form is well conditioned. */
static double gelu_tanh(double g)
{
    double z = sqrt(2.0 / OR_PI) * (g + 0.044715 * g * g * g);
    return g / (1.0 + exp(-2.0 * z));
}

/* out[rows, d] = act(g) * u with [g || u] = gate_up[rows, 2d] (gate first). */
int oracle_glu_act(void* out, int out_fmt, double* pre, const void* gate_up, int f, int64_t rows,
                   int64_t d, int act, float inv_scale)
{
    if (!common_ok(out_fmt, f, rows, d, 0)) return 1;
    if (act != OR_SILU && act != OR_GELU_TANH) return 1;
    for (int64_t t = 0; t < rows; ++t) {
        for (int64_t i = 0; i < d; ++i) {
            double g = load(gate_up, f, t * 2 * d + i);
            double u = load(gate_up, f, t * 2 * d + d + i);
            double y = (act == OR_SILU ? silu(g) : gelu_tanh(g)) * u;
            store(out, out_fmt, t * d + i, emit(y, out_fmt, inv_scale));
            if (pre) pre[t * d + i] = y;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Rotary embedding and the fused QK prologue                          */
/* ------------------------------------------------------------------ */

/* Test hook for the strength control of [NIN] "Output": a factor applied to
 * the rotation.  It is 1 except inside the test that plants the mistake. */
static double g_rot_scale = 1.0;

void oracle_set_rotation_scale(double s) { g_rot_scale = s; }

/* Index of the two members of rotary pair j ([TEO] section 5.1):
 * rotate-half (GPT-NeoX) pairs (j, j + rho/2); interleaved (GPT-J) pairs
 * (2j, 2j + 1).  Pair j uses entry j of the cached cos and sin rows. */
static void pair_index(int layout, int rho, int j, int* ia, int* ib)
{
    if (layout == OR_INTERLEAVED) { *ia = 2 * j; *ib = 2 * j + 1; }
    else { *ia = j; *ib = j + rho / 2; }
}

/* The position gate of [TEO] R5 and section 5.4: a token rotates only when its
 * position indexes a row of the cache. */
static int in_cache(int64_t p, int64_t cache_len) { return p >= 0 && p < cache_len; }

/* One rotation of pair (a, b) by the cached (c, s) (RoFormer):
 * a' = a c - b s, b' = b c + a s. */
static void rotate(double a, double b, double c, double s, double* ra, double* rb)
{
    c *= g_rot_scale;
    s *= g_rot_scale;
    *ra = a * c - b * s;
    *rb = b * c + a * s;
}

/* Standalone rotary embedding ([TEO] section 5.1, the rotary operator) of
 * heads x[tokens, heads, D] (values in format f): rotate the first rho
 * channels of every head of token t by cos/sin row positions[t] and round
 * once to out_fmt (or take the FP8 epilogue).  A token whose position is
 * outside the cache is copied unchanged. */
int oracle_rope(void* out, int out_fmt, double* pre, double* mag, const void* x, int f,
                int64_t tokens, int heads, int head_dim, int rotary_dim, int layout,
                const int64_t* positions, const float* cos_cache, const float* sin_cache,
                int64_t cache_len, float inv_scale)
{
    if (!common_ok(out_fmt, f, tokens, head_dim, 0)) return 1;
    if (rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return 1;
    int half = rotary_dim / 2;
    double* y = malloc(sizeof(double) * (size_t)(head_dim + 1));
    if (!y) return 2;
    for (int64_t t = 0; t < tokens; ++t) {
        int64_t p = positions ? positions[t] : -1;
        int rot = rotary_dim > 0 && in_cache(p, cache_len);
        for (int h = 0; h < heads; ++h) {
            int64_t base = (t * heads + h) * head_dim;
            for (int i = 0; i < head_dim; ++i) y[i] = load(x, f, base + i);
            if (rot) {
                for (int j = 0; j < half; ++j) {
                    int ia, ib;
                    pair_index(layout, rotary_dim, j, &ia, &ib);
                    double ra, rb;
                    rotate(y[ia], y[ib], (double)cos_cache[p * half + j],
                           (double)sin_cache[p * half + j], &ra, &rb);
                    y[ia] = ra;
                    y[ib] = rb;
                }
            }
            for (int i = 0; i < head_dim; ++i) {
                store(out, out_fmt, base + i, emit(y[i], out_fmt, inv_scale));
                if (pre) pre[base + i] = y[i];
                if (mag) {
                    double m2 = fabs(y[i]);
                    if (rot && i < rotary_dim) {
                        int partner = layout == OR_INTERLEAVED ? (i ^ 1)
                                                               : (i < half ? i + half : i - half);
                        m2 = sqrt(y[i] * y[i] + y[partner] * y[partner]);
                    }
                    mag[base + i] = m2;
                }
            }
        }
    }
    free(y);
    return 0;
}

/* Diagnostics of one output element of the QK prologue, for the tests'
 * tie policy (GPU and oracle round in different precisions):
 *   pre  the exact value whose output rounding (or FP8 epilogue) gives out;
 *   lo, hi  the smallest and largest such value over every combination of
 *        the intermediate roundings of the element (and of its rotation
 *        partner) that were decided within the near-tie band: each near-tie
 *        member may have gone to either neighbour;
 *   mag  the magnitude that sets the error scale: the pair norm for a
 *        rotated channel, |pre| otherwise. */
typedef struct {
    double* pre;
    double* lo;
    double* hi;
    double* mag;
} qk_diag;

/* True when the rounding of v to f is decided within a relative band eta of
 * a rounding boundary; *other receives the neighbour on the far side. */
static int near_tie(double v, int f, double eta, double* other)
{
    double r = oracle_round(v, f);
    double lo = oracle_round(v - eta * fabs(v), f);
    double hi = oracle_round(v + eta * fabs(v), f);
    if (lo == hi) return 0;
    *other = (r == lo) ? hi : lo;
    return 1;
}

/* Test hook: the near-tie decision of the tie policy for one value v (1 when
 * its rounding to f is decided within the relative band eta; *other then
 * receives the neighbour on the far side of the boundary, else v's rounding). */
int oracle_near_tie(double v, int f, double eta, double* other)
{
    double o = oracle_round(v, f);
    int t = near_tie(v, f, eta, &o);
    if (other) *other = o;
    return t;
}

/* `heads` heads of D elements read from x at element offset x_off and
 * written to out (and the diagnostics) at element offset out_off; without
 * `normalize` the head passes through unnormalized (standalone rotation, or
 * the value heads of the fused QKV op). */
static void qk_heads(void* out, int out_fmt, qk_diag dg, const void* x, int64_t x_off,
                     int64_t out_off, const double* w, int f, int heads, int D, int rho,
                     int layout, int rot, int64_t p, const float* cs, const float* sn, float eps,
                     int delta, float inv_scale, double eta, int unrounded, int normalize,
                     double* xr, double* n, double* m, double* malt, int* tie, double* y,
                     double* ylo, double* yhi)
{
    int half = rho / 2;
    for (int h = 0; h < heads; ++h) {
        int64_t xb = x_off + (int64_t)h * D;
        int64_t base = out_off + (int64_t)h * D;
        for (int i = 0; i < D; ++i) xr[i] = load(x, f, xb + i);
        /* per-head RMSNorm with the head's own weight, then rounding to the
         * input dtype before the rotation ([TEO] section 5.4; [NIN]
         * "Implementation": the rotation consumes the rounded value). */
        if (normalize) rms_row(xr, w, delta, D, (double)eps, n);
        else for (int i = 0; i < D; ++i) n[i] = xr[i];
        for (int i = 0; i < D; ++i) {
            m[i] = oracle_round(n[i], f);
            malt[i] = m[i];
            tie[i] = (f != OR_F32) && near_tie(n[i], f, eta, &malt[i]);
            y[i] = m[i];
            ylo[i] = fmin(m[i], malt[i]);
            yhi[i] = fmax(m[i], malt[i]);
        }
        if (rot && unrounded) {
            /* variant of the [NIN] review, item 1: the rotation consumes the
             * normalized value itself, and the output is rounded once */
            for (int j = 0; j < half; ++j) {
                int ia, ib;
                pair_index(layout, rho, j, &ia, &ib);
                double c = (double)cs[p * half + j], s = (double)sn[p * half + j];
                rotate(n[ia], n[ib], c, s, &y[ia], &y[ib]);
                ylo[ia] = yhi[ia] = y[ia];
                ylo[ib] = yhi[ib] = y[ib];
            }
        } else if (rot) {
            for (int j = 0; j < half; ++j) {
                int ia, ib;
                pair_index(layout, rho, j, &ia, &ib);
                double c = (double)cs[p * half + j], s = (double)sn[p * half + j];
                rotate(m[ia], m[ib], c, s, &y[ia], &y[ib]);
                /* bounds over every near-tie neighbour combination of the pair */
                const double ca[2] = {m[ia], malt[ia]}, cb[2] = {m[ib], malt[ib]};
                double alo = INFINITY, ahi = -INFINITY, blo = INFINITY, bhi = -INFINITY;
                for (int u = 0; u < (tie[ia] ? 2 : 1); ++u) {
                    for (int v = 0; v < (tie[ib] ? 2 : 1); ++v) {
                        double ra, rb;
                        rotate(ca[u], cb[v], c, s, &ra, &rb);
                        alo = fmin(alo, ra);
                        ahi = fmax(ahi, ra);
                        blo = fmin(blo, rb);
                        bhi = fmax(bhi, rb);
                    }
                }
                ylo[ia] = alo;
                yhi[ia] = ahi;
                ylo[ib] = blo;
                yhi[ib] = bhi;
            }
        }
        for (int i = 0; i < D; ++i) {
            int rotated = rot && i < rho;
            int partner = i;
            if (rotated) {
                if (layout == OR_INTERLEAVED) partner = i ^ 1;
                else partner = i < half ? i + half : i - half;
            }
            store(out, out_fmt, base + i, emit(y[i], out_fmt, inv_scale));
            double pre, lo, hi, mag;
            if (rotated) {
                pre = y[i];
                lo = ylo[i];
                hi = yhi[i];
                mag = sqrt(y[i] * y[i] + y[partner] * y[partner]);
            } else if (out_fmt == OR_E4M3) {
                /* the epilogue quantizes the rounded m (or its near-tie neighbour) */
                pre = m[i];
                lo = ylo[i];
                hi = yhi[i];
                mag = fabs(pre);
            } else {
                /* the output is the rounding of n itself */
                pre = lo = hi = n[i];
                mag = fabs(pre);
            }
            if (dg.pre) dg.pre[base + i] = pre;
            if (dg.lo) dg.lo[base + i] = lo;
            if (dg.hi) dg.hi[base + i] = hi;
            if (dg.mag) dg.mag[base + i] = mag;
        }
    }
}

/* Fused per-head QK-RMSNorm + RoPE ([TEO] section 5.4, [NIN]
 * "Implementation").  q[tokens, q_heads, D] with weight wq and
 * k[tokens, k_heads, D] with weight wk (each of length D) are normalized per
 * head, rounded to the input dtype, and the first rotary_dim channels of every
 * head of token t are rotated by cos/sin row positions[t] of the cache
 * (cache_len rows of rotary_dim/2 fp32 entries each).  Channels at or past
 * rotary_dim carry the rounded normalized value.  A token whose position is
 * negative or at least cache_len is normalized but not rotated and reads no
 * cache row.  eta is the relative band of the near-tie diagnostics. */
int oracle_qk_norm_rope(void* q_out, void* k_out, int out_fmt, double* q_pre, double* k_pre,
                        double* q_lo, double* k_lo, double* q_hi, double* k_hi,
                        double* q_mag, double* k_mag,
                        const void* q, const void* k, const void* wq, const void* wk, int f,
                        int64_t tokens, int q_heads, int k_heads, int head_dim, int rotary_dim,
                        int layout, const int64_t* positions, const float* cos_cache,
                        const float* sin_cache, int64_t cache_len, float eps, int weight_offset,
                        float inv_scale, double eta, int unrounded)
{
    if (!common_ok(out_fmt, f, tokens, head_dim, weight_offset)) return 1;
    if (q_heads < 0 || k_heads < 0 || head_dim <= 0) return 1;
    if (rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return 1;
    if (layout != OR_ROTATE_HALF && layout != OR_INTERLEAVED) return 1;
    size_t nd = (size_t)head_dim + 1;
    double* wqr = malloc(sizeof(double) * nd);
    double* wkr = malloc(sizeof(double) * nd);
    double* buf = malloc(sizeof(double) * nd * 8);
    int* tie = malloc(sizeof(int) * nd);
    if (!wqr || !wkr || !buf || !tie) { free(wqr); free(wkr); free(buf); free(tie); return 2; }
    for (int i = 0; i < head_dim; ++i) {
        wqr[i] = wq ? load(wq, f, i) : 1.0;
        wkr[i] = wk ? load(wk, f, i) : 1.0;
    }
    qk_diag dq = {q_pre, q_lo, q_hi, q_mag}, dk = {k_pre, k_lo, k_hi, k_mag};
    for (int64_t t = 0; t < tokens; ++t) {
        int64_t p = positions ? positions[t] : -1;
        int rot = rotary_dim > 0 && in_cache(p, cache_len);
        const int64_t qo = t * q_heads * (int64_t)head_dim, ko = t * k_heads * (int64_t)head_dim;
        qk_heads(q_out, out_fmt, dq, q, qo, qo, wq ? wqr : NULL, f, q_heads, head_dim, rotary_dim,
                 layout, rot, p, cos_cache, sin_cache, eps, weight_offset, inv_scale, eta,
                 unrounded, 1, buf, buf + nd, buf + 2 * nd, buf + 3 * nd, tie, buf + 4 * nd,
                 buf + 5 * nd, buf + 6 * nd);
        qk_heads(k_out, out_fmt, dk, k, ko, ko, wk ? wkr : NULL, f, k_heads, head_dim, rotary_dim,
                 layout, rot, p, cos_cache, sin_cache, eps, weight_offset, inv_scale, eta,
                 unrounded, 1, buf, buf + nd, buf + 2 * nd, buf + 3 * nd, tie, buf + 4 * nd,
                 buf + 5 * nd, buf + 6 * nd);
    }
    free(wqr); free(wkr); free(buf); free(tie);
    return 0;
}

/* Fused QKV split + QK-norm + RoPE + KV-cache write ([FRT]
 * qkv_split_rope_kvcache; [TEO] roadmap item 4).  Row t of qkv [T,
 * (Hq + 2 Hk) D] holds Hq query, Hk key and Hk value heads.  Query heads get
 * the prologue (per-head RMSNorm if `normalize`, rounding to the dtype, the
 * rotation) into q_out[t]; key heads the same into k_cache[slots[t]]; value
 * heads are copied into v_cache[slots[t]].  Caches are [num_slots, Hk, D]; a
 * slot outside [0, num_slots) writes no cache row (the other rows keep their
 * contents).  Diagnostics are laid out like q_out and k_cache. */
int oracle_qkv_rope_cache(void* q_out, void* k_cache, void* v_cache, double* q_pre, double* q_lo,
                          double* q_hi, double* q_mag, double* k_pre, double* k_lo, double* k_hi,
                          double* k_mag, const void* qkv, const void* wq, const void* wk, int f,
                          int64_t tokens, int q_heads, int kv_heads, int head_dim, int rotary_dim,
                          int layout, const int64_t* positions, const float* cos_cache,
                          const float* sin_cache, int64_t cache_len, const int64_t* slots,
                          int64_t num_slots, float eps, int weight_offset, int normalize,
                          double eta)
{
    if (!common_ok(f, f, tokens, head_dim, weight_offset)) return 1;
    if (q_heads < 1 || kv_heads < 0 || head_dim <= 0 || num_slots < 0) return 1;
    if (rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return 1;
    if (layout != OR_ROTATE_HALF && layout != OR_INTERLEAVED) return 1;
    size_t nd = (size_t)head_dim + 1;
    double* wqr = malloc(sizeof(double) * nd);
    double* wkr = malloc(sizeof(double) * nd);
    double* buf = malloc(sizeof(double) * nd * 8);
    int* tie = malloc(sizeof(int) * nd);
    if (!wqr || !wkr || !buf || !tie) { free(wqr); free(wkr); free(buf); free(tie); return 2; }
    for (int i = 0; i < head_dim; ++i) {
        wqr[i] = wq ? load(wq, f, i) : 1.0;
        wkr[i] = wk ? load(wk, f, i) : 1.0;
    }
    const int64_t row = (int64_t)(q_heads + 2 * kv_heads) * head_dim;
    qk_diag dq = {q_pre, q_lo, q_hi, q_mag}, dk = {k_pre, k_lo, k_hi, k_mag}, dv = {0, 0, 0, 0};
    for (int64_t t = 0; t < tokens; ++t) {
        int64_t p = positions ? positions[t] : -1;
        int rot = rotary_dim > 0 && in_cache(p, cache_len);
        qk_heads(q_out, f, dq, qkv, t * row, t * q_heads * (int64_t)head_dim, wq ? wqr : NULL, f,
                 q_heads, head_dim, rotary_dim, layout, rot, p, cos_cache, sin_cache, eps,
                 weight_offset, 1.0f, eta, 0, normalize, buf, buf + nd, buf + 2 * nd,
                 buf + 3 * nd, tie, buf + 4 * nd, buf + 5 * nd, buf + 6 * nd);
        int64_t sl = slots ? slots[t] : -1;
        if (kv_heads == 0 || sl < 0 || sl >= num_slots) continue;
        const int64_t co = sl * kv_heads * (int64_t)head_dim;
        qk_heads(k_cache, f, dk, qkv, t * row + (int64_t)q_heads * head_dim, co,
                 wk ? wkr : NULL, f, kv_heads, head_dim, rotary_dim, layout, rot, p, cos_cache,
                 sin_cache, eps, weight_offset, 1.0f, eta, 0, normalize, buf, buf + nd,
                 buf + 2 * nd, buf + 3 * nd, tie, buf + 4 * nd, buf + 5 * nd, buf + 6 * nd);
        qk_heads(v_cache, f, dv, qkv, t * row + (int64_t)(q_heads + kv_heads) * head_dim, co,
                 NULL, f, kv_heads, head_dim, 0, layout, 0, -1, NULL, NULL, eps, 0, 1.0f, eta, 0,
                 0, buf, buf + nd, buf + 2 * nd, buf + 3 * nd, tie, buf + 4 * nd, buf + 5 * nd,
                 buf + 6 * nd);
    }
    free(wqr); free(wkr); free(buf); free(tie);
    return 0;
}

int oracle_version(void) { return 1; }
