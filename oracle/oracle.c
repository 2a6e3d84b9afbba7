/*
 * CSA2 CPU oracle — TEST INFRASTRUCTURE ONLY (see oracle.h for scope and sources).
 *
 * Plain C, fp64 arithmetic, no blocking or fusion: each function restates one
 * step of the method in the order the pages give it. Format encoders are
 * brute-force nearest-value searches over the format's code table, which is the
 * format definition written out (round to nearest, ties to the even code).
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Number formats                                                             */
/* ------------------------------------------------------------------------- */

double orc_e2m1_value(int code) {
    /* 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent field
     * 0 is subnormal (0 or 0.5). No inf/NaN. */
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double orc_e4m3_value(int code) {
    /* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field
     * 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities. */
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest value among codes [0, n_codes) of a non-negative ascending table,
 * ties to the even code. */
static int nearest_code(double a, int n_codes, double (*value)(int)) {
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < n_codes; ++c) {
        double d = fabs(value(c) - a);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1))) {
            bd = d;
            best = c;
        }
    }
    return best;
}

int orc_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    double a = fabs((double)x);
    if (a > 448.0) a = 448.0; /* satfinite */
    int c = nearest_code(a, 127, orc_e4m3_value); /* 0x00..0x7E: finite, >= 0 */
    return c | (signbit(x) ? 0x80 : 0);
}

int orc_e2m1_encode(float x) {
    if (isnan(x)) return 0;
    double a = fabs((double)x);
    if (a > 6.0) a = 6.0; /* satfinite */
    int c = nearest_code(a, 8, orc_e2m1_value);
    return c | (signbit(x) ? 0x8 : 0);
}

void orc_nvfp4_quantize(const float* x, int64_t n_groups, uint8_t* vals, uint8_t* scales) {
    for (int64_t g = 0; g < n_groups; ++g) {
        const float* xg = x + g * 16;
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(xg[i]);
            if (a > amax) amax = a;
        }
        /* s = fl32(amax / 6): fp64 division then one rounding to fp32 equals
         * the correctly rounded fp32 quotient (53 >= 2*24 + 2). */
        float s = (float)((double)amax / 6.0);
        int sc = orc_e4m3_encode(s);
        double S = orc_e4m3_value(sc);
        scales[g] = (uint8_t)sc;
        uint8_t* vg = vals + g * 8;
        memset(vg, 0, 8);
        if (S == 0.0) continue; /* zero scale: all codes 0 */
        for (int i = 0; i < 16; ++i) {
            float y = (float)((double)xg[i] / S); /* fl32(x_i / S) */
            int code = orc_e2m1_encode(y);
            vg[i >> 1] |= (uint8_t)((i & 1) ? (code << 4) : code);
        }
    }
}

double orc_nvfp4_value(const uint8_t* vals, const uint8_t* scales, int64_t i) {
    int byte = vals[i >> 1];
    int code = (i & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_value(code) * orc_e4m3_value(scales[i >> 4]);
}

/* ------------------------------------------------------------------------- */
/* Compressor                                                                 */
/* ------------------------------------------------------------------------- */

float orc_pool(float kv0, float kv1, float g0, float g1) {
    /* alpha = softmax over the pair of the gate logits, per channel. */
    double m = fmax((double)g0, (double)g1);
    double e0 = exp((double)g0 - m), e1 = exp((double)g1 - m);
    return (float)((e0 * kv0 + e1 * kv1) / (e0 + e1));
}

int64_t orc_compress_append(int64_t T, int n_new, int D, int W,
                            const float* kv_new, const float* g_new,
                            float* pend_kv, float* pend_g,
                            uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                            uint8_t* win_u8, float* win_f32) {
    return orc_compress_append_ratio(T, n_new, D, W, 2, kv_new, g_new, pend_kv, pend_g,
                                     comp_vals, comp_scales, comp_f32, win_u8, win_f32);
}

int64_t orc_compress_append_ratio(int64_t T, int n_new, int D, int W, int ratio,
                                  const float* kv_new, const float* g_new,
                                  float* pend_kv, float* pend_g,
                                  uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                                  uint8_t* win_u8, float* win_f32) {
    return orc_compress_append_rope(T, n_new, D, W, ratio, NULL, kv_new, g_new, pend_kv, pend_g,
                                    comp_vals, comp_scales, comp_f32, win_u8, win_f32);
}

/* ------------------------------------------------------------------------- */
/* Rotary position embedding of the compressed KV (RoFormer rotation, YaRN    */
/* NTK-by-parts frequencies)                                                  */
/* ------------------------------------------------------------------------- */

void orc_rope_freqs(const orc_rope* r, double* theta) {
    const double two_pi = 2.0 * acos(-1.0);
    for (int i = 0; i < r->dim / 2; ++i) {
        double th = pow(r->base, -2.0 * i / r->dim); /* RoFormer frequency of pair i */
        double wavelength = two_pi / th;
        double rotations = r->orig_len / wavelength; /* turns over the original context */
        double gamma;
        if (rotations < r->beta_slow)
            gamma = 0.0; /* long wavelength: interpolate */
        else if (rotations > r->beta_fast)
            gamma = 1.0; /* short wavelength: keep */
        else
            gamma = (rotations - r->beta_slow) / (r->beta_fast - r->beta_slow);
        theta[i] = (1.0 - gamma) * th / r->factor + gamma * th;
    }
}

void orc_rope_rotate(float* x, int D, int64_t pos, const orc_rope* r) {
    if (!r || r->dim <= 0) return;
    double* theta = (double*)malloc(sizeof(double) * (size_t)(r->dim / 2));
    orc_rope_freqs(r, theta);
    float* part = x + (D - r->dim);
    for (int i = 0; i < r->dim / 2; ++i) {
        double angle = (double)pos * theta[i];
        double c = cos(angle), s = sin(angle);
        double a = part[2 * i], b = part[2 * i + 1];
        part[2 * i] = (float)(a * c - b * s);
        part[2 * i + 1] = (float)(a * s + b * c);
    }
    free(theta);
}

void orc_compress_row(int D, int ratio, int64_t j, const float* kv0, const float* kv1,
                      const float* g0, const float* g1, const orc_rope* rope,
                      uint8_t* vals, uint8_t* scales, float* f32) {
    float* row = (float*)malloc(sizeof(float) * (size_t)D);
    for (int d = 0; d < D; ++d) row[d] = ratio == 1 ? kv0[d] : orc_pool(kv0[d], kv1[d], g0[d], g1[d]);
    orc_rope_rotate(row, D, (int64_t)ratio * j, rope); /* raw position of the pair's first token */
    if (f32)
        memcpy(f32, row, sizeof(float) * (size_t)D);
    else
        orc_nvfp4_quantize(row, D / 16, vals, scales);
    free(row);
}

int64_t orc_compress_append_rope(int64_t T, int n_new, int D, int W, int ratio,
                                 const orc_rope* rope, const float* kv_new, const float* g_new,
                                 float* pend_kv, float* pend_g,
                                 uint8_t* comp_vals, uint8_t* comp_scales, float* comp_f32,
                                 uint8_t* win_u8, float* win_f32) {
    int has_comp = (comp_vals != NULL) || (comp_f32 != NULL);
    for (int i = 0; i < n_new; ++i) {
        int64_t p = T + i; /* raw position of this token */
        const float* kv = kv_new + (int64_t)i * D;
        const float* g = g_new ? g_new + (int64_t)i * D : NULL;
        int64_t slot = p % W;
        if (win_u8)
            for (int d = 0; d < D; ++d) win_u8[slot * D + d] = (uint8_t)orc_e4m3_encode(kv[d]);
        if (win_f32)
            for (int d = 0; d < D; ++d) win_f32[slot * D + d] = kv[d];
        if (!has_comp) continue;
        int64_t j = p / ratio; /* ratio 1 (1:1 layer): raw token p is compressed row p */
        if (ratio == 2 && (p & 1) == 0) { /* first token of a pair: wait for its partner */
            memcpy(pend_kv, kv, sizeof(float) * (size_t)D);
            memcpy(pend_g, g, sizeof(float) * (size_t)D);
            continue;
        }
        orc_compress_row(D, ratio, j, ratio == 1 ? kv : pend_kv, kv, pend_g, g, rope,
                         comp_f32 ? NULL : comp_vals + j * (D / 2),
                         comp_f32 ? NULL : comp_scales + j * (D / 16),
                         comp_f32 ? comp_f32 + j * D : NULL);
    }
    return T + n_new;
}

/* ------------------------------------------------------------------------- */
/* Indexer                                                                    */
/* ------------------------------------------------------------------------- */

/* Exponent of the least significant set bit of a non-zero double. */
static int lsb_exp(double v) {
    int e;
    double f = frexp(fabs(v), &e);
    uint64_t M = (uint64_t)ldexp(f, 53);
    return e - 53 + __builtin_ctzll(M);
}

/* Smallest lsb exponent over the non-zero entries of v[0..n), INT32_MAX if all zero. */
static int min_lsb(const double* v, int n) {
    int m = INT32_MAX;
    for (int i = 0; i < n; ++i)
        if (v[i] != 0.0 && lsb_exp(v[i]) < m) m = lsb_exp(v[i]);
    return m;
}

int64_t orc_index_scores(int Hi, int Di, const uint8_t* q_vals, const uint8_t* q_scales,
                         const float* w, int64_t n_c, const uint8_t* k_vals,
                         const uint8_t* k_scales, float* scores) {
    double* q = (double*)malloc(sizeof(double) * (size_t)Hi * Di);
    double* k = (double*)malloc(sizeof(double) * (size_t)Di);
    int* q_lsb = (int*)malloc(sizeof(int) * (size_t)Hi);
    for (int h = 0; h < Hi; ++h) {
        for (int d = 0; d < Di; ++d)
            q[h * Di + d] = orc_nvfp4_value(q_vals + (int64_t)h * (Di / 2),
                                            q_scales + (int64_t)h * (Di / 16), d);
        q_lsb[h] = min_lsb(q + h * Di, Di);
    }
    int64_t inexact = 0;
    for (int64_t t = 0; t < n_c; ++t) {
        for (int d = 0; d < Di; ++d)
            k[d] = orc_nvfp4_value(k_vals + t * (Di / 2), k_scales + t * (Di / 16), d);
        const int k_lsb = min_lsb(k, Di);
        double s = 0.0, s_bound = 0.0;
        int s_lsb = INT32_MAX, ok = 1;
        for (int h = 0; h < Hi; ++h) {
            double dot = 0.0, d_bound = 0.0;
            for (int d = 0; d < Di; ++d) {
                double p = q[h * Di + d] * k[d];
                dot += p;
                d_bound += fabs(p);
            }
            /* every product is a multiple of 2^(q_lsb + k_lsb); so is every partial sum */
            if (d_bound != 0.0 && d_bound > ldexp(1.0, 24 + q_lsb[h] + k_lsb)) ok = 0;
            double term = (double)w[h] * (dot > 0.0 ? dot : 0.0); /* w_h * ReLU(q_h . k_t) */
            s += term;
            s_bound += fabs(term);
            if (term != 0.0 && lsb_exp(term) < s_lsb) s_lsb = lsb_exp(term);
        }
        if (s_lsb != INT32_MAX && s_bound > ldexp(1.0, 24 + s_lsb)) ok = 0;
        scores[t] = (float)s;
        if (!ok) ++inexact;
    }
    free(q_lsb);
    free(q);
    free(k);
    return inexact;
}

void orc_block_max(const float* scores, int64_t n_c, int blk, float* block_max) {
    int64_t n_b = (n_c + blk - 1) / blk;
    for (int64_t b = 0; b < n_b; ++b) {
        double m = -INFINITY;
        for (int64_t t = b * blk; t < n_c && t < (b + 1) * blk; ++t)
            if (scores[t] > m) m = scores[t];
        block_max[b] = (float)m;
    }
}

/* ------------------------------------------------------------------------- */
/* Two-level selection                                                        */
/* ------------------------------------------------------------------------- */

typedef struct {
    double key;
    int64_t index;
} keyed;

/* Order: key descending, then index ascending. */
static int by_key_desc_index_asc(const void* a, const void* b) {
    const keyed* x = (const keyed*)a;
    const keyed* y = (const keyed*)b;
    if (x->key > y->key) return -1;
    if (x->key < y->key) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int by_index_asc(const void* a, const void* b) {
    const keyed* x = (const keyed*)a;
    const keyed* y = (const keyed*)b;
    return (x->index > y->index) - (x->index < y->index);
}

int orc_select(const float* scores, int64_t n_c, int blk, int Kb, int Kp, int32_t* idx) {
    for (int i = 0; i < Kp; ++i) idx[i] = -1;
    if (n_c <= 0) return 0;
    int64_t n_b = (n_c + blk - 1) / blk;
    float* bm = (float*)malloc(sizeof(float) * (size_t)n_b);
    orc_block_max(scores, n_c, blk, bm);
    unsigned char* keep = (unsigned char*)calloc((size_t)n_b, 1);
    if (n_b <= Kb) {
        memset(keep, 1, (size_t)n_b);
    } else {
        int64_t newest = (n_c - 1) / blk; /* block of the newest compressed position */
        keyed* order = (keyed*)malloc(sizeof(keyed) * (size_t)n_b);
        int64_t n = 0;
        for (int64_t b = 0; b < n_b; ++b)
            if (b != newest) {
                order[n].key = bm[b];
                order[n].index = b;
                ++n;
            }
        qsort(order, (size_t)n, sizeof(keyed), by_key_desc_index_asc);
        for (int64_t i = 0; i < Kb - 1; ++i) keep[order[i].index] = 1;
        keep[newest] = 1;
        free(order);
    }
    keyed* cand = (keyed*)malloc(sizeof(keyed) * (size_t)n_c);
    int64_t n = 0;
    for (int64_t t = 0; t < n_c; ++t)
        if (keep[t / blk]) {
            cand[n].key = scores[t];
            cand[n].index = t;
            ++n;
        }
    qsort(cand, (size_t)n, sizeof(keyed), by_key_desc_index_asc);
    int64_t m = n < Kp ? n : Kp;
    qsort(cand, (size_t)m, sizeof(keyed), by_index_asc);
    for (int64_t i = 0; i < m; ++i) idx[i] = (int32_t)cand[i].index;
    free(cand);
    free(keep);
    free(bm);
    return (int)m;
}

/* ------------------------------------------------------------------------- */
/* sparse attention with sink                                                 */
/* ------------------------------------------------------------------------- */

int orc_sparse_attn(int H, int D, const double* q, const double* sink, double scale,
                    int64_t T, int W, const uint8_t* win_u8, const float* win_f32,
                    const uint8_t* comp_vals, const uint8_t* comp_scales, const float* comp_f32,
                    const int32_t* idx, int n_idx, double* out) {
    int64_t n_win = (win_u8 || win_f32) ? (T < W ? T : W) : 0;
    double* rows = (double*)malloc(sizeof(double) * (size_t)(n_win + n_idx + 1) * D);
    int n = 0;
    for (int64_t p = T - n_win; p < T; ++p) { /* window: the newest min(T, W) raw tokens */
        int64_t slot = p % W;
        for (int d = 0; d < D; ++d)
            rows[(int64_t)n * D + d] =
                win_u8 ? orc_e4m3_value(win_u8[slot * D + d]) : (double)win_f32[slot * D + d];
        ++n;
    }
    for (int i = 0; i < n_idx; ++i) { /* selected compressed positions */
        int64_t j = idx[i];
        if (j < 0) continue;
        for (int d = 0; d < D; ++d)
            rows[(int64_t)n * D + d] =
                comp_f32 ? (double)comp_f32[j * D + d]
                         : orc_nvfp4_value(comp_vals + j * (D / 2), comp_scales + j * (D / 16), d);
        ++n;
    }
    double* z = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    for (int h = 0; h < H; ++h) {
        const double* qh = q + (int64_t)h * D;
        double M = sink[h];
        for (int j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qh[d] * rows[(int64_t)j * D + d];
            z[j] = scale * dot;
            if (z[j] > M) M = z[j];
        }
        double* oh = out + (int64_t)h * D;
        for (int d = 0; d < D; ++d) oh[d] = 0.0;
        if (isinf(M) || isnan(M)) continue; /* no finite logit: output 0 */
        double den = exp(sink[h] - M);
        for (int j = 0; j < n; ++j) {
            double p = exp(z[j] - M);
            den += p;
            for (int d = 0; d < D; ++d) oh[d] += p * rows[(int64_t)j * D + d];
        }
        for (int d = 0; d < D; ++d) oh[d] /= den;
    }
    free(z);
    free(rows);
    return n;
}

/* ------------------------------------------------------------------------- */
/* Closed forms                                                               */
/* ------------------------------------------------------------------------- */

int64_t orc_nvfp4_payload_bytes(int64_t n, int D) { return n * D / 2; }
int64_t orc_nvfp4_scale_bytes(int64_t n, int D) { return n * D / 16; }
