/*
 * tq_oracle.c -- the oracle for the rotated, bit-packed KV cache.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: loaded only by tests/, by the smoke check and
 * by the benchmark's CPU-baseline leg.  Independent of the CUDA library (no shared
 * code, header, table or constant).  See tq_oracle.h for the sources and the pins.
 *
 * Packed block layout (the pages fix only the sizes -- 128 values plus one fp16 norm,
 * 0.39 / 0.27 bytes per value, [TQ] "How small does it get" -- so the bit order below
 * is this project's reading, chosen so that a GPU can turn codes into table lookups
 * with whole-word shifts and masks):
 *
 *   bytes [0, 2)   norm, IEEE binary16, little-endian.
 *   bytes [2, 34)  low plane: 8 little-endian 32-bit words W_0..W_7.  Value i
 *                  (0..127): w = i / 16, j = i % 16, r = j / 8, k = j % 8; bits
 *                  4k+2r (code bit 0) and 4k+2r+1 (code bit 1) of W_w.
 *   bytes [34, 50) turbo3 only, high plane: 4 little-endian 32-bit words V_0..V_3.
 *                  Value i: u = i / 32, j = i % 32, p = j / 8, k = j % 8; bit 4k+p
 *                  of V_u holds code bit 2.
 *
 * turbo2 blocks are the first 34 bytes of that layout (norm + low plane).
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* The binary32 value nearest to 1/sqrt(128) = 2^-3.5 (0.08838834764831844...). */
static const float ORACLE_INV_SQRT128 = 0x1.6a09e6p-4f;
#define ORACLE_BLOCK 128

size_t oracle_block_bytes(int type)
{
    if (type != ORACLE_TURBO2 && type != ORACLE_TURBO3) return 0;
    return 2u + (size_t)ORACLE_BLOCK * (size_t)type / 8u;
}

uint64_t oracle_kv_bytes(uint64_t layers, uint64_t kv_heads, uint64_t head_dim,
                         uint64_t ctx, uint64_t bytes_num, uint64_t bytes_den)
{
    /* layers x heads x head_dim x ctx x 2 x bytes/value */
    return layers * kv_heads * head_dim * ctx * 2u * bytes_num / bytes_den;
}

/* ---------------------------------------------------------------- binary16 */

float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);                 /* zero or subnormal */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);    /* (1.m) * 2^(e-15) */
    }
    return (float)(sign ? -v : v);
}

uint16_t oracle_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    double a = fabs((double)f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);   /* rounds past 65504 */
    /* quantum of the binary16 grid at this magnitude */
    int ex;
    double q;
    if (a < 0x1p-14) {
        q = 0x1p-24;
    } else {
        frexp(a, &ex);                      /* a = fr * 2^ex, fr in [0.5, 1) */
        q = ldexp(1.0, ex - 1 - 10);        /* 2^(floor(log2 a) - 10) */
    }
    double mq = a / q;                      /* exact: q is a power of two */
    double fl = floor(mq);
    double fr = mq - fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = fl * q;                      /* rounded magnitude, exact */
    if (r == 0.0) return sign;
    if (r < 0x1p-14) return (uint16_t)(sign | (uint16_t)(r / 0x1p-24));
    frexp(r, &ex);
    int e = ex - 1;                         /* r = 1.m * 2^e */
    uint16_t m = (uint16_t)(r / ldexp(1.0, e - 10) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | m);
}

/* ---------------------------------------------------------------- FWHT */

void oracle_fwht_f32(float *x, int n)
{
    for (int h = 1; h < n; h *= 2) {
        for (int i = 0; i < n; ++i) {
            if (i & h) continue;
            float a = x[i], b = x[i + h];
            x[i] = a + b;
            x[i + h] = a - b;
        }
    }
}

void oracle_fwht_f64(double *x, int n)
{
    for (int h = 1; h < n; h *= 2) {
        for (int i = 0; i < n; ++i) {
            if (i & h) continue;
            double a = x[i], b = x[i + h];
            x[i] = a + b;
            x[i + h] = a - b;
        }
    }
}

/* ---------------------------------------------------------------- codebook */

/* Unnormalised density of one coordinate of a uniform unit vector in R^d:
 * (1 - y^2)^((d-3)/2) on [-1, 1].  The normalising constant cancels in every ratio
 * the Lloyd conditions use. */
typedef struct { double a; int moment; } dens_arg;

static double dens_eval(const dens_arg *p, double y)
{
    double u = 1.0 - y * y;
    if (u <= 0.0) return 0.0;
    double g = (p->a == 0.0) ? 1.0 : pow(u, p->a);
    return p->moment ? y * g : g;
}

/* Composite Gauss-Legendre quadrature: GL_N-point rule on GL_PANELS equal panels.
 * The nodes and weights are the roots of the Legendre polynomial P_N, found by
 * Newton's method from the usual cosine starting guesses (textbook construction). */
#define GL_N 16
#define GL_PANELS 64
static double gl_x[GL_N], gl_w[GL_N];
static int gl_ready = 0;

static void gl_init(void)
{
    const double pi = 3.14159265358979323846;
    for (int i = 0; i < GL_N; ++i) {
        double x = cos(pi * (i + 0.75) / (GL_N + 0.5));
        double dp = 1.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = x;               /* P_0, P_1 */
            for (int n = 2; n <= GL_N; ++n) {      /* Bonnet recursion */
                double p2 = ((2.0 * n - 1.0) * x * p1 - (n - 1.0) * p0) / n;
                p0 = p1;
                p1 = p2;
            }
            dp = GL_N * (x * p1 - p0) / (x * x - 1.0);   /* P_N'(x) */
            double dx = p1 / dp;
            x -= dx;
            if (fabs(dx) < 1e-17) break;
        }
        gl_x[i] = x;
        gl_w[i] = 2.0 / ((1.0 - x * x) * dp * dp);
    }
    gl_ready = 1;
}

static double integrate(const dens_arg *p, double a, double b)
{
    if (b <= a) return 0.0;
    if (!gl_ready) gl_init();
    double total = 0.0;
    double hw = 0.5 * (b - a) / GL_PANELS;
    for (int s = 0; s < GL_PANELS; ++s) {
        double mid = a + (2.0 * s + 1.0) * hw;
        double acc = 0.0;
        for (int i = 0; i < GL_N; ++i) acc += gl_w[i] * dens_eval(p, mid + hw * gl_x[i]);
        total += hw * acc;
    }
    return total;
}

int oracle_codebook(int d, int levels, double *centroids_f64, float *centroids,
                    float *thresholds)
{
    if (d < 3 || levels < 2 || levels > 64) return -1;
    double c[64], cn[64], b[65];
    dens_arg mass = { 0.5 * (d - 3), 0 }, mom = { 0.5 * (d - 3), 1 };
    /* start: evenly spaced centroids over +-2.5 standard deviations, kept in (-1,1) */
    double sd = 1.0 / sqrt((double)d);
    for (int j = 0; j < levels; ++j) {
        double t = -2.5 * sd + 5.0 * sd * (j + 0.5) / levels;
        if (t < -0.999) t = -0.999 + 0.001 * j / levels;
        if (t > 0.999) t = 0.999 - 0.001 * (levels - 1 - j) / levels;
        c[j] = t;
    }
    int it;
    for (it = 1; it <= 200000; ++it) {
        b[0] = -1.0;
        b[levels] = 1.0;
        for (int j = 1; j < levels; ++j) b[j] = 0.5 * (c[j - 1] + c[j]);
        double move = 0.0;
        for (int j = 0; j < levels; ++j) {
            double m0 = integrate(&mass, b[j], b[j + 1]);
            double m1 = integrate(&mom, b[j], b[j + 1]);
            cn[j] = m1 / m0;                  /* centroid condition */
            double dlt = fabs(cn[j] - c[j]);
            if (dlt > move) move = dlt;
        }
        memcpy(c, cn, sizeof(double) * (size_t)levels);
        if (move < 1e-14) break;
    }
    for (int j = 0; j < levels; ++j) {
        if (centroids_f64) centroids_f64[j] = c[j];
        if (centroids) centroids[j] = (float)c[j];
    }
    if (thresholds && centroids)
        for (int j = 0; j + 1 < levels; ++j)
            thresholds[j] = (centroids[j] + centroids[j + 1]) * 0.5f;
    return it;
}

/* ---------------------------------------------------------------- bit layout */

static void put_bit(uint8_t *base, int bit, int v)
{
    if (v) base[bit >> 3] = (uint8_t)(base[bit >> 3] | (1u << (bit & 7)));
}

static int get_bit(const uint8_t *base, int bit)
{
    return (base[bit >> 3] >> (bit & 7)) & 1;
}

/* bit index (within the 32-byte low plane) of code bit 0 of value i */
static int low_plane_bit(int i)
{
    int w = i / 16, j = i % 16, r = j / 8, k = j % 8;
    return 32 * w + 4 * k + 2 * r;
}

/* bit index (within the 16-byte high plane) of code bit 2 of value i */
static int high_plane_bit(int i)
{
    int u = i / 32, j = i % 32, p = j / 8, k = j % 8;
    return 32 * u + 4 * k + p;
}

static void pack_block(int type, uint16_t norm, const uint8_t *codes, uint8_t *out)
{
    memset(out, 0, oracle_block_bytes(type));
    out[0] = (uint8_t)(norm & 0xff);
    out[1] = (uint8_t)(norm >> 8);
    for (int i = 0; i < ORACLE_BLOCK; ++i) {
        int lb = low_plane_bit(i);
        put_bit(out + 2, lb, codes[i] & 1);
        put_bit(out + 2, lb + 1, (codes[i] >> 1) & 1);
        if (type == ORACLE_TURBO3) put_bit(out + 34, high_plane_bit(i), (codes[i] >> 2) & 1);
    }
}

void oracle_unpack_block(int type, const uint8_t *blk, uint8_t *codes, uint16_t *norm_f16)
{
    if (norm_f16) *norm_f16 = (uint16_t)(blk[0] | (blk[1] << 8));
    for (int i = 0; i < ORACLE_BLOCK; ++i) {
        int lb = low_plane_bit(i);
        int c = get_bit(blk + 2, lb) | (get_bit(blk + 2, lb + 1) << 1);
        if (type == ORACLE_TURBO3) c |= get_bit(blk + 34, high_plane_bit(i)) << 2;
        codes[i] = (uint8_t)c;
    }
}

/* ---------------------------------------------------------------- encode / decode */

static int sign_bit(const oracle_variant *var, int i)
{
    return var ? (int)((var->signs[i / 32] >> (i % 32)) & 1u) : 0;
}

void oracle_encode_block_v(int type, const uint16_t *x_f16, const float *thresholds,
                           const float *centroids, const oracle_variant *var, uint8_t *out)
{
    const int levels = 1 << type;
    float x[ORACLE_BLOCK], s[ORACLE_BLOCK], z[ORACLE_BLOCK];
    uint8_t codes[ORACLE_BLOCK];
    for (int i = 0; i < ORACLE_BLOCK; ++i) x[i] = oracle_f16_to_f32(x_f16[i]);

    /* 0. variant: the rotation is W D, so coordinates with a sign bit are negated first
     *    (exact; the norm does not change) */
    for (int i = 0; i < ORACLE_BLOCK; ++i)
        if (sign_bit(var, i)) x[i] = -x[i];

    /* 1. norm: pairwise tree, level by level, element i pairs with i + len/2 */
    for (int i = 0; i < ORACLE_BLOCK; ++i) s[i] = x[i] * x[i];
    for (int len = ORACLE_BLOCK; len > 1; len /= 2)
        for (int i = 0; i < len / 2; ++i) s[i] = s[i] + s[i + len / 2];
    float n = sqrtf(s[0]);

    /* 2. stored norm, saturated to the largest finite binary16 (set in step 5 for the
     *    norm-correcting variant) */
    uint16_t norm16 = oracle_f32_to_f16(n < 65504.0f ? n : 65504.0f);

    /* 3. rotation: unnormalised Walsh-Hadamard butterflies */
    memcpy(z, x, sizeof z);
    oracle_fwht_f32(z, ORACLE_BLOCK);

    /* 4. one scale brings the rotated block to the unit sphere (W/sqrt(128) is
     *    orthonormal, so |W x| / sqrt(128) = n) */
    float k = (n > 0.0f) ? ORACLE_INV_SQRT128 / n : 0.0f;

    /* 5. symmetric Lloyd-Max scalar quantiser: magnitude index against the positive
     *    thresholds t_{L/2} .. t_{L-2}, sign bit picks the half of the codebook */
    for (int i = 0; i < ORACLE_BLOCK; ++i) {
        float y = z[i] * k;
        float a = fabsf(y);
        int m = 0;
        for (int j = levels / 2; j <= levels - 2; ++j)
            if (a > thresholds[j]) ++m;
        codes[i] = (uint8_t)(signbit(y) ? levels / 2 - 1 - m : levels / 2 + m);
    }

    /* 5b. variant: store |x| / |c|, |c| the norm of the centroid vector of the codes
     *     (same pairwise tree as step 1, then an IEEE sqrt and divide), so that the decoded
     *     block keeps the norm of its input up to the fp16 rounding */
    if (var && var->norm_correction) {
        float c2[ORACLE_BLOCK];
        for (int i = 0; i < ORACLE_BLOCK; ++i) c2[i] = centroids[codes[i]] * centroids[codes[i]];
        for (int len = ORACLE_BLOCK; len > 1; len /= 2)
            for (int i = 0; i < len / 2; ++i) c2[i] = c2[i] + c2[i + len / 2];
        float r = n / sqrtf(c2[0]);
        norm16 = oracle_f32_to_f16(r < 65504.0f ? r : 65504.0f);
    }

    /* 6. pack */
    pack_block(type, norm16, codes, out);
}

void oracle_encode_block(int type, const uint16_t *x_f16, const float *thresholds,
                         uint8_t *out)
{
    oracle_encode_block_v(type, x_f16, thresholds, NULL, NULL, out);
}

void oracle_decode_block_v(int type, const uint8_t *blk, const float *centroids,
                           const oracle_variant *var, double *out)
{
    uint8_t codes[ORACLE_BLOCK];
    uint16_t norm16;
    oracle_unpack_block(type, blk, codes, &norm16);
    for (int i = 0; i < ORACLE_BLOCK; ++i) out[i] = (double)centroids[codes[i]];
    oracle_fwht_f64(out, ORACLE_BLOCK);     /* W is its own inverse up to 1/128 */
    double sc = (double)oracle_f16_to_f32(norm16) / sqrt(128.0);
    for (int i = 0; i < ORACLE_BLOCK; ++i) out[i] *= sign_bit(var, i) ? -sc : sc;   /* D W c */
}

void oracle_decode_block(int type, const uint8_t *blk, const float *centroids, double *out)
{
    oracle_decode_block_v(type, blk, centroids, NULL, out);
}

void oracle_encode_rows(int type, const uint16_t *src, int64_t n_tokens,
                        int n_kv_heads, int head_dim, int64_t src_stride,
                        const float *thresholds, uint8_t *dst)
{
    oracle_encode_rows_v(type, src, n_tokens, n_kv_heads, head_dim, src_stride, thresholds,
                         NULL, NULL, dst);
}

void oracle_encode_rows_v(int type, const uint16_t *src, int64_t n_tokens,
                          int n_kv_heads, int head_dim, int64_t src_stride,
                          const float *thresholds, const float *centroids,
                          const oracle_variant *var, uint8_t *dst)
{
    const size_t bb = oracle_block_bytes(type);
    const int nb = head_dim / ORACLE_BLOCK;
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int h = 0; h < n_kv_heads; ++h)
            for (int b = 0; b < nb; ++b) {
                const uint16_t *x = src + t * src_stride + (int64_t)h * head_dim + b * ORACLE_BLOCK;
                uint8_t *o = dst + ((size_t)t * (size_t)(n_kv_heads * nb) + (size_t)(h * nb + b)) * bb;
                oracle_encode_block_v(type, x, thresholds, centroids, var, o);
            }
}

void oracle_decode_rows(int type, const uint8_t *src, int64_t n_tokens,
                        int n_kv_heads, int head_dim, const float *centroids,
                        double *dst)
{
    oracle_decode_rows_v(type, src, n_tokens, n_kv_heads, head_dim, centroids, NULL, dst);
}

void oracle_decode_rows_v(int type, const uint8_t *src, int64_t n_tokens,
                          int n_kv_heads, int head_dim, const float *centroids,
                          const oracle_variant *var, double *dst)
{
    const size_t bb = oracle_block_bytes(type);
    const int nb = head_dim / ORACLE_BLOCK;
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int h = 0; h < n_kv_heads; ++h)
            for (int b = 0; b < nb; ++b) {
                const uint8_t *blk = src + ((size_t)t * (size_t)(n_kv_heads * nb) + (size_t)(h * nb + b)) * bb;
                double *o = dst + (t * n_kv_heads + h) * (int64_t)head_dim + b * ORACLE_BLOCK;
                oracle_decode_block_v(type, blk, centroids, var, o);
            }
}

/* ---------------------------------------------------------------- attention */

void oracle_dense_attention(const double *q, const double *k, const double *v,
                            int64_t n_tokens, int n_q_heads, int n_kv_heads,
                            int head_dim, double scale, double *out)
{
    const int group = n_q_heads / n_kv_heads;
    for (int h = 0; h < n_q_heads; ++h) {
        const int g = h / group;             /* shared K/V head of this query head */
        const double *qh = q + (int64_t)h * head_dim;
        double *oh = out + (int64_t)h * head_dim;
        for (int i = 0; i < head_dim; ++i) oh[i] = 0.0;
        if (n_tokens <= 0) continue;
        double mx = -INFINITY;
        for (int64_t t = 0; t < n_tokens; ++t) {
            const double *kt = k + (t * n_kv_heads + g) * (int64_t)head_dim;
            double sdot = 0.0;
            for (int i = 0; i < head_dim; ++i) sdot += qh[i] * kt[i];
            sdot *= scale;
            if (sdot > mx) mx = sdot;
        }
        double den = 0.0;
        for (int64_t t = 0; t < n_tokens; ++t) {
            const double *kt = k + (t * n_kv_heads + g) * (int64_t)head_dim;
            const double *vt = v + (t * n_kv_heads + g) * (int64_t)head_dim;
            double sdot = 0.0;
            for (int i = 0; i < head_dim; ++i) sdot += qh[i] * kt[i];
            double p = exp(sdot * scale - mx);
            den += p;
            for (int i = 0; i < head_dim; ++i) oh[i] += p * vt[i];
        }
        for (int i = 0; i < head_dim; ++i) oh[i] /= den;
    }
}

void oracle_attn_decode(int type_k, int type_v, const uint8_t *k_rows,
                        const uint8_t *v_rows, const uint16_t *q_f16,
                        int64_t n_tokens, int n_q_heads, int n_kv_heads,
                        int head_dim, double scale, const float *centroids_k,
                        const float *centroids_v, double *out)
{
    oracle_attn_decode_v(type_k, type_v, k_rows, v_rows, q_f16, n_tokens, n_q_heads,
                         n_kv_heads, head_dim, scale, centroids_k, centroids_v, NULL, NULL, out);
}

void oracle_attn_decode_v(int type_k, int type_v, const uint8_t *k_rows,
                          const uint8_t *v_rows, const uint16_t *q_f16,
                          int64_t n_tokens, int n_q_heads, int n_kv_heads,
                          int head_dim, double scale, const float *centroids_k,
                          const float *centroids_v, const oracle_variant *var_k,
                          const oracle_variant *var_v, double *out)
{
    size_t per_tok = (size_t)n_kv_heads * (size_t)head_dim;
    size_t n_el = (size_t)(n_tokens > 0 ? n_tokens : 0) * per_tok;
    double *k = (double *)malloc((n_el ? n_el : 1) * sizeof(double));
    double *v = (double *)malloc((n_el ? n_el : 1) * sizeof(double));
    double *q = (double *)malloc((size_t)n_q_heads * (size_t)head_dim * sizeof(double));
    if (!k || !v || !q) { free(k); free(v); free(q); return; }
    for (int64_t i = 0; i < (int64_t)n_q_heads * head_dim; ++i) q[i] = oracle_f16_to_f32(q_f16[i]);
    if (n_tokens > 0) {
        oracle_decode_rows_v(type_k, k_rows, n_tokens, n_kv_heads, head_dim, centroids_k, var_k, k);
        oracle_decode_rows_v(type_v, v_rows, n_tokens, n_kv_heads, head_dim, centroids_v, var_v, v);
    }
    oracle_dense_attention(q, k, v, n_tokens, n_q_heads, n_kv_heads, head_dim, scale, out);
    free(k); free(v); free(q);
}

void oracle_attn_prefill(int type_k, int type_v, const uint8_t *k_rows,
                         const uint8_t *v_rows, const uint16_t *q_f16, int64_t pos0,
                         int64_t n_q, int n_q_heads, int n_kv_heads, int head_dim,
                         double scale, const float *centroids_k, const float *centroids_v,
                         double *out)
{
    oracle_attn_prefill_v(type_k, type_v, k_rows, v_rows, q_f16, pos0, n_q, n_q_heads,
                          n_kv_heads, head_dim, scale, centroids_k, centroids_v, NULL, NULL, out);
}

void oracle_attn_prefill_v(int type_k, int type_v, const uint8_t *k_rows,
                           const uint8_t *v_rows, const uint16_t *q_f16, int64_t pos0,
                           int64_t n_q, int n_q_heads, int n_kv_heads, int head_dim,
                           double scale, const float *centroids_k, const float *centroids_v,
                           const oracle_variant *var_k, const oracle_variant *var_v,
                           double *out)
{
    const int64_t n_rows = pos0 + n_q;
    const size_t per_tok = (size_t)n_kv_heads * (size_t)head_dim;
    const size_t per_q = (size_t)n_q_heads * (size_t)head_dim;
    size_t n_el = (size_t)(n_rows > 0 ? n_rows : 0) * per_tok;
    double *k = (double *)malloc((n_el ? n_el : 1) * sizeof(double));
    double *v = (double *)malloc((n_el ? n_el : 1) * sizeof(double));
    double *q = (double *)malloc((per_q ? per_q : 1) * sizeof(double));
    if (!k || !v || !q) { free(k); free(v); free(q); return; }
    if (n_rows > 0) {
        oracle_decode_rows_v(type_k, k_rows, n_rows, n_kv_heads, head_dim, centroids_k, var_k, k);
        oracle_decode_rows_v(type_v, v_rows, n_rows, n_kv_heads, head_dim, centroids_v, var_v, v);
    }
    /* query j sees the first pos0 + j + 1 rows */
    for (int64_t j = 0; j < n_q; ++j) {
        for (size_t i = 0; i < per_q; ++i) q[i] = oracle_f16_to_f32(q_f16[(size_t)j * per_q + i]);
        oracle_dense_attention(q, k, v, pos0 + j + 1, n_q_heads, n_kv_heads, head_dim, scale,
                               out + (size_t)j * per_q);
    }
    free(k); free(v); free(q);
}
