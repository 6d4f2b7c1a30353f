/*
 * tq_oracle.h -- the oracle for the rotated, bit-packed KV cache ("turbo3" / "turbo2").
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library in rotated_bit_kv_tq_gb300/csrc, and it
 * includes nothing from there.
 *
 * Plain, slow, single-threaded C99.  Built with -O2 -ffp-contract=off and without
 * fast-math, so every float operation below is one IEEE-754 binary32 (or binary64)
 * operation in program order.
 *
 * Sources (web pages; cited by title and section):
 *   [TQ]   "llama.cpp に TurboQuant を実装 -- 2bit・3bit の KV キャッシュ圧縮"
 *          (TurboQuant in llama.cpp, openalchemy.io blog).  Sections:
 *          "Why the KV cache is so heavy", "What TurboQuant does differently",
 *          "How small does it get", "Numbers on real models", "How to use",
 *          "Current implementation and what's next".
 *   [ENG]  kenji.blog, "Python nicht nötig! Ich habe eine AI-Inferenz-Engine nur
 *          mit C++ aufgebaut", section 8 "Attention und KV-Cache" (scaled
 *          dot-product attention formula and the decode-step data-flow figure).
 *   [TINY] kenji.blog, "Entwicklungsschritte für kleine KI-Modelle (wie TinyLLaMA)
 *          mit C++", section 4.3 "Grouped-Query Attention" and section 7
 *          "Details zur Implementierung des KV-Caches".
 *
 * Parity status per function is listed beside each declaration.  Every function
 * here is pinned by a CPU test against something other than itself; none is
 * "parity unpinned".
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Types: the code width in bits.  turbo3 = 3 bits/value, turbo2 = 2 bits/value
 * ([TQ] intro and "How to use"). */
#define ORACLE_TURBO2 2
#define ORACLE_TURBO3 3

/* Block bytes: 128 values + one fp16 norm ([TQ] "How small does it get"):
 * 2 + 128*bits/8  ->  50 (turbo3), 34 (turbo2).  Returns 0 for an unknown type.
 * Pinned: the pages' 0.39 / 0.27 bytes per value. */
size_t oracle_block_bytes(int type);

/* KV-cache size from [TQ] "Why the KV cache is so heavy":
 * layers x heads x head_dim x ctx x 2 (K and V) x bytes/value, with the bytes per
 * value given as a ratio num/den so that packed formats come out exact.
 * Pinned: the 14B-shape numbers worked out from the same formula. */
uint64_t oracle_kv_bytes(uint64_t layers, uint64_t kv_heads, uint64_t head_dim,
                         uint64_t ctx, uint64_t bytes_num, uint64_t bytes_den);

/* IEEE binary16 <-> binary32, written from the format definition.
 * f32 -> f16 rounds to nearest, ties to even; overflow goes to infinity.
 * Pinned: exhaustive comparison with numpy's float16 over all 65536 codes and a
 * sweep of float32 inputs. */
float    oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_f16(float f);

/* Unnormalised fast Walsh-Hadamard transform of length n (a power of two, 2..128)
 * in binary32, in place: for h = 1, 2, 4, ..., n/2, every pair (i, i+h) with
 * (i & h) == 0 becomes (a + b, a - b).  Adds and subtracts only
 * ([TQ] "What TurboQuant does differently").  Pinned: equals the dense Sylvester
 * Hadamard product on integer vectors, W*W = n*I, spikes map to +-1 rows. */
void oracle_fwht_f32(float *x, int n);
/* Same butterflies in binary64 (used by decode and attention). */
void oracle_fwht_f64(double *x, int n);

/* Lloyd-Max codebook for one coordinate of a uniformly random unit vector in R^d,
 * density f(y) proportional to (1 - y^2)^((d-3)/2) on [-1, 1]
 * ([TQ] "What TurboQuant does differently": rotate, then an optimal Lloyd-Max
 * scalar quantiser per coordinate).  Lloyd iterations in binary64 with composite
 * Gauss-Legendre quadrature, until no centroid moves by more than 1e-14.
 *   centroids_f64[levels]  the converged centroids (ascending), may be NULL
 *   centroids[levels]      the same rounded to binary32
 *   thresholds[levels-1]   binary32 midpoints (c_j + c_{j+1}) * 0.5f
 * Returns the number of Lloyd iterations, or -1 on bad arguments.
 * Pinned: d = 3 gives the uniform quantiser exactly; symmetry; centroid and
 * midpoint conditions re-checked with scipy quadrature; large d tends to the
 * Gaussian Lloyd-Max levels of Max (1960). */
int oracle_codebook(int d, int levels, double *centroids_f64, float *centroids,
                    float *thresholds);

/* Encode one 128-value block (fp16 bit patterns) into oracle_block_bytes(type)
 * bytes.  Steps ([TQ] "What TurboQuant does differently", "How small does it get"):
 *   1. s = pairwise sum of x_i*x_i: at each level element i (i < len/2) becomes
 *      s[i] + s[i + len/2], len = 128, 64, ..., 2; n = sqrtf(s).
 *   2. stored norm = fp16(min(n, 65504)).
 *   3. z = unnormalised FWHT of x (oracle_fwht_f32).
 *   4. k = n > 0 ? fl(INV_SQRT128 / n) : 0;  y_i = fl(z_i * k)   (unit-vector scale).
 *   5. code: a = |y_i|, m = #{ positive thresholds tau with a > tau },
 *      code = signbit(y_i) ? L/2 - 1 - m : L/2 + m  (L = 2^bits levels).
 *   6. pack (layout described in tq_oracle.c).
 * thresholds: the levels-1 thresholds of oracle_codebook(128, ...).
 * Pinned: brute-force dense-Hadamard quantiser on random blocks, round trip of
 * codeword vectors, the fp16 norm against numpy, the bit layout by a spec test. */
void oracle_encode_block(int type, const uint16_t *x_f16, const float *thresholds,
                         uint8_t *out);

/* Decode one block: x_hat = fp32(norm) * (1/sqrt(128)) * W * c, in binary64. */
void oracle_decode_block(int type, const uint8_t *blk, const float *centroids,
                         double *out);

/* Read back the codes of a block (0 .. 2^bits - 1) and its norm bits. */
void oracle_unpack_block(int type, const uint8_t *blk, uint8_t *codes,
                         uint16_t *norm_f16);

/* Encode n_tokens rows of [n_kv_heads][head_dim] fp16 values, row t starting at
 * src + t * src_stride (elements), into n_tokens packed rows of
 * n_kv_heads * (head_dim/128) blocks each, written back to back at dst.
 * head_dim must be a multiple of 128 ([TQ] "Numbers on real models": head_dim
 * 256 is two stacked 128-blocks). */
void oracle_encode_rows(int type, const uint16_t *src, int64_t n_tokens,
                        int n_kv_heads, int head_dim, int64_t src_stride,
                        const float *thresholds, uint8_t *dst);

/* Decode n_tokens packed rows into [n_tokens][n_kv_heads][head_dim] binary64. */
void oracle_decode_rows(int type, const uint8_t *src, int64_t n_tokens,
                        int n_kv_heads, int head_dim, const float *centroids,
                        double *dst);

/* Textbook scaled dot-product attention for one query row, in binary64
 * ([ENG] section 8: softmax(q K^T * scale) V; [TINY] 4.3: query head h reads
 * KV head floor(h / (n_q_heads / n_kv_heads))).
 *   q[n_q_heads][head_dim], k, v [n_tokens][n_kv_heads][head_dim]
 *   out[n_q_heads][head_dim].   Softmax subtracts the row maximum. */
void oracle_dense_attention(const double *q, const double *k, const double *v,
                            int64_t n_tokens, int n_q_heads, int n_kv_heads,
                            int head_dim, double scale, double *out);

/* Decode-step attention over a packed cache: dequantise K and V rows with
 * oracle_decode_rows (original domain), then oracle_dense_attention.
 * q_f16[n_q_heads][head_dim] (fp16 bits), k_rows / v_rows: n_tokens packed rows.
 * Pinned through its two parts and by closed forms in the tests. */
void oracle_attn_decode(int type_k, int type_v, const uint8_t *k_rows,
                        const uint8_t *v_rows, const uint16_t *q_f16,
                        int64_t n_tokens, int n_q_heads, int n_kv_heads,
                        int head_dim, double scale, const float *centroids_k,
                        const float *centroids_v, double *out);

/* Prompt-chunk (multi-token) attention over a packed cache.  Query token j of the chunk
 * sits at position pos0 + j and attends to rows 0 .. pos0 + j: the rule of the TinyLLaMA
 * article, section 7 (the token at position N writes row N and attends to the view of
 * rows 0..N), applied at every position of the chunk ("llama.cpp に TurboQuant を実装",
 * "Numbers on real models": prompt processing runs over the compressed cache too).
 *   q_f16[n_q][n_q_heads][head_dim] (fp16 bits); k_rows / v_rows: pos0 + n_q packed rows;
 *   out[n_q][n_q_heads][head_dim].
 * Each query is oracle_dense_attention over its prefix of the dequantised rows. */
void oracle_attn_prefill(int type_k, int type_v, const uint8_t *k_rows,
                         const uint8_t *v_rows, const uint16_t *q_f16, int64_t pos0,
                         int64_t n_q, int n_q_heads, int n_kv_heads, int head_dim,
                         double scale, const float *centroids_k, const float *centroids_v,
                         double *out);

/* ---------------------------------------------------------------- quality variants
 * Quality variants of the method.  NULL selects the plain method everywhere.
 *  - signs: bit i (word i / 32, bit i % 32) negates coordinate i of every block before the
 *    rotation, which becomes W D: a random-sign Hadamard.  [TQ] "What TurboQuant does
 *    differently": a random orthogonal rotation spreads the energy, and the FWHT is said to
 *    have the same spreading in expectation; W D is the randomised form of that FWHT.  The
 *    inverse is D W, so decode negates the same coordinates after the inverse rotation.
 *    The sign bits are an input (the caller draws them).
 *  - norm_correction: store |x| / |c|, where |c| is the norm of the block's centroid vector
 *    (pairwise fp32 tree of c_i^2 as for the norm, IEEE sqrt and divide), so that a decoded
 *    block keeps the norm of its input up to the fp16 rounding.  Not on the pages. */
typedef struct oracle_variant {
    uint32_t signs[4];
    int32_t norm_correction;
} oracle_variant;

/* oracle_encode_block with a variant; centroids (2^type fp32) are read only for the norm
 * correction. */
void oracle_encode_block_v(int type, const uint16_t *x_f16, const float *thresholds,
                           const float *centroids, const oracle_variant *var, uint8_t *out);
/* oracle_decode_block with a variant: x_hat = D * (norm / sqrt(128)) * W * c. */
void oracle_decode_block_v(int type, const uint8_t *blk, const float *centroids,
                           const oracle_variant *var, double *out);
void oracle_encode_rows_v(int type, const uint16_t *src, int64_t n_tokens,
                          int n_kv_heads, int head_dim, int64_t src_stride,
                          const float *thresholds, const float *centroids,
                          const oracle_variant *var, uint8_t *dst);
void oracle_decode_rows_v(int type, const uint8_t *src, int64_t n_tokens,
                          int n_kv_heads, int head_dim, const float *centroids,
                          const oracle_variant *var, double *dst);
/* Attention over caches encoded with variants var_k / var_v (dequantised with them). */
void oracle_attn_decode_v(int type_k, int type_v, const uint8_t *k_rows,
                          const uint8_t *v_rows, const uint16_t *q_f16,
                          int64_t n_tokens, int n_q_heads, int n_kv_heads,
                          int head_dim, double scale, const float *centroids_k,
                          const float *centroids_v, const oracle_variant *var_k,
                          const oracle_variant *var_v, double *out);
void oracle_attn_prefill_v(int type_k, int type_v, const uint8_t *k_rows,
                           const uint8_t *v_rows, const uint16_t *q_f16, int64_t pos0,
                           int64_t n_q, int n_q_heads, int n_kv_heads, int head_dim,
                           double scale, const float *centroids_k, const float *centroids_v,
                           const oracle_variant *var_k, const oracle_variant *var_v,
                           double *out);

#ifdef __cplusplus
}
#endif
#endif
