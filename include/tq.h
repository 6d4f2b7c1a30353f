/*
 * tq.h -- C ABI of the GB300 rotated, bit-packed KV cache (turbo3 / turbo2).
 *
 * The method ("llama.cpp に TurboQuant を実装", openalchemy.io): every 128-value K or V
 * block is stored as one fp16 norm plus one Lloyd-Max code per value of the block
 * rotated by a 128-point Walsh-Hadamard transform ("What TurboQuant does
 * differently"); 50 bytes per block for turbo3 (3-bit codes), 34 bytes for turbo2
 * (2-bit codes) ("How small does it get").  Decode attention reads the packed cache
 * directly, in the rotated domain ("Current implementation and what's next":
 * dequantisation fused into the attention kernel, no FP16 K or V materialised).
 *
 * Conventions shared by every call:
 *  - All pointers marked "device" are CUDA device pointers owned by the caller; the
 *    library never allocates, frees or keeps them.  Pointers marked "host" are
 *    ordinary host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Calls that launch work are asynchronous on that stream and never synchronise,
 *    except tq_device_status.
 *  - Arguments are validated on the host before anything is launched; a failing
 *    check returns a status and launches nothing.  No call aborts or throws.
 *  - Conditions only the GPU can see (a page id outside the pool, a position beyond
 *    the capacity, a sequence length beyond max_seq_len) skip the offending row and
 *    record TQ_ERR_OUT_OF_RANGE in a device status word read by tq_device_status.
 *  - The current CUDA device at the time of the call is the device used.
 *
 * Packed block layout (the pages fix the sizes; the bit order is this library's
 * reading, chosen so that codes turn into table lookups with whole-word shifts):
 *   bytes [0,2)   norm = fp16(min(|x|, 65504)), little-endian
 *   bytes [2,34)  8 little-endian u32 words W_0..W_7; value i (w=i/16, j=i%16,
 *                 r=j/8, k=j%8) has code bits 0,1 at bits 4k+2r, 4k+2r+1 of W_w
 *   bytes [34,50) turbo3 only: 4 u32 words V_0..V_3; value i (u=i/32, j=i%32,
 *                 p=j/8, k=j%8) has code bit 2 at bit 4k+p of V_u
 *
 * Cache layout (kenji.blog TinyLLaMA article, section 7: preallocate rows for the
 * maximum context, write the K/V of position N into row N, attend over rows 0..N):
 *   a packed row holds one token: n_kv_heads x (head_dim/128) blocks, head-major,
 *   row_bytes = n_kv_heads * head_dim/128 * block_bytes, rows back to back.
 *   Contiguous cache (page_tokens == 0): row (seq, pos) is at
 *     base + (seq * capacity_tokens + pos) * row_bytes.
 *   Paged cache (page_tokens > 0): page = page_table[seq * max_pages_per_seq +
 *     pos / page_tokens]; row (seq, pos) is at
 *     base + (page * page_tokens + pos % page_tokens) * row_bytes.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_BLOCK_VALUES 128

/* Symbols of this header are the library's only exported symbols. */
#if defined(__GNUC__)
#define TQ_API __attribute__((visibility("default")))
#else
#define TQ_API
#endif

/* Cache types: the code width in bits ("llama.cpp に TurboQuant を実装", intro and
 * "How to use": turbo3 is the default, turbo2 the experimental 2-bit type). */
typedef enum tq_type { TQ_TURBO2 = 2, TQ_TURBO3 = 3 } tq_type;

typedef enum tq_status {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size, bad alignment, bad enum */
    TQ_ERR_UNSUPPORTED = 2,        /* head_dim not a multiple of 128, shape out of range */
    TQ_ERR_NOT_INITIALIZED = 3,    /* tq_codebook_init not called for this type/device */
    TQ_ERR_WORKSPACE_TOO_SMALL = 4,
    TQ_ERR_CUDA = 5,               /* a CUDA runtime call failed */
    TQ_ERR_DEVICE_TIMEOUT = 6,     /* a bounded device-side wait gave up */
    TQ_ERR_OUT_OF_RANGE = 7        /* device saw a page/position/length outside bounds */
} tq_status;

/* A K or V cache of one layer.  Plain data; the caller fills it and owns `base` and
 * `page_table`.  K and V are separate caches ("-ctk" / "-ctv": quantised
 * independently, "How to use"). */
typedef struct tq_cache {
    int32_t type;               /* TQ_TURBO3 or TQ_TURBO2 */
    int32_t n_kv_heads;         /* >= 1 */
    int32_t head_dim;           /* multiple of 128 ("Numbers on real models") */
    int32_t page_tokens;        /* 0 = contiguous; else rows per page, multiple of 32 */
    void *base;                 /* device, 16-byte aligned: the row pool */
    int64_t capacity_tokens;    /* contiguous: rows reserved per sequence */
    int32_t n_seqs;             /* sequences addressed by this cache (>= 1) */
    int32_t max_pages_per_seq;  /* paged: columns of page_table */
    const int32_t *page_table;  /* paged: device int32 [n_seqs][max_pages_per_seq] */
    int64_t n_pages;            /* paged: pages in the pool at base */
    /* Quality variants (all zero: the plain method).
     * rotation_signs: bit i (word i / 32, bit i % 32) negates coordinate i of every
     *   128-value block before the rotation, which becomes W D, a random-sign Hadamard
     *   ("What TurboQuant does differently": a random orthogonal rotation, whose energy
     *   spreading the FWHT matches in expectation).  Decode negates the same coordinates
     *   after the inverse rotation (D W); attention rotates queries with the K cache's
     *   signs and un-rotates outputs with the V cache's.  The caller draws the bits; they
     *   must stay the same for the life of the cache.
     * norm_correction: 0 stores |x|; 1 stores |x| / |c|, where |c| is the norm of the
     *   block's centroid vector (pairwise fp32 sum of c_i^2, IEEE sqrt and divide), so a
     *   decoded block keeps the norm of its input up to the fp16 rounding.  It changes only
     *   the stored norm; decode and attention are unchanged.  Not on the pages. */
    uint32_t rotation_signs[4];
    int32_t norm_correction;
} tq_cache;

/* 50 (turbo3) or 34 (turbo2); 0 for an unknown type.  "How small does it get":
 * 128 values plus one FP16 norm, 0.39 / 0.27 bytes per value. */
TQ_API size_t tq_block_bytes(int type);

/* Bytes of one packed token row: n_kv_heads * head_dim/128 * tq_block_bytes(type);
 * 0 if the arguments are invalid. */
TQ_API size_t tq_row_bytes(int type, int n_kv_heads, int head_dim);

/* Build the type's Lloyd-Max codebook and upload it to `device`.
 * The codebook is the optimal scalar quantiser for one coordinate of a uniformly
 * random unit vector in R^128, density (1-y^2)^(125/2) on [-1,1] ("What TurboQuant
 * does differently": after the rotation every coordinate follows the same law, so a
 * fixed, data-independent Lloyd-Max codebook is near optimal).  Centroids are solved
 * in double precision and rounded to fp32; thresholds are the fp32 midpoints.
 * Idempotent and cheap after the first call; must precede tq_encode / tq_decode /
 * tq_attn_decode of that type on that device.  Not thread-safe against itself. */
TQ_API tq_status tq_codebook_init(int type, int device);

/* Host copy of the type's codebook: centroids[2^type] (ascending) and
 * thresholds[2^type - 1].  Either pointer may be NULL. */
TQ_API tq_status tq_codebook_get(int type, float *centroids, float *thresholds);

/* Encode n_tokens fp16 token rows into the cache (the per-token write path,
 * "What TurboQuant does differently": the rotation is cheap enough to live in the
 * cache-write path).
 *   src_f16        device fp16 [n_tokens][n_kv_heads][head_dim]; row i starts at
 *                  src_f16 + i * src_token_stride elements.  16-byte aligned;
 *                  src_token_stride >= n_kv_heads*head_dim and a multiple of 8.
 *   seq_ids        device int32 [n_tokens] or NULL (then every token uses seq_id)
 *   positions      device int32 [n_tokens] or NULL (then token i goes to pos0 + i)
 * Per block: n = |x| (fixed pairwise fp32 sum, IEEE sqrt), norm = fp16(min(n,65504)),
 * z = unnormalised FWHT of x, y = z * fl(fl(1/sqrt(128)) / n), code = sign-magnitude
 * Lloyd-Max index of y.  Codes and norms are bit-identical to the CPU oracle.
 * n_tokens == 0 is a no-op. */
TQ_API tq_status tq_encode(const tq_cache *dst, const void *src_f16, int64_t n_tokens,
                    int64_t src_token_stride, const int32_t *seq_ids,
                    const int32_t *positions, int32_t seq_id, int64_t pos0,
                    void *stream);

/* tq_encode of the K rows into `k` and of the V rows into `v` in one launch (K and V
 * are quantised independently, "How to use": -ctk / -ctv; the decode step appends both
 * before attending, kenji.blog article section 8).  Arguments as for tq_encode, per
 * cache; seq_ids / positions / seq_id / pos0 apply to both.  Caches of different types
 * are encoded by two launches. */
TQ_API tq_status tq_encode_kv(const tq_cache *k, const tq_cache *v, const void *k_src_f16,
                              const void *v_src_f16, int64_t n_tokens, int64_t k_token_stride,
                              int64_t v_token_stride, const int32_t *seq_ids,
                              const int32_t *positions, int32_t seq_id, int64_t pos0,
                              void *stream);

/* Dequantise rows pos0 .. pos0+n_tokens-1 of sequence seq_id to fp32
 * dst [n_tokens][n_kv_heads][head_dim] (device): x_hat = norm * W c / sqrt(128)
 * ("What TurboQuant does differently": the rotation is undone at read time). */
TQ_API tq_status tq_decode(const tq_cache *src, int32_t seq_id, int64_t pos0, int64_t n_tokens,
                    float *dst, void *stream);

/* Workspace bytes tq_attn_decode needs for this shape on the current device. */
TQ_API size_t tq_attn_workspace_bytes(int n_seqs, int n_q_heads, int head_dim,
                               int64_t max_seq_len);

/* Single-token decode attention over the packed caches (kenji.blog article, section
 * 8: out = softmax(q K^T * scale) V over the cached positions; TinyLLaMA article 4.3:
 * query head h reads KV head floor(h / (n_q_heads / n_kv_heads))).
 *   k, v           caches of one layer; same n_kv_heads and head_dim; the types may
 *                  differ (mixed "-ctk" / "-ctv").  Batch entry s reads cache
 *                  sequence s.
 *   q_f16          device fp16 [n_seqs][n_q_heads][head_dim], 16-byte aligned
 *   seq_lens       device int32 [n_seqs]: attend to positions [0, seq_lens[s]); the
 *                  caller appends the current token first (decode-step data flow of
 *                  the kenji.blog article, section 8).  0 gives a zero output.
 *   max_seq_len    host upper bound of seq_lens (sizes the split-K grid)
 *   softmax_scale  score scale; pass 0 for 1/sqrt(head_dim)
 *   out            device fp32 [n_seqs][n_q_heads][head_dim]
 *   workspace      device scratch of at least tq_attn_workspace_bytes(...) bytes,
 *                  16-byte aligned; contents need no initialisation.  Its first 4 KiB
 *                  hold an epoch word that the next call on the same workspace reads
 *                  (see below), so calls that share a workspace must be ordered (one
 *                  stream, or events), as they must be for the partials anyway.
 * The scores are computed as |k| * (W q / sqrt(128)) . c(codes) and the values
 * accumulated as sum p |v| c(codes), both in the rotated domain, with one inverse
 * FWHT per output block; no fp16 K or V is formed.  The keys are split over the SMs
 * (split-K) and the partial results merged by log-sum-exp.  On the tensor-core path a
 * single sequence whose splits fit one wave is one cooperative launch: its CTAs merge the
 * partials themselves, each partial value stored with a tag derived from the epoch word
 * (which the launch advances), so that a reader knows a current value from a stale one
 * without a grid barrier.  Otherwise a merge kernel follows the attention kernel. */
TQ_API tq_status tq_attn_decode(const tq_cache *k, const tq_cache *v, const void *q_f16,
                         int n_seqs, int n_q_heads, const int32_t *seq_lens,
                         int64_t max_seq_len, float softmax_scale, float *out,
                         void *workspace, size_t ws_bytes, void *stream);

/* One decode step of a layer: append each sequence's new token to the caches, then attend
 * over the positions that include it.  This is the decode-step data flow of the kenji.blog
 * article, section 8 (the token at position N writes row N, then attends to rows 0..N),
 * in one call: the result equals tq_encode_kv of the new rows followed by tq_attn_decode.
 *   k_new_f16,     device fp16 [n_seqs][n_kv_heads][head_dim], 16-byte aligned: the new K
 *   v_new_f16      and V rows; sequence s's rows are encoded (bit-identical to tq_encode_kv)
 *                  into position seq_lens[s] - 1 of cache sequence s.  A sequence with
 *                  seq_lens[s] == 0 appends nothing and gets a zero output.
 *   other arguments as for tq_attn_decode; seq_lens counts the appended token.
 * On the tensor-core path the CTA whose split holds position seq_lens[s] - 1 encodes the
 * rows itself, so the step is one attention launch (plus the merge kernel where
 * tq_attn_decode has one); shapes that path does not take append in a launch of their own
 * first.  A row whose position the cache cannot
 * address is skipped and TQ_ERR_OUT_OF_RANGE is recorded for tq_device_status. */
TQ_API tq_status tq_attn_decode_append(const tq_cache *k, const tq_cache *v,
                                       const void *k_new_f16, const void *v_new_f16,
                                       const void *q_f16, int n_seqs, int n_q_heads,
                                       const int32_t *seq_lens, int64_t max_seq_len,
                                       float softmax_scale, float *out, void *workspace,
                                       size_t ws_bytes, void *stream);

/* Causal attention of a prompt chunk (multi-token / prefill) over the packed caches.
 * Query token j of the chunk sits at position pos0 + j and attends to rows 0 .. pos0 + j of
 * cache sequence seq_id: the KV-cache rule of the kenji.blog TinyLLaMA article, section 7
 * (the token at position N writes row N and attends to the view of rows 0..N), applied at
 * every position of the chunk.  Prompt processing over the compressed cache is what
 * "llama.cpp に TurboQuant を実装" measures in "Numbers on real models"; dequantising
 * inside the Flash-Attention tiles, never forming FP16 K or V in memory, is its roadmap
 * ("Current implementation and what's next").
 *   k, v           caches of one layer; same n_kv_heads and head_dim, 128 or 256 (other
 *                  head dims return TQ_ERR_UNSUPPORTED); types may differ
 *   q_f16          device fp16 [n_q][n_q_heads][head_dim], 16-byte aligned
 *   seq_id         the chunk's sequence; pos0 >= 0 its first position.  The rows of the
 *                  chunk itself must already be in the caches (encode them first).
 *   n_q            queries in the chunk; 0 is a no-op
 *   softmax_scale  score scale; pass 0 for 1/sqrt(head_dim)
 *   out            device fp32 [n_q][n_q_heads][head_dim], 16-byte aligned
 *   n_q_heads      a multiple of n_kv_heads, at most 128 query heads per KV head
 * No workspace: one CTA per (block of 128 / G query tokens, KV head) covers all the keys
 * its queries see, or, at head_dim 128 when that would leave much of the last wave of CTAs
 * idle, a cluster of two CTAs splits those keys and merges by log-sum-exp in shared
 * memory.  Rows the device cannot address (page id or position out of range) are skipped
 * and TQ_ERR_OUT_OF_RANGE is recorded for tq_device_status. */
TQ_API tq_status tq_attn_prefill(const tq_cache *k, const tq_cache *v, const void *q_f16,
                                 int32_t seq_id, int64_t pos0, int64_t n_q, int n_q_heads,
                                 float softmax_scale, float *out, void *stream);

/* Size of the fixed scratch array of tq_attn_decode_noalloc: 8 MiB per device. */
#define TQ_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* tq_attn_decode without a workspace argument, for callers that cannot allocate device
 * memory when they need attention.  Examples are code that runs between the steps of
 * a serving loop whose memory pools are fully reserved at start-up, and embedders whose
 * allocator must not be re-entered, or whose policy forbids cudaMalloc (it can
 * synchronise the device) on the decode path.  The pages have no counterpart to this
 * entry point; it is a packaging variant of tq_attn_decode.
 *   Arguments and results are those of tq_attn_decode, minus workspace / ws_bytes; the
 *   argument checks are the same code.
 *   Scratch: a fixed array of TQ_NOALLOC_SCRATCH_BYTES in the library's device memory
 *   (every GPU that loads the library holds it until the process exits).  A shape whose
 *   tq_attn_workspace_bytes(...) exceeds it returns TQ_ERR_WORKSPACE_TOO_SMALL and
 *   launches nothing.  The call never allocates or frees memory.
 *   Set-up: every call looks up the array's device address in the current context (with
 *   the call's device current), so a device reset or a second context on the device is
 *   followed.  The first call on a device loads the library's device code there; make
 *   that first call before any stream capture.
 *   Sharing: all calls on a device share the array and it keeps the last call's
 *   contents (each call writes every partial it reads, so nothing needs clearing; the
 *   epoch word of tq_attn_decode's workspace lives in it too).
 *   Calls whose kernels overlap on the GPU (different streams without ordering) race on
 *   it; order them on one stream or with events. */
TQ_API tq_status tq_attn_decode_noalloc(const tq_cache *k, const tq_cache *v,
                                        const void *q_f16, int n_seqs, int n_q_heads,
                                        const int32_t *seq_lens, int64_t max_seq_len,
                                        float softmax_scale, float *out, void *stream);

/* Fault injection for tests of the bounded device-side waits: failure detection without a
 * GPU fault (nothing traps, hangs or touches bad memory).  The next
 * n_calls launches of the tensor-core decode-attention kernel (tq_attn_decode,
 * tq_attn_decode_append and tq_attn_decode_noalloc on the shapes that kernel takes) request
 * no tile copies and give every wait on a tile a limit of 64 polls.  With no copy in flight
 * each wait runs out, the kernel records TQ_ERR_DEVICE_TIMEOUT for tq_device_status,
 * writes empty partials (a zero output) and returns normally; later calls run as usual.
 * Process-wide; n_calls = 0 cancels.  Returns TQ_ERR_INVALID_ARGUMENT for n_calls < 0. */
TQ_API tq_status tq_inject_wait_timeout(int n_calls);

/* Synchronise `stream`, then read and clear the device status word of the current
 * device: *status_out = TQ_OK or the first device-side error recorded since the
 * last read.  Returns TQ_ERR_CUDA if synchronisation fails. */
TQ_API tq_status tq_device_status(void *stream, int32_t *status_out);

/* Static, human-readable name of a status code. */
TQ_API const char *tq_status_str(int status);

#ifdef __cplusplus
}
#endif
#endif
