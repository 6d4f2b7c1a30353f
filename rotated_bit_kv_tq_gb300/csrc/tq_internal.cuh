// tq_internal.cuh -- definitions shared by the CUDA translation units of the library.
// Nothing here is shared with the oracle.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq.h"

namespace tq {

constexpr int kBlock = TQ_BLOCK_VALUES;  // values per block

// The binary32 value nearest to 1/sqrt(128) = 2^-3.5.
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

__host__ __device__ constexpr int block_bytes(int type) { return 2 + kBlock * type / 8; }

// Split-K CTAs of one cluster for a single sequence: the tensor-core attention kernel merges
// the partials of these consecutive splits in distributed shared memory before writing one
// row.  Batches run without pairs (in a batch of mixed lengths a pair often joins a split
// with work to an empty one, which then holds its SM until its partner is done).
constexpr int kClusterSplits = 2;

// Decode workspace: the grid-merge area (an epoch word and one arrival flag per CTA of a
// decode launch that merges its own partials after a grid barrier), then the partial rows.
constexpr int kGridMergeMaxCtas = 160;   // one wave on 152 SMs; a multiple of 32, 16 and 8
constexpr size_t kGridBarrierBytes = 4096;   // >= 8 * (1 + kGridMergeMaxCtas), 256-aligned

// Floats per split-partial row of one (sequence, split, query head): head_dim rotated-domain
// sums, the running max m, the running sum l, two pad floats (rows stay 16-byte aligned).
__host__ __device__ constexpr int part_stride(int head_dim) { return head_dim + 4; }

__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Device-side view of a tq_cache.
struct CacheView {
    uint8_t *base;
    const int32_t *page_table;
    int64_t capacity;
    int64_t n_pages;
    int32_t page_tokens;
    int32_t max_pages;
    int32_t n_seqs;
    int32_t row_bytes;
    uint32_t signs[4];          // rotation_signs of tq_cache (all zero: plain FWHT)
    int32_t norm_correction;
    int32_t has_signs;          // any sign bit set
};

#if defined(__CUDACC__)
// -1.0f-sign mask of coordinate i under a cache's rotation signs: 0x80000000 or 0.
// (The word is picked with selects: a run-time index into a parameter array would copy
// the array to local memory.)
__device__ __forceinline__ uint32_t sign_mask(const CacheView &c, int i) {
    const int w = i >> 5;
    const uint32_t word = w == 0 ? c.signs[0] : w == 1 ? c.signs[1] : w == 2 ? c.signs[2] : c.signs[3];
    return ((word >> (i & 31)) & 1u) << 31;
}

// Negate the values of coordinates i0 .. i0+3 whose rotation-sign bit is set (D v): on a
// query before its rotation with the K cache's signs, on an output after its inverse
// rotation with the V cache's.
__device__ __forceinline__ void apply_signs4(float (&v)[4], const CacheView &c, int i0) {
    if (!c.has_signs) return;
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(__float_as_uint(v[e]) ^ sign_mask(c, i0 + e));
}
#endif

#if defined(__CUDACC__)
// First device-side error of the current device (0 = none); read by tq_device_status.
extern __device__ int32_t g_status;

__device__ __forceinline__ void record_error(int32_t code) { atomicCAS(&g_status, 0, code); }

// Address of row (seq, pos), or nullptr (and TQ_ERR_OUT_OF_RANGE recorded) when the row
// lies outside the cache.
__device__ __forceinline__ uint8_t *row_ptr(const CacheView &c, int64_t seq, int64_t pos) {
    if (seq < 0 || seq >= c.n_seqs || pos < 0) {
        record_error(TQ_ERR_OUT_OF_RANGE);
        return nullptr;
    }
    int64_t row;
    if (c.page_tokens == 0) {
        if (pos >= c.capacity) {
            record_error(TQ_ERR_OUT_OF_RANGE);
            return nullptr;
        }
        row = seq * c.capacity + pos;
    } else {
        int64_t pi = pos / c.page_tokens;
        if (pi >= c.max_pages) {
            record_error(TQ_ERR_OUT_OF_RANGE);
            return nullptr;
        }
        int64_t page = c.page_table[seq * c.max_pages + pi];
        if (page < 0 || page >= c.n_pages) {
            record_error(TQ_ERR_OUT_OF_RANGE);
            return nullptr;
        }
        row = page * c.page_tokens + pos % c.page_tokens;
    }
    return c.base + row * (int64_t)c.row_bytes;
}

// Programmatic dependent launch.  Kernels launched with the programmatic-serialization
// attribute may start while the previous kernel in the stream is still running; they call
// pdl_wait() before their first global-memory access (it returns once that kernel has
// completed and its writes are visible, and at once for a normal launch).
// pdl_launch_dependents() lets the next such kernel be scheduled early; it still waits for
// this one to complete before it touches memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
// Issued before pdl_wait() it is safe even for data the previous kernel still writes: it
// fills nothing in the SM, and L2 is where device memory is coherent, so the loads after
// the wait see the final contents; what it saves is the first access's latency (DRAM and
// address translation), which otherwise falls after the wait.
__device__ __forceinline__ void l2_prefetch(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ phase trace
// Only in the traced library (TQ_TRACE_PHASES; build.build(trace=True) makes libtq_trace.so):
// %globaltimer stamps at phase boundaries of every CTA of the decode-attention and merge
// kernels, read back through tq_phase_trace_read.  The product library has no trace code.
constexpr int kTraceCtas = 2048;     // attention CTA slots; merge CTAs at kTraceCtas + index
constexpr int kTracePoints = 12;
#if defined(TQ_TRACE_PHASES)
extern __device__ unsigned long long g_phase_trace[2 * kTraceCtas][kTracePoints];
__device__ __forceinline__ unsigned long long phase_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#define TQ_PHASE(slot, point) \
    do { if ((slot) < 2 * kTraceCtas) g_phase_trace[(slot)][(point)] = phase_clock(); } while (0)
#define TQ_PHASE_MAX(slot, point) \
    do { if ((slot) < 2 * kTraceCtas) atomicMax(&g_phase_trace[(slot)][(point)], phase_clock()); } while (0)
#else
#define TQ_PHASE(slot, point) ((void)0)
#define TQ_PHASE_MAX(slot, point) ((void)0)
#endif

// Launch configuration with the programmatic-serialization attribute set (attrs[0]); a
// caller may add a second attribute at attrs[1].
struct PdlConfig {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    PdlConfig(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) : cfg(), attrs() {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
};
#endif  // __CUDACC__

// ------------------------------------------------------------------ codebook tables
// Uploaded by tq_codebook_init.  Index 0 = turbo2 (4 levels), 1 = turbo3 (8 levels).
struct Codebook {
    float centroid[8];
    float threshold[7];
    // fp16 operands of the tensor-core attention kernels: centroid_h[j] = fp16(h_scale *
    // centroid[j]), with h_scale in [1, 2) chosen so that every scaled centroid lies within
    // a few 1e-5 (relative) of an fp16 value.  The kernels divide h_scale out in fp32 (the
    // query scale on the key side, the value norms on the value side), so a centroid's
    // systematic fp16 error drops from up to 2.3e-4 to 2.2e-5 (turbo3) and 7e-7 (turbo2).
    __half centroid_h[8];
    float h_scale;
};
#if defined(__CUDACC__)
extern __constant__ Codebook c_codebook[2];
#endif

__host__ __device__ constexpr int cb_index(int type) { return type == TQ_TURBO3 ? 1 : 0; }

// ------------------------------------------------------------------ host side
bool codebook_ready(int type, int device);
tq_status check_cuda(cudaError_t e);
int device_sm_count();   // SM count of the current device (queried once per device)
// One-time set-up of a kernel on the current device, cached per (kernel, device): raises
// its dynamic shared-memory limit to smem_bytes and computes how many CTAs of `threads`
// threads and smem_bytes bytes fit on one SM (*per_sm, may be null).  Later calls with the
// same or a smaller size cost a table lookup instead of two runtime calls.
tq_status kernel_setup(const void *kernel, int smem_bytes, int threads, int *per_sm);
CacheView make_view(const tq_cache &c);
tq_status validate_cache(const tq_cache *c);
// Argument checks of the single-token attention entry points (tq_attn_decode,
// tq_attn_decode_append, tq_attn_decode_noalloc), everything but the scratch memory; on
// success *scale_out is the softmax scale to use (1/sqrt(head_dim) when 0 is passed).
tq_status check_attn_args(const tq_cache *k, const tq_cache *v, const void *q_f16, int n_seqs,
                          int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len,
                          float softmax_scale, const float *out, float *scale_out);

// Kernel launchers (one per .cu file).
tq_status launch_encode(const tq_cache &dst, const void *src, int64_t n_tokens, int64_t stride,
                        const int32_t *seq_ids, const int32_t *positions, int32_t seq_id,
                        int64_t pos0, cudaStream_t stream);
tq_status launch_encode_kv(const tq_cache &k, const tq_cache &v, const void *k_src,
                           const void *v_src, int64_t n_tokens, int64_t k_stride,
                           int64_t v_stride, const int32_t *seq_ids, const int32_t *positions,
                           int32_t seq_id, int64_t pos0, cudaStream_t stream);
tq_status launch_decode(const tq_cache &src, int32_t seq_id, int64_t pos0, int64_t n_tokens,
                        float *dst, cudaStream_t stream);
size_t attn_workspace_bytes(int n_seqs, int n_q_heads, int head_dim, int64_t max_seq_len,
                            int sm_count);
// k_new / v_new (fp16 [n_seqs][Hkv][D], or null): append sequence s's new token at position
// seq_lens[s] - 1 before attending (the tensor-core kernel does it in the same launch).
tq_status launch_attn(const tq_cache &k, const tq_cache &v, const void *q, int n_seqs,
                      int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len, float scale,
                      float *out, void *ws, size_t ws_bytes, cudaStream_t stream,
                      const void *k_new = nullptr, const void *v_new = nullptr);
tq_status launch_append(const tq_cache &k, const tq_cache &v, const void *k_new, const void *v_new,
                        const int32_t *seq_lens, int n_seqs, cudaStream_t stream);

// Tensor-core decode attention (tq_attn_mma.cu): writes split partials like the fp32 kernel.
bool attn_mma_supported(const tq_cache &k, const tq_cache &v, int n_q_heads);
// `cluster` consecutive splits (2 or 1) merge their partials in distributed shared memory;
// the kernel writes n_splits / cluster partial rows per (sequence, head).  With `out` set
// (grid_merge_fits: one sequence, one wave; cluster 1) the CTAs merge the partials
// themselves and write the output, no merge kernel following; `bar` is the grid-merge area
// (its epoch word persists from call to call) and `part` holds tagged 64-bit words.
bool grid_merge_fits(int n_seqs, int n_splits);
tq_status launch_attn_mma(const tq_cache &k, const tq_cache &v, const void *q, int n_seqs,
                          int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len, float scale,
                          float *part, int n_splits, int tokens_per_split, int cluster,
                          const void *k_new, const void *v_new, float *out, uint64_t *bar,
                          cudaStream_t stream);

// Fault injection of tq_inject_wait_timeout (tq_attn_mma.cu).
tq_status inject_wait_timeout(int n_calls);

// Prompt-chunk attention on the 5th-generation tensor cores (tq_prefill_tc.cu).
bool prefill_supported(const tq_cache &k, const tq_cache &v, int n_q_heads);
tq_status launch_prefill(const tq_cache &k, const tq_cache &v, const void *q, int32_t seq_id,
                         int64_t pos0, int64_t n_q, int n_q_heads, float scale, float *out,
                         cudaStream_t stream);

// h_scale of a type's fp16 centroid table (see Codebook); 1 for an unknown type.
float centroid_h_scale(int type);

// Host Lloyd-Max solver (tq_codebook.cpp).
void solve_codebook(int levels, double *centroids);

}  // namespace tq
