// tq_api.cu -- the C ABI: host-side validation, codebook set-up, status word.
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "tq_internal.cuh"

namespace tq {

__device__ int32_t g_status = 0;
#if defined(TQ_TRACE_PHASES)
__device__ unsigned long long g_phase_trace[2 * kTraceCtas][kTracePoints];
#endif
__constant__ Codebook c_codebook[2];

namespace {

constexpr int kMaxDevices = 64;
bool g_ready[kMaxDevices][2];
Codebook g_host_cb[2];
bool g_host_cb_done[2];
std::atomic<float> g_h_scale[2];   // Codebook::h_scale, published once the table exists
std::mutex g_mu;
std::atomic<int> g_sm_count[kMaxDevices];

struct KernelState {
    int smem = -1;      // dynamic shared-memory limit set so far
    int threads = 0;    // occupancy computed for this block size and smem
    int per_sm = 0;
};
std::map<std::pair<const void *, int>, KernelState> g_kernels;
std::mutex g_kernels_mu;

bool valid_type(int type) { return type == TQ_TURBO2 || type == TQ_TURBO3; }

// Worst relative error, over the centroid magnitudes mag[0..n), of the fp16 table scaled by
// a: |fp16(a m) / a - m| / m (evaluated in double; a is the fp32 value the kernels use).
double scaled_table_error(float a, const float *mag, int n) {
    double worst = 0.0;
    for (int j = 0; j < n; ++j) {
        const double v = (double)a * (double)mag[j];
        const double h = (double)__half2float(__double2half(v));
        const double e = std::fabs(h / (double)a - (double)mag[j]) / (double)mag[j];
        worst = e > worst ? e : worst;
    }
    return worst;
}

// The scale in [1, 2) that puts every centroid magnitude closest to an fp16 value.  A best
// scale puts at least one magnitude exactly on an fp16 value, so the candidates are
// a = g / m_j for every magnitude m_j and every fp16 value g with a in [1, 2); the first
// candidate with the smallest worst-case error wins (a deterministic search over at most
// 4 x 2048 candidates).
float choose_h_scale(const float *centroid, int levels) {
    float mag[4];
    const int n = levels / 2;
    for (int j = 0; j < n; ++j) mag[j] = centroid[levels / 2 + j];
    float best = 1.0f;
    double best_err = scaled_table_error(1.0f, mag, n);
    for (int j = 0; j < n; ++j) {
        // fp16 values g in [m_j, 2 m_j): every mantissa of the one or two binades involved
        for (int e = -15; e <= 15; ++e) {
            for (int m = 0; m < 1024; ++m) {
                const double g = std::ldexp(1.0 + m / 1024.0, e);
                const double a = g / (double)mag[j];
                if (a < 1.0 || a >= 2.0) continue;
                const float af = (float)a;
                const double err = scaled_table_error(af, mag, n);
                if (err < best_err) {
                    best_err = err;
                    best = af;
                }
            }
        }
    }
    return best;
}

const Codebook &host_codebook(int type) {
    int i = cb_index(type);
    if (!g_host_cb_done[i]) {
        const int levels = 1 << type;
        double c[8];
        solve_codebook(levels, c);
        Codebook cb;
        std::memset(&cb, 0, sizeof cb);
        for (int j = 0; j < levels; ++j) cb.centroid[j] = (float)c[j];
        cb.h_scale = choose_h_scale(cb.centroid, levels);
        for (int j = 0; j < levels; ++j)
            cb.centroid_h[j] = __double2half((double)cb.h_scale * (double)cb.centroid[j]);
        // fp32 midpoints of the fp32 centroids
        for (int j = 0; j + 1 < levels; ++j)
            cb.threshold[j] = (cb.centroid[j] + cb.centroid[j + 1]) * 0.5f;
        g_host_cb[i] = cb;
        g_host_cb_done[i] = true;
        g_h_scale[i].store(cb.h_scale);
    }
    return g_host_cb[i];
}

}  // namespace

float centroid_h_scale(int type) {
    if (!valid_type(type)) return 1.0f;
    const float h = g_h_scale[cb_index(type)].load();
    if (h > 0.0f) return h;   // published by host_codebook (always, once a cache is valid)
    std::lock_guard<std::mutex> lock(g_mu);
    return host_codebook(type).h_scale;
}

bool codebook_ready(int type, int device) {
    if (device < 0 || device >= kMaxDevices || !valid_type(type)) return false;
    return g_ready[device][cb_index(type)];
}

tq_status check_cuda(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < kMaxDevices && (n = g_sm_count[dev].load()) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 1;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n);
    return n;
}

tq_status kernel_setup(const void *kernel, int smem_bytes, int threads, int *per_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_kernels_mu);
    KernelState &st = g_kernels[std::make_pair(kernel, dev)];
    if (st.smem < smem_bytes) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess)
            return TQ_ERR_CUDA;
        st.smem = smem_bytes;
        st.threads = 0;
    }
    if (per_sm) {
        if (st.threads != threads) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, st.smem) !=
                cudaSuccess)
                return TQ_ERR_CUDA;
            st.threads = threads;
            st.per_sm = n < 1 ? 1 : n;
        }
        *per_sm = st.per_sm;
    }
    return TQ_OK;
}

CacheView make_view(const tq_cache &c) {
    CacheView v;
    v.base = static_cast<uint8_t *>(c.base);
    v.page_table = c.page_table;
    v.capacity = c.capacity_tokens;
    v.n_pages = c.n_pages;
    v.page_tokens = c.page_tokens;
    v.max_pages = c.max_pages_per_seq;
    v.n_seqs = c.n_seqs;
    v.row_bytes = (int32_t)tq_row_bytes(c.type, c.n_kv_heads, c.head_dim);
    for (int w = 0; w < 4; ++w) v.signs[w] = c.rotation_signs[w];
    v.norm_correction = c.norm_correction;
    v.has_signs = (c.rotation_signs[0] | c.rotation_signs[1] | c.rotation_signs[2] |
                   c.rotation_signs[3]) != 0;
    return v;
}

tq_status validate_cache(const tq_cache *c) {
    if (!c || !c->base) return TQ_ERR_INVALID_ARGUMENT;
    if (!valid_type(c->type)) return TQ_ERR_INVALID_ARGUMENT;
    if (c->n_kv_heads < 1 || c->head_dim < 1 || c->n_seqs < 1) return TQ_ERR_INVALID_ARGUMENT;
    if (c->head_dim % kBlock != 0) return TQ_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(c->base) % 16 != 0) return TQ_ERR_INVALID_ARGUMENT;
    if ((int64_t)c->n_kv_heads * (c->head_dim / kBlock) > 128) return TQ_ERR_UNSUPPORTED;
    if (c->page_tokens < 0) return TQ_ERR_INVALID_ARGUMENT;
    if (c->norm_correction != 0 && c->norm_correction != 1) return TQ_ERR_INVALID_ARGUMENT;
    if (c->page_tokens == 0) {
        if (c->capacity_tokens < 1) return TQ_ERR_INVALID_ARGUMENT;
    } else {
        if (c->page_tokens % 32 != 0) return TQ_ERR_UNSUPPORTED;
        if (!c->page_table || c->max_pages_per_seq < 1 || c->n_pages < 1)
            return TQ_ERR_INVALID_ARGUMENT;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (!codebook_ready(c->type, dev)) return TQ_ERR_NOT_INITIALIZED;
    return TQ_OK;
}

}  // namespace tq

using namespace tq;

extern "C" {

size_t tq_block_bytes(int type) { return valid_type(type) ? (size_t)block_bytes(type) : 0; }

size_t tq_row_bytes(int type, int n_kv_heads, int head_dim) {
    if (!valid_type(type) || n_kv_heads < 1 || head_dim < kBlock || head_dim % kBlock) return 0;
    return (size_t)n_kv_heads * (size_t)(head_dim / kBlock) * (size_t)block_bytes(type);
}

tq_status tq_codebook_get(int type, float *centroids, float *thresholds) {
    if (!valid_type(type)) return TQ_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(g_mu);
    const Codebook &cb = host_codebook(type);
    const int levels = 1 << type;
    if (centroids) std::memcpy(centroids, cb.centroid, sizeof(float) * levels);
    if (thresholds) std::memcpy(thresholds, cb.threshold, sizeof(float) * (levels - 1));
    return TQ_OK;
}

tq_status tq_codebook_init(int type, int device) {
    if (!valid_type(type) || device < 0 || device >= kMaxDevices) return TQ_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ready[device][cb_index(type)]) return TQ_OK;
    const Codebook &cb = host_codebook(type);
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return TQ_ERR_CUDA;
    cudaError_t e = cudaMemcpyToSymbol(c_codebook, &cb, sizeof(Codebook),
                                       sizeof(Codebook) * cb_index(type));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    cudaSetDevice(prev);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    g_ready[device][cb_index(type)] = true;
    return TQ_OK;
}

tq_status tq_encode(const tq_cache *dst, const void *src_f16, int64_t n_tokens,
                    int64_t src_token_stride, const int32_t *seq_ids, const int32_t *positions,
                    int32_t seq_id, int64_t pos0, void *stream) {
    tq_status st = validate_cache(dst);
    if (st != TQ_OK) return st;
    if (n_tokens < 0) return TQ_ERR_INVALID_ARGUMENT;
    if (n_tokens == 0) return TQ_OK;
    if (!src_f16 || reinterpret_cast<uintptr_t>(src_f16) % 16) return TQ_ERR_INVALID_ARGUMENT;
    const int64_t row_elems = (int64_t)dst->n_kv_heads * dst->head_dim;
    if (src_token_stride < row_elems || src_token_stride % 8) return TQ_ERR_INVALID_ARGUMENT;
    if (!positions && pos0 < 0) return TQ_ERR_INVALID_ARGUMENT;
    if (!seq_ids && (seq_id < 0 || seq_id >= dst->n_seqs)) return TQ_ERR_INVALID_ARGUMENT;
    if (n_tokens > (int64_t)1 << 40) return TQ_ERR_UNSUPPORTED;
    return launch_encode(*dst, src_f16, n_tokens, src_token_stride, seq_ids, positions, seq_id,
                         pos0, static_cast<cudaStream_t>(stream));
}

tq_status tq_encode_kv(const tq_cache *k, const tq_cache *v, const void *k_src_f16,
                       const void *v_src_f16, int64_t n_tokens, int64_t k_token_stride,
                       int64_t v_token_stride, const int32_t *seq_ids, const int32_t *positions,
                       int32_t seq_id, int64_t pos0, void *stream) {
    tq_status st = validate_cache(k);
    if (st != TQ_OK) return st;
    st = validate_cache(v);
    if (st != TQ_OK) return st;
    if (n_tokens < 0) return TQ_ERR_INVALID_ARGUMENT;
    if (n_tokens == 0) return TQ_OK;
    if (!k_src_f16 || reinterpret_cast<uintptr_t>(k_src_f16) % 16 || !v_src_f16 ||
        reinterpret_cast<uintptr_t>(v_src_f16) % 16)
        return TQ_ERR_INVALID_ARGUMENT;
    if (k_token_stride < (int64_t)k->n_kv_heads * k->head_dim || k_token_stride % 8 ||
        v_token_stride < (int64_t)v->n_kv_heads * v->head_dim || v_token_stride % 8)
        return TQ_ERR_INVALID_ARGUMENT;
    if (!positions && pos0 < 0) return TQ_ERR_INVALID_ARGUMENT;
    if (!seq_ids && (seq_id < 0 || seq_id >= k->n_seqs || seq_id >= v->n_seqs))
        return TQ_ERR_INVALID_ARGUMENT;
    if (n_tokens > (int64_t)1 << 40) return TQ_ERR_UNSUPPORTED;
    return launch_encode_kv(*k, *v, k_src_f16, v_src_f16, n_tokens, k_token_stride,
                            v_token_stride, seq_ids, positions, seq_id, pos0,
                            static_cast<cudaStream_t>(stream));
}

tq_status tq_decode(const tq_cache *src, int32_t seq_id, int64_t pos0, int64_t n_tokens,
                    float *dst, void *stream) {
    tq_status st = validate_cache(src);
    if (st != TQ_OK) return st;
    if (n_tokens < 0 || pos0 < 0 || seq_id < 0 || seq_id >= src->n_seqs)
        return TQ_ERR_INVALID_ARGUMENT;
    if (n_tokens == 0) return TQ_OK;
    if (!dst || reinterpret_cast<uintptr_t>(dst) % 16) return TQ_ERR_INVALID_ARGUMENT;
    return launch_decode(*src, seq_id, pos0, n_tokens, dst, static_cast<cudaStream_t>(stream));
}

size_t tq_attn_workspace_bytes(int n_seqs, int n_q_heads, int head_dim, int64_t max_seq_len) {
    if (n_seqs < 1 || n_q_heads < 1 || head_dim < kBlock || head_dim % kBlock || max_seq_len < 0)
        return 0;
    return attn_workspace_bytes(n_seqs, n_q_heads, head_dim, max_seq_len, device_sm_count());
}

}  // extern "C"

namespace tq {

tq_status check_attn_args(const tq_cache *k, const tq_cache *v, const void *q_f16, int n_seqs,
                          int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len,
                          float softmax_scale, const float *out, float *scale_out) {
    tq_status st = validate_cache(k);
    if (st != TQ_OK) return st;
    st = validate_cache(v);
    if (st != TQ_OK) return st;
    if (k->n_kv_heads != v->n_kv_heads || k->head_dim != v->head_dim)
        return TQ_ERR_INVALID_ARGUMENT;
    if (n_seqs < 1 || n_seqs > k->n_seqs || n_seqs > v->n_seqs) return TQ_ERR_INVALID_ARGUMENT;
    if (n_q_heads < 1 || n_q_heads % k->n_kv_heads) return TQ_ERR_INVALID_ARGUMENT;
    if (n_q_heads / k->n_kv_heads > 16 || n_q_heads > 128) return TQ_ERR_UNSUPPORTED;
    if (max_seq_len < 0 || max_seq_len > ((int64_t)1 << 31) - 1) return TQ_ERR_INVALID_ARGUMENT;
    if (!q_f16 || !seq_lens || !out) return TQ_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(q_f16) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
        return TQ_ERR_INVALID_ARGUMENT;
    if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale)) return TQ_ERR_INVALID_ARGUMENT;
    *scale_out = softmax_scale == 0.0f ? 1.0f / std::sqrt((float)k->head_dim) : softmax_scale;
    return TQ_OK;
}

}  // namespace tq

namespace {
// tq_attn_decode and tq_attn_decode_append: the shared checks, then the workspace's.
tq_status attn_decode_checked(const tq_cache *k, const tq_cache *v, const void *q_f16, int n_seqs,
                              int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len,
                              float softmax_scale, float *out, void *workspace, size_t ws_bytes,
                              void *stream, const void *k_new, const void *v_new) {
    float scale = 0.0f;
    tq_status st = check_attn_args(k, v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len,
                                   softmax_scale, out, &scale);
    if (st != TQ_OK) return st;
    size_t need = tq_attn_workspace_bytes(n_seqs, n_q_heads, k->head_dim, max_seq_len);
    if (need > 0 && (!workspace || ws_bytes < need)) return TQ_ERR_WORKSPACE_TOO_SMALL;
    if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16) return TQ_ERR_INVALID_ARGUMENT;
    return launch_attn(*k, *v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len, scale, out,
                       workspace, ws_bytes, static_cast<cudaStream_t>(stream), k_new, v_new);
}
}  // namespace

extern "C" {

tq_status tq_attn_decode_append(const tq_cache *k, const tq_cache *v, const void *k_new_f16,
                                const void *v_new_f16, const void *q_f16, int n_seqs,
                                int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len,
                                float softmax_scale, float *out, void *workspace,
                                size_t ws_bytes, void *stream) {
    if (!k_new_f16 || reinterpret_cast<uintptr_t>(k_new_f16) % 16 || !v_new_f16 ||
        reinterpret_cast<uintptr_t>(v_new_f16) % 16)
        return TQ_ERR_INVALID_ARGUMENT;
    return attn_decode_checked(k, v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len,
                               softmax_scale, out, workspace, ws_bytes, stream, k_new_f16,
                               v_new_f16);
}

tq_status tq_attn_decode(const tq_cache *k, const tq_cache *v, const void *q_f16, int n_seqs,
                         int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len,
                         float softmax_scale, float *out, void *workspace, size_t ws_bytes,
                         void *stream) {
    return attn_decode_checked(k, v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len,
                               softmax_scale, out, workspace, ws_bytes, stream, nullptr, nullptr);
}

tq_status tq_attn_prefill(const tq_cache *k, const tq_cache *v, const void *q_f16,
                          int32_t seq_id, int64_t pos0, int64_t n_q, int n_q_heads,
                          float softmax_scale, float *out, void *stream) {
    tq_status st = validate_cache(k);
    if (st != TQ_OK) return st;
    st = validate_cache(v);
    if (st != TQ_OK) return st;
    if (k->n_kv_heads != v->n_kv_heads || k->head_dim != v->head_dim)
        return TQ_ERR_INVALID_ARGUMENT;
    if (seq_id < 0 || seq_id >= k->n_seqs || seq_id >= v->n_seqs) return TQ_ERR_INVALID_ARGUMENT;
    if (pos0 < 0 || n_q < 0 || pos0 > (((int64_t)1 << 40) - n_q)) return TQ_ERR_INVALID_ARGUMENT;
    if (n_q_heads < 1 || n_q_heads % k->n_kv_heads) return TQ_ERR_INVALID_ARGUMENT;
    if (!(softmax_scale >= 0.0f) || std::isinf(softmax_scale)) return TQ_ERR_INVALID_ARGUMENT;
    if (!prefill_supported(*k, *v, n_q_heads)) return TQ_ERR_UNSUPPORTED;
    if (n_q == 0) return TQ_OK;   // empty chunk: q and out may be null
    if (!q_f16 || !out) return TQ_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(q_f16) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
        return TQ_ERR_INVALID_ARGUMENT;
    if (softmax_scale == 0.0f) softmax_scale = 1.0f / std::sqrt((float)k->head_dim);
    return launch_prefill(*k, *v, q_f16, seq_id, pos0, n_q, n_q_heads, softmax_scale, out,
                          static_cast<cudaStream_t>(stream));
}

tq_status tq_device_status(void *stream, int32_t *status_out) {
    if (!status_out) return TQ_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t host = 0, zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaMemcpyFromSymbolAsync(&host, g_status, sizeof host, 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return TQ_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return TQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
    *status_out = host;
    return TQ_OK;
}

#if defined(TQ_TRACE_PHASES)
// Traced library only: copy the phase stamps (2 * kTraceCtas x kTracePoints u64) to host
// memory, or clear them.  Not part of the product ABI.
TQ_API int tq_phase_trace_read(void *host, size_t bytes) {
    return (int)cudaMemcpyFromSymbol(host, g_phase_trace, bytes);
}
TQ_API int tq_phase_trace_clear(void) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_phase_trace) != cudaSuccess) return 1;
    return (int)cudaMemset(p, 0, sizeof g_phase_trace);
}
#endif

const char *tq_status_str(int status) {
    switch (status) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_INVALID_ARGUMENT: return "TQ_ERR_INVALID_ARGUMENT";
        case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED";
        case TQ_ERR_NOT_INITIALIZED: return "TQ_ERR_NOT_INITIALIZED";
        case TQ_ERR_WORKSPACE_TOO_SMALL: return "TQ_ERR_WORKSPACE_TOO_SMALL";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA";
        case TQ_ERR_DEVICE_TIMEOUT: return "TQ_ERR_DEVICE_TIMEOUT";
        case TQ_ERR_OUT_OF_RANGE: return "TQ_ERR_OUT_OF_RANGE";
        default: return "TQ_UNKNOWN_STATUS";
    }
}

}  // extern "C"
