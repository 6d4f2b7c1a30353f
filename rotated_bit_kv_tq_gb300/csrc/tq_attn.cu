// tq_attn.cu -- fused single-token decode attention over the packed cache
// (CUDA-core, fp32 arithmetic).
//
// kenji.blog inference-engine article, section 8: out = softmax(q K^T / sqrt(d)) V over
// the cached positions; TinyLLaMA article 4.3: query head h reads KV head floor(h / G).
// "llama.cpp に TurboQuant を実装", "Current implementation and what's next": the
// dequantisation is fused into the attention kernel so that no FP16 key or value is
// materialised.  Because W/sqrt(128) is orthonormal and symmetric,
//     q . k_hat = |k| (W q / sqrt(128)) . c(codes_k)
//     sum_t p_t v_hat_t = (1/sqrt(128)) W sum_t p_t |v_t| c(codes_v)
// so q is rotated once per call, scores and the value sum run in the rotated domain,
// and one inverse FWHT per output block finishes the job.
//
// Split-K: the context of every sequence is cut into equal token ranges, one CTA per
// (range, sequence).  Each CTA streams its packed K/V rows through shared memory in
// tiles, keeps an online softmax (running max m, sum l) and a rotated-domain value
// accumulator per query head, and writes (acc, m, l) to the workspace.  A second kernel
// merges the ranges with the usual log-sum-exp rescaling and applies the inverse FWHT.
#include <cmath>

#include "tq_internal.cuh"
#include "tq_simd.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMinSplitTokens = 16;       // fewest tokens per split
constexpr int kMaxG = 8;              // query heads per KV head handled in registers
constexpr int kMaxNb = 2;             // 128-blocks per head handled in registers
constexpr int kTileBudget = 96 * 1024;  // shared bytes for one K+V tile

struct AttnParams {
    CacheView kc, vc;
    const __half *q;
    const int32_t *seq_lens;
    float *part;   // [n_seqs][n_splits][Hq][part_stride(D)]
    float *out;    // [n_seqs][Hq][D]
    float scale;   // softmax scale (1/sqrt(D) by default)
    int64_t max_len;
    int32_t n_q_heads, n_kv_heads, group, head_dim, nb;
    int32_t n_splits, tokens_per_split, tile_tokens;
};

struct SplitPlan {
    int n_splits;
    int tokens_per_split;
};

SplitPlan plan_splits(int n_seqs, int head_dim, int64_t max_len, int sm_count) {
    SplitPlan pl;
    (void)head_dim;
    // One wave of one CTA per SM if every sequence had max_len tokens.  The host knows only
    // the longest length: in a batch of mixed lengths the trailing splits of the shorter
    // sequences are empty (those CTAs end at once), so long splits would leave a tail of a
    // few long CTAs.  When a CTA would get more than kLongSplit tokens of a batch, the splits
    // are cut to a quarter (at least kMinSplit tokens): several waves of short CTAs, which
    // the scheduler balances.
    constexpr int64_t kLongSplit = 2048, kMinSplit = 1024;
    const int64_t per_seq = max64(1, (sm_count + n_seqs - 1) / n_seqs);
    int64_t tps = (max64(max_len, 1) + per_seq - 1) / per_seq;
    if (n_seqs > 1 && tps > kLongSplit) tps = max64(kMinSplit, (tps + 3) / 4);
    // no rounding of tps: a split may start at any row (tiles and page runs do not care),
    // and rounding up would leave SMs idle (32,896 tokens: 148 CTAs of 224 instead of 152
    // of 217)
    if (tps < kMinSplitTokens) tps = kMinSplitTokens;
    pl.tokens_per_split = (int)tps;
    pl.n_splits = (int)max64(1, (max_len + tps - 1) / tps);
    // one sequence: whole clusters of splits (a trailing split with no tokens writes neutral
    // partials); a batch runs without clusters
    if (n_seqs == 1)
        pl.n_splits = (pl.n_splits + kClusterSplits - 1) / kClusterSplits * kClusterSplits;
    return pl;
}

// Rotate the query of one (head, block) pair held by a warp, four values per lane:
// returns the lane's four values of W q_b (canonical butterfly order).
__device__ __forceinline__ void warp_fwht4(float v[4], int lane) {
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
            v[e] = upper ? o - v[e] : v[e] + o;
        }
    }
}

// Code of value i of a packed block (layout of tq.h).
template <int TYPE>
__device__ __forceinline__ int code_of(const uint8_t *b, int i) {
    const int j = i & 15;
    const int lb = 32 * (i >> 4) + 4 * (j & 7) + 2 * (j >> 3);
    int code = (b[2 + (lb >> 3)] >> (lb & 7)) & 3;
    if (TYPE == TQ_TURBO3) {
        const int jv = i & 31;
        const int hb = 32 * (i >> 5) + 4 * (jv & 7) + (jv >> 3);
        code |= ((b[34 + (hb >> 3)] >> (hb & 7)) & 1) << 2;
    }
    return code;
}

__device__ __forceinline__ float norm_of(const uint8_t *b) {
    return __half2float(__ushort_as_half((uint16_t)(b[0] | (b[1] << 8))));
}

// Copy `bytes` bytes of one packed row (2-byte aligned, 16-byte when possible) into smem.
__device__ __forceinline__ void copy_row(uint8_t *dst, const uint8_t *src, int bytes, int lane) {
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && (bytes & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
        for (int c = lane; c < bytes / 16; c += 32)
            reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
    } else {
        for (int c = lane; c < bytes / 2; c += 32)
            reinterpret_cast<uint16_t *>(dst)[c] = reinterpret_cast<const uint16_t *>(src)[c];
    }
}

template <int TK, int TV>
__global__ void __launch_bounds__(kThreads, 1) attn_partial_kernel(const AttnParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int Hq = p.n_q_heads, D = p.head_dim, G = p.group, Hkv = p.n_kv_heads;
    const int TT = p.tile_tokens;
    const int Rk = p.kc.row_bytes, Rv = p.vc.row_bytes;
    const int Rk16 = (Rk + 15) & ~15, Rv16 = (Rv + 15) & ~15;
    float *qs = reinterpret_cast<float *>(smem);                 // [Hq][D]
    float *S = qs + Hq * D;                                      // [Hq][TT]
    float *m_run = S + Hq * TT;                                  // [Hq]
    float *l_run = m_run + Hq;                                   // [Hq]
    float *alpha = l_run + Hq;                                   // [Hq]
    float *ck = alpha + Hq;                                      // [8]
    float *cv = ck + 8;                                          // [8]
    uint8_t *kt = reinterpret_cast<uint8_t *>(cv + 8);           // [TT][Rk16]
    kt = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(kt) + 15) & ~uintptr_t(15));
    uint8_t *vt = kt + TT * Rk16;                                // [TT][Rv16]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seq = blockIdx.y, split = blockIdx.x;
    int64_t len = p.seq_lens[seq];
    if (len < 0 || len > p.max_len) {
        if (tid == 0) record_error(TQ_ERR_OUT_OF_RANGE);
        len = len < 0 ? 0 : p.max_len;
    }
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    const int64_t t_end = min64(len, t_begin + p.tokens_per_split);

    if (tid < 8) {
        ck[tid] = tid < (1 << TK) ? c_codebook[cb_index(TK)].centroid[tid] : 0.f;
        cv[tid] = tid < (1 << TV) ? c_codebook[cb_index(TV)].centroid[tid] : 0.f;
    }
    for (int h = tid; h < Hq; h += kThreads) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
    }
    // ---- rotate q once: qs = W q_b * (scale / sqrt(128)) per (head, block)
    const float qscale = p.scale * kInvSqrt128;
    for (int hb = warp; hb < Hq * p.nb; hb += kWarps) {
        const int h = hb / p.nb, b = hb - h * p.nb;
        const __half *qp = p.q + ((int64_t)seq * Hq + h) * D + b * kBlock + 4 * lane;
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __half2float(qp[e]);
        apply_signs4(v, p.kc, 4 * lane);   // rotation W D of the K cache
        warp_fwht4(v, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) qs[h * D + b * kBlock + 4 * lane + e] = v[e] * qscale;
    }

    // V accumulators: warp w owns KV heads g = w, w + 8, ...; lane owns values
    // 4*lane .. 4*lane+3 of every block.  acc[h_local * nb + b][e].
    float acc[kMaxG][kMaxNb][4];

    for (int g0 = 0; g0 < Hkv; g0 += kWarps) {
        const int g = g0 + warp;  // this warp's KV head in this pass
#pragma unroll
        for (int a = 0; a < kMaxG; ++a)
#pragma unroll
            for (int b = 0; b < kMaxNb; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[a][b][e] = 0.f;
        // (heads of other passes keep running statistics in m_run / l_run, but the
        //  accumulators are per pass, so passes re-stream the tiles: Hkv <= 8 is one pass)
        __syncthreads();
        for (int64_t t0 = t_begin; t0 < t_end; t0 += TT) {
            const int nt = (int)min64(TT, t_end - t0);
            // ---- stage K and V rows
            for (int r = warp; r < nt; r += kWarps) {
                const uint8_t *krow = row_ptr(p.kc, seq, t0 + r);
                const uint8_t *vrow = row_ptr(p.vc, seq, t0 + r);
                if (krow) copy_row(kt + r * Rk16, krow, Rk, lane);
                if (vrow) copy_row(vt + r * Rv16, vrow, Rv, lane);
            }
            __syncthreads();
            // ---- scores: thread <-> (KV head gg, token t); only this pass's heads
            const int gpass = min(kWarps, Hkv - g0);
            for (int pi = tid; pi < gpass * TT; pi += kThreads) {
                const int gg = g0 + pi / TT, t = pi % TT;
                float sc[kMaxG];
#pragma unroll
                for (int h = 0; h < kMaxG; ++h) sc[h] = 0.f;
                if (t < nt) {
                    for (int b = 0; b < p.nb; ++b) {
                        const uint8_t *blk = kt + t * Rk16 + (gg * p.nb + b) * block_bytes(TK);
                        float dot[kMaxG];
#pragma unroll
                        for (int h = 0; h < kMaxG; ++h) dot[h] = 0.f;
                        const float *qb = qs + (gg * G) * D + b * kBlock;
                        for (int i = 0; i < kBlock; ++i) {
                            const float c = ck[code_of<TK>(blk, i)];
#pragma unroll
                            for (int h = 0; h < kMaxG; ++h)
                                if (h < G) dot[h] = fmaf(c, qb[h * D + i], dot[h]);
                        }
                        const float n = norm_of(blk);
#pragma unroll
                        for (int h = 0; h < kMaxG; ++h) sc[h] = fmaf(n, dot[h], sc[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < kMaxG; ++h)
                    if (h < G) S[(gg * G + h) * TT + t] = t < nt ? sc[h] : -INFINITY;
            }
            __syncthreads();
            // ---- online softmax, warp per query head of this pass
            for (int hh = warp; hh < gpass * G; hh += kWarps) {
                const int h = g0 * G + hh;
                float mx = -INFINITY;
                for (int t = lane; t < TT; t += 32) mx = fmaxf(mx, S[h * TT + t]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = m_run[h];
                const float m_new = fmaxf(m_old, mx);
                float sum = 0.f;
                for (int t = lane; t < TT; t += 32) {
                    const float s = S[h * TT + t];
                    const float pr = (s == -INFINITY) ? 0.f : __expf(s - m_new);
                    S[h * TT + t] = pr;
                    sum += pr;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                __syncwarp();
                if (lane == 0) {
                    const float al = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                    alpha[h] = al;
                    m_run[h] = m_new;
                    l_run[h] = l_run[h] * al + sum;
                }
            }
            __syncthreads();
            // ---- rotated-domain value accumulation
            if (g < Hkv) {
#pragma unroll
                for (int hl = 0; hl < kMaxG; ++hl) {
                    if (hl < G) {
                        const float al = alpha[g * G + hl];
#pragma unroll
                        for (int b = 0; b < kMaxNb; ++b)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[hl][b][e] *= al;
                    }
                }
                for (int t = 0; t < nt; ++t) {
#pragma unroll
                    for (int b = 0; b < kMaxNb; ++b) {
                        if (b >= p.nb) break;
                        const uint8_t *blk = vt + t * Rv16 + (g * p.nb + b) * block_bytes(TV);
                        const float n = norm_of(blk);
                        float c[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) c[e] = cv[code_of<TV>(blk, 4 * lane + e)];
#pragma unroll
                        for (int hl = 0; hl < kMaxG; ++hl) {
                            if (hl < G) {
                                const float w = S[(g * G + hl) * TT + t] * n;
#pragma unroll
                                for (int e = 0; e < 4; ++e) acc[hl][b][e] = fmaf(w, c[e], acc[hl][b][e]);
                            }
                        }
                    }
                }
            }
            __syncthreads();
        }
        // ---- write this pass's partials
        if (g < Hkv) {
#pragma unroll
            for (int hl = 0; hl < kMaxG; ++hl) {
                if (hl >= G) break;
                const int h = g * G + hl;
                float *dst = p.part + (((int64_t)seq * p.n_splits + split) * Hq + h) * part_stride(D);
#pragma unroll
                for (int b = 0; b < kMaxNb; ++b) {
                    if (b >= p.nb) break;
                    float *d = dst + b * kBlock + 4 * lane;
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[e] = acc[hl][b][e];
                }
                if (lane == 0) {
                    dst[D] = m_run[h];
                    dst[D + 1] = l_run[h];
                }
            }
        }
    }
}

// Merge the split partials of one (sequence, head, 128-block) and undo the rotation.
// Warps take splits round-robin, lanes take four coordinates each (float4 loads of the
// partial rows), the eight warp sums meet in shared memory, and one warp applies the
// inverse FWHT with shuffles.
// Rows of split partials each warp keeps in flight at once.
constexpr int kMergeRows = 24;

__global__ void __launch_bounds__(256) attn_merge_kernel(const AttnParams p) {
    const int trace_slot = kTraceCtas + blockIdx.y * gridDim.x + blockIdx.x;   // phase trace only
    (void)trace_slot;
    if (threadIdx.x == 0) TQ_PHASE(trace_slot, 0);
    __shared__ float red_m[8], red_l[8];
    __shared__ float4 red_o[8][32];
    const int h = blockIdx.x, seq = blockIdx.y, b = blockIdx.z, D = p.head_dim;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *base = p.part + ((int64_t)seq * p.n_splits * p.n_q_heads + h) * part_stride(D);
    const int64_t sstride = (int64_t)p.n_q_heads * part_stride(D);
    // the rows of this warp's first round into L2 while the partial kernel finishes
    if (lane < kMergeRows && warp + 8 * lane < p.n_splits) {
        const float *row = base + (warp + 8 * lane) * sstride;
        l2_prefetch(row + b * kBlock, kBlock * sizeof(float));
        l2_prefetch(row + D, 4 * sizeof(float));
    }
    // launched as a programmatic dependent of the partial kernel: wait for its results
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) TQ_PHASE(trace_slot, 1);
    // One pass: warp w takes splits w, w + 8, ...; all rows of a round are loaded before
    // any is used, and the warp's running maximum rescales what it has summed so far.
    float M = -INFINITY, lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = warp; s0 < p.n_splits; s0 += 8 * kMergeRows) {
        float2 ml[kMergeRows];
        float4 v[kMergeRows];
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u) {
            const int s = s0 + 8 * u;
            if (s < p.n_splits) {
                const float *row = base + s * sstride;
                ml[u] = *reinterpret_cast<const float2 *>(row + D);
                v[u] = *reinterpret_cast<const float4 *>(row + b * kBlock + 4 * lane);
            } else {
                ml[u] = make_float2(-INFINITY, 0.f);
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float mc = M;
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u) mc = fmaxf(mc, ml[u].x);
        if (mc != M) {   // new maximum: rescale (M = -inf means nothing was summed yet)
            const float r = M == -INFINITY ? 0.f : __expf(M - mc);
            lsum *= r;
            acc.x *= r;
            acc.y *= r;
            acc.z *= r;
            acc.w *= r;
            M = mc;
        }
#pragma unroll
        for (int u = 0; u < kMergeRows; ++u) {
            const float wgt = (ml[u].x == -INFINITY) ? 0.f : __expf(ml[u].x - M);
            lsum += wgt * ml[u].y;
            acc.x = fmaf(wgt, v[u].x, acc.x);
            acc.y = fmaf(wgt, v[u].y, acc.y);
            acc.z = fmaf(wgt, v[u].z, acc.z);
            acc.w = fmaf(wgt, v[u].w, acc.w);
        }
    }
    red_o[warp][lane] = acc;
    if (threadIdx.x == 0 && acc.x != acc.x + 1.0f) TQ_PHASE(trace_slot, 2);   // loads consumed
    if (lane == 0) {
        red_m[warp] = M;
        red_l[warp] = lsum;
    }
    __syncthreads();
    if (warp != 0) return;
    float mx = red_m[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red_m[w]);
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const float mw = red_m[w];
        const float wgt = mw == -INFINITY ? 0.f : __expf(mw - mx);
        const float4 a = red_o[w][lane];
        v[0] = fmaf(wgt, a.x, v[0]);
        v[1] = fmaf(wgt, a.y, v[1]);
        v[2] = fmaf(wgt, a.z, v[2]);
        v[3] = fmaf(wgt, a.w, v[3]);
        L = fmaf(wgt, red_l[w], L);
    }
    const float inv = L > 0.f ? kInvSqrt128 / L : 0.f;
    // inverse rotation (1/sqrt(128)) W o_b, values 4*lane .. 4*lane+3
    warp_fwht4(v, lane);
    apply_signs4(v, p.vc, 4 * lane);     // inverse D W of the V cache
    float4 o4 = make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
    *reinterpret_cast<float4 *>(p.out + ((int64_t)seq * p.n_q_heads + h) * D + b * kBlock + 4 * lane) = o4;
    if (lane == 0) TQ_PHASE(trace_slot, 3);
}

// Few partial rows per head (batches): one warp merges one (head, sequence, block).  Lane r
// loads the (m, l) of row r and every lane the float4 of its coordinates of every row, all in
// one round; the warp reduces with shuffles and applies the inverse FWHT itself.
constexpr int kMergeWarpRows = 16;   // rows one warp merges in its single round of loads

__global__ void __launch_bounds__(256) attn_merge_warp_kernel(const AttnParams p) {
    const int trace_slot = kTraceCtas + blockIdx.y * gridDim.x + blockIdx.x;   // phase trace only
    (void)trace_slot;
    if (threadIdx.x == 0) TQ_PHASE(trace_slot, 0);
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);   // (head, block) of sequence blockIdx.y
    const int D = p.head_dim, Hq = p.n_q_heads;
    const int b = item % p.nb, h = item / p.nb;
    const int64_t seq = blockIdx.y;
    const int R = p.n_splits;
    const float *base = p.part + (seq * R * Hq + h) * part_stride(D);
    const int64_t sstride = (int64_t)Hq * part_stride(D);
    // this warp's rows into L2 while the partial kernel finishes
    if (item < Hq * p.nb && lane < R) {
        const float *row = base + lane * sstride;
        l2_prefetch(row + b * kBlock, kBlock * sizeof(float));
        l2_prefetch(row + D, 4 * sizeof(float));
    }
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) TQ_PHASE(trace_slot, 1);
    if (item >= Hq * p.nb) return;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < R) ml = *reinterpret_cast<const float2 *>(base + lane * sstride + D);
    float4 v[kMergeWarpRows];
#pragma unroll
    for (int r = 0; r < kMergeWarpRows; ++r)
        v[r] = r < R ? *reinterpret_cast<const float4 *>(base + r * sstride + b * kBlock + 4 * lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    float M = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = ml.x == -INFINITY ? 0.f : __expf(ml.x - M);
    float L = w * ml.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < kMergeWarpRows; ++r) {
        const float wr = __shfl_sync(0xffffffffu, w, r);
        o4[0] = fmaf(wr, v[r].x, o4[0]);
        o4[1] = fmaf(wr, v[r].y, o4[1]);
        o4[2] = fmaf(wr, v[r].z, o4[2]);
        o4[3] = fmaf(wr, v[r].w, o4[3]);
    }
    if (threadIdx.x == 0 && o4[0] != o4[0] + 1.0f) TQ_PHASE(trace_slot, 2);   // loads consumed
    const float inv = L > 0.f ? kInvSqrt128 / L : 0.f;
    warp_fwht4(o4, lane);                    // inverse rotation (1/sqrt(128)) W o_b
    apply_signs4(o4, p.vc, 4 * lane);        // inverse D W of the V cache
    *reinterpret_cast<float4 *>(p.out + (seq * Hq + h) * D + b * kBlock + 4 * lane) =
        make_float4(o4[0] * inv, o4[1] * inv, o4[2] * inv, o4[3] * inv);
    if (lane == 0) TQ_PHASE(trace_slot, 3);
}

size_t partial_smem(const AttnParams &p) {
    const int Rk16 = (p.kc.row_bytes + 15) & ~15, Rv16 = (p.vc.row_bytes + 15) & ~15;
    return sizeof(float) * ((size_t)p.n_q_heads * p.head_dim + (size_t)p.n_q_heads * p.tile_tokens +
                            3 * (size_t)p.n_q_heads + 16) +
           16 + (size_t)p.tile_tokens * (Rk16 + Rv16);
}

tq_status launch_merge(const AttnParams &p, int n_seqs, cudaStream_t stream) {
    if (p.n_splits <= kMergeWarpRows) {   // one warp per (head, sequence, block)
        PdlConfig lc(dim3((unsigned)((p.n_q_heads * p.nb + 7) / 8), (unsigned)n_seqs), dim3(256), 0,
                     stream);
        return check_cuda(cudaLaunchKernelEx(&lc.cfg, attn_merge_warp_kernel, p));
    }
    PdlConfig lc(dim3(p.n_q_heads, n_seqs, p.nb), dim3(256), 0, stream);
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, attn_merge_kernel, p));
}

template <int TK, int TV>
tq_status launch_attn_t(const AttnParams &p, int n_seqs, cudaStream_t stream) {
    const size_t smem = partial_smem(p);
    if (smem > 220 * 1024) return TQ_ERR_UNSUPPORTED;
    const tq_status st = kernel_setup(reinterpret_cast<const void *>(attn_partial_kernel<TK, TV>),
                                      (int)smem, kThreads, nullptr);
    if (st != TQ_OK) return st;
    attn_partial_kernel<TK, TV><<<dim3(p.n_splits, n_seqs), kThreads, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return TQ_ERR_CUDA;
    return launch_merge(p, n_seqs, stream);
}

}  // namespace

size_t attn_workspace_bytes(int n_seqs, int n_q_heads, int head_dim, int64_t max_seq_len,
                            int sm_count) {
    const SplitPlan pl = plan_splits(n_seqs, head_dim, max_seq_len, sm_count);
    const size_t rows = sizeof(float) * (size_t)n_seqs * pl.n_splits * n_q_heads * part_stride(head_dim);
    // the grid merge of one sequence keeps every value with a 32-bit tag (64-bit words)
    const bool grid = n_seqs == 1 && pl.n_splits <= std::min(sm_count, kGridMergeMaxCtas);
    return kGridBarrierBytes + (grid ? 2 : 1) * rows;
}

tq_status launch_attn(const tq_cache &k, const tq_cache &v, const void *q, int n_seqs,
                      int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len, float scale,
                      float *out, void *ws, size_t ws_bytes, cudaStream_t stream,
                      const void *k_new, const void *v_new) {
    AttnParams p;
    p.kc = make_view(k);
    p.vc = make_view(v);
    p.q = static_cast<const __half *>(q);
    p.seq_lens = seq_lens;
    // the grid-merge area, then the partial rows
    p.part = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kGridBarrierBytes);
    p.out = out;
    p.scale = scale;
    p.max_len = max_seq_len;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = k.n_kv_heads;
    p.group = n_q_heads / k.n_kv_heads;
    p.head_dim = k.head_dim;
    p.nb = k.head_dim / kBlock;
    if ((size_t)n_q_heads * k.head_dim > 16384) return TQ_ERR_UNSUPPORTED;
    const SplitPlan pl = plan_splits(n_seqs, k.head_dim, max_seq_len, device_sm_count());
    p.n_splits = pl.n_splits;
    p.tokens_per_split = pl.tokens_per_split;
    const int Rk16 = (p.kc.row_bytes + 15) & ~15, Rv16 = (p.vc.row_bytes + 15) & ~15;
    p.tile_tokens = std::max(1, std::min(32, kTileBudget / (Rk16 + Rv16)));
    if (ws_bytes < attn_workspace_bytes(n_seqs, n_q_heads, k.head_dim, max_seq_len,
                                        device_sm_count()))
        return TQ_ERR_WORKSPACE_TOO_SMALL;
    if (attn_mma_supported(k, v, n_q_heads)) {
        // One wave of CTAs merges its own partials after a grid barrier (no merge kernel, no
        // kernel boundary before the output); otherwise a single sequence pairs its splits
        // in clusters, and the merge kernel follows.
        const bool grid = grid_merge_fits(n_seqs, p.n_splits);
        const int cluster = grid ? 1 : n_seqs == 1 ? kClusterSplits : 1;
        tq_status st = launch_attn_mma(k, v, q, n_seqs, n_q_heads, seq_lens, max_seq_len, scale,
                                       p.part, p.n_splits, p.tokens_per_split, cluster, k_new,
                                       v_new, grid ? out : nullptr,
                                       grid ? static_cast<uint64_t *>(ws) : nullptr, stream);
        if (st != TQ_OK || grid) return st;
        AttnParams pm = p;
        pm.n_splits = p.n_splits / cluster;   // one partial row per cluster
        return launch_merge(pm, n_seqs, stream);
    }
    if (p.group > kMaxG || p.nb > kMaxNb) return TQ_ERR_UNSUPPORTED;
    if (k_new) {   // the fp32 kernel reads the caches only: append in a launch of its own
        tq_status st = launch_append(k, v, k_new, v_new, seq_lens, n_seqs, stream);
        if (st != TQ_OK) return st;
    }
    const int tk = k.type, tv = v.type;
    if (tk == TQ_TURBO3 && tv == TQ_TURBO3) return launch_attn_t<3, 3>(p, n_seqs, stream);
    if (tk == TQ_TURBO2 && tv == TQ_TURBO2) return launch_attn_t<2, 2>(p, n_seqs, stream);
    if (tk == TQ_TURBO3 && tv == TQ_TURBO2) return launch_attn_t<3, 2>(p, n_seqs, stream);
    return launch_attn_t<2, 3>(p, n_seqs, stream);
}

}  // namespace tq

// ---------------------------------------------------------------------------------
// Allocation-free variant of tq_attn_decode.  The split partials live in a fixed
// file-scope device array instead of a caller-provided workspace.
// ---------------------------------------------------------------------------------
namespace tq {
namespace {

constexpr size_t kStaticScratchBytes = TQ_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

// Device address of g_attn_scratch in the current device's context.  It is looked up on
// every call rather than cached: after cudaDeviceReset, or in another context on the same
// device, the library's device code is loaded anew and the array may move.  (The host-side
// name of the array is only a stand-in and must never reach a kernel.)
tq_status scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
    *out = p;
    return TQ_OK;
}

}  // namespace
}  // namespace tq

extern "C" tq_status tq_attn_decode_noalloc(const tq_cache *k, const tq_cache *v,
                                             const void *q_f16, int n_seqs, int n_q_heads,
                                             const int32_t *seq_lens, int64_t max_seq_len,
                                             float softmax_scale, float *out, void *stream) {
    using namespace tq;
    float scale = 0.0f;
    tq_status st = check_attn_args(k, v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len,
                                   softmax_scale, out, &scale);
    if (st != TQ_OK) return st;
    // The shape must fit the fixed array; larger shapes are refused, never truncated.
    const size_t need = attn_workspace_bytes(n_seqs, n_q_heads, k->head_dim, max_seq_len,
                                             device_sm_count());
    if (need > kStaticScratchBytes) return TQ_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != TQ_OK) return st;
    // Every partial the merge reads is written by the same call first, so nothing in
    // the array needs clearing between calls.
    return launch_attn(*k, *v, q_f16, n_seqs, n_q_heads, seq_lens, max_seq_len, scale, out,
                       scratch, kStaticScratchBytes, static_cast<cudaStream_t>(stream));
}
