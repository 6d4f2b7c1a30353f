// tq_attn_mma.cu -- decode attention over the packed cache with the dequantisation fused
// into tensor-core fragments.
//
// Same mathematics as tq_attn.cu (rotated domain, split-K, online softmax; kenji.blog
// inference-engine article section 8, TinyLLaMA article 4.3; "llama.cpp に TurboQuant を
// 実装", "Current implementation and what's next": dequantise inside the attention kernel,
// never materialise FP16 K or V).  What changes is where the multiply-adds run.
//
// Why tensor cores here.  At GQA group G every 128-value block costs G*128 multiply-adds on
// the K side and G*128 on the V side, plus the unpacking of its codes.  On CUDA cores that
// is >= 4 FMAs + ~6 unpack instructions per value at G = 4, while the HBM budget of a
// GB300 SM is ~2.1 issue slots per packed value (23 B/clk/SM at 3/8 B per value), so the
// fp32 design cannot approach the memory roofline.  Here each value is unpacked once into
// an fp16 MMA operand with four byte-permute (prmt) table lookups per 8 values and the
// products run on mma.sync.m16n8k16 (fp16 x fp16 -> fp32 accumulate):
//   scores   S^T[token, head]  = C_k[token, coord] . Qr^T[coord, head]   (M = 16 tokens)
//   values   O^T[coord, head] += C_v^T[coord, token] . (p |v|)^T[token, head]
// The operands are formed in registers, so nothing but the packed rows passes through
// shared memory; the probabilities move from the score accumulators to the value
// operand with movmatrix (an 8x8 transpose across the warp).
//
// Operand precision: the rotated query is held as an fp16 pair q~ = hi + lo (lo the fp16
// rounding of the remainder), and the centroid tables are scaled so that their fp16 values
// are nearly exact (Codebook::h_scale, divided out in fp32).  With at most four query heads
// per KV head the low halves sit in the four otherwise empty columns of the score MMA, so
// they cost no extra MMA; with more, a second MMA per k-step adds them.
//
// Data movement: one CTA per (split, sequence), one CTA per SM; warp w owns KV head w % Hkv,
// and the warps of one KV head take consecutive 32-row slices of each half of every tile.
// Tiles of whole packed rows (all KV heads) are copied by TMA bulk copies (one per
// contiguous run of rows, split at page boundaries) into a ring of shared-memory stages
// completed through mbarriers; waits are bounded.
//
// Merge of the split partials (log-sum-exp): a single sequence whose splits fit one wave is
// one cooperative launch whose CTAs merge the partials themselves (the grid merge below);
// otherwise pairs of splits merge in distributed shared memory (one sequence) or every CTA
// writes its own partial rows (batches), and the merge kernel of tq_attn.cu follows.
#include <atomic>
#include <cmath>

#include "tq_internal.cuh"
#include "tq_simd.cuh"
#include "tq_codes.cuh"
#include "tq_encode_warp.cuh"

namespace tq {
namespace {

// Compute warps per CTA (warp 0 lane 0 also issues the TMA copies), one CTA per SM: 16
// warps at 128 registers with one 128-value block per head, 8 with two (whose output
// accumulators need more registers).  Two warps per KV head at 8 KV heads share every
// tile, so all warps of an SM advance through the same ring and finish together (two
// CTAs of 8 warps per SM ran unevenly: the later one took 60 % longer).
__host__ __device__ constexpr int consumers(int nb) { return nb == 1 ? 16 : 8; }
constexpr int kWarpTokens = 64;            // 4 m-tiles of 16 tokens per warp per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kWaitLimit = 1u << 26;  // bounded mbarrier wait (tens of ms)
constexpr uint32_t kInjectedWaitLimit = 64;   // polls per wait under tq_inject_wait_timeout
constexpr uint32_t kGridWaitLimit = 1u << 16;  // grid-merge polls (each an L2 round trip)
constexpr uint32_t kEpochMark = 0x7154e90cu;   // high half of an epoch word this form wrote

// Launches still to run with injected timeouts (tq_inject_wait_timeout).
std::atomic<int> g_inject_timeouts{0};
constexpr size_t kSmemBudget = 227 * 1024;   // per CTA (one per SM): the sm_100 family's maximum

// Rotated queries in shared memory, in MMA-fragment order: head h, block b, k-step j and
// lane quarter q4 hold the four values 32 q4 + 4j .. +3 at halfs h*QS + 128 b + 16 j + 4 q4
// (the high fp16 parts; the low parts follow in the same layout, Hq * QS halfs later, then
// one row of zeros that lanes without a head read, so their loads need no select).
// QS = 128 nb + 16 puts consecutive heads 8 banks apart, so each half-warp's 8-byte
// B-fragment loads (four heads x four quarters) cover all 32 banks once.
__host__ __device__ constexpr int q_stride(int nb) { return 128 * nb + 16; }
inline size_t q_bytes(int n_q_heads, int nb) {
    return ((size_t)(2 * n_q_heads + 1) * q_stride(nb) * 2 + 127) & ~size_t(127);
}

struct MmaParams {
    CacheView kc, vc;
    const __half *q;
    const __half *k_new, *v_new;   // decode-step append: [n_seqs][Hkv][D] fp16, or null
    const int32_t *seq_lens;
    float *part;        // [n_seqs][n_splits][Hq][part_stride(D)]
    float score_scale;  // softmax scale * log2(e) / (sqrt(128) * h_scale of the K table)
    float v_unscale;    // 1 / h_scale of the V table (applied to the value norms)
    int64_t max_len;
    int32_t n_q_heads, n_kv_heads, group, head_dim;
    int32_t n_splits, tokens_per_split;
    int32_t wph;        // warps per KV head (8 / n_kv_heads)
    int32_t tile_tokens;
    int32_t stages;
    int32_t stage_bytes;
    int32_t cpart_offset;   // bytes from the first stage to this CTA's partial rows
    int32_t cl;             // CTAs per cluster: 2 (pairs of splits merge in shared memory) or 1
    uint32_t wait_limit;    // polls per bounded mbarrier wait
    // grid merge (one wave, cooperative launch): the output and the barrier area, else null
    float *out;
    uint64_t *bar;          // [0] epoch of the next call, [1 + cta] arrival flags
    uint32_t grid_wait_limit;   // polls of the grid barrier
    int32_t withhold_tiles; // fault injection: request no tile copies (every tile wait runs out)
    // 2, 4, 2^16, 2^30, 2^31: shift amounts as multipliers passed at run time, so that the
    // selector shifts compile to integer multiply-adds (FMA pipe) instead of ALU shifts
    uint32_t mul2, mul4, hi16, hi30, hi31;
};



// mbarrier helpers (shared::cta addresses)
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}


// Issue the TMA bulk copies of one tile (rows [t0, t0+nt) of both caches) into a stage.
// Runs of rows are split at page boundaries; every row run is a multiple of 16 bytes.
__device__ __forceinline__ void issue_tile(const MmaParams &p, int seq, int64_t t0, int nt,
                                           uint8_t *dk, uint8_t *dv, uint32_t bar) {
    const CacheView *cs[2] = {&p.kc, &p.vc};
    uint8_t *ds[2] = {dk, dv};
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const CacheView &cv = *cs[c];
        int r = 0;
        while (r < nt) {
            const int64_t pos = t0 + r;
            int run = nt - r;
            if (cv.page_tokens) run = (int)min64(run, cv.page_tokens - pos % cv.page_tokens);
            const uint8_t *src = row_ptr(cv, seq, pos);
            // the whole run must lie inside the cache (the first row's check covers a
            // page; a contiguous run also needs its last row below the capacity)
            if (src && !cv.page_tokens && !row_ptr(cv, seq, pos + run - 1)) src = nullptr;
            if (src) {
                const uint32_t bytes = (uint32_t)run * (uint32_t)cv.row_bytes;
                asm volatile("mbarrier.expect_tx.shared.b64 [%0], %1;\n" ::"r"(bar), "r"(bytes)
                             : "memory");
                bulk_g2s(smem_u32(ds[c] + (size_t)r * cv.row_bytes), src, bytes, bar);
            }
            r += run;
        }
    }
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];\n" ::"r"(bar) : "memory");
}


__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *a) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t *a, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

// (value, tag) as one 64-bit word: the value's bits low, the tag high
__device__ __forceinline__ uint64_t tagged(float v, uint32_t tag) {
    return ((uint64_t)tag << 32) | __float_as_uint(v);
}

// A CTA's partial rows in shared memory: coordinate c of a 128-value block sits at word
// c ^ 2((c >> 5) & 3).  The epilogue's stores in accumulator order (lane (g8, q4) holds
// coordinates 32(g8 >> 1) + (g8 & 1) + 4j + 2t of heads 2 q4 + e) then fall in 32 distinct
// banks; unswizzled, lanes g8 = 0, 2, 4, 6 met in one bank.
__device__ __forceinline__ int cpart_pos(int c) { return c ^ (((c >> 5) & 3) << 1); }
// Word offset of the float4 that holds coordinates 4 lane .. 4 lane + 3 of a block; its halves
// come swapped when bit 3 of the lane is set (cpart_fix4).
__device__ __forceinline__ int cpart_off4(int lane) { return 4 * (lane ^ ((lane >> 4) & 1)); }
__device__ __forceinline__ float4 cpart_fix4(float4 x, int lane) {
    return (lane & 8) ? make_float4(x.z, x.w, x.x, x.y) : x;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// Bounded wait on an mbarrier phase; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// The merge half of the grid merge, after this CTA's tagged partial rows are stored.
template <int kConsumers>
__device__ __forceinline__ void grid_merge(const float *part, uint64_t *bar, float *out, uint8_t *stage0,
                                        uint64_t E, bool marked, uint32_t e, uint32_t tag, int Hq,
                                        int D, int n_splits, uint32_t wait_limit, int trace_slot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int PS = part_stride(D);
    const int64_t rw = (int64_t)Hq * PS;
    (void)trace_slot;
    const int n_ctas = gridDim.x, me = blockIdx.x;
    // merge scratch at the start of the (idle) ring; the partial rows above sit at its end
    int *s_ok = reinterpret_cast<int *>(stage0);
    float *s_red = reinterpret_cast<float *>(stage0) + 32;     // [2][kConsumers]
    float *s_w = s_red + 2 * kConsumers;                       // [kGridMergeMaxCtas]
    float *s_acc = s_w + kGridMergeMaxCtas;                    // [kConsumers][32]
    if (!marked) {
        if (warp == 0) {
            const uint64_t token = (E + 1) * 0x9E3779B97F4A7C15ull;
            if (lane == 0) {
                __threadfence();   // this CTA's rows before its flag
                st_relaxed_u64(bar + 1 + me, token);
            }
            bool all = false;
            for (uint32_t it = 0; it < wait_limit && !all; ++it) {
                uint64_t f[kGridMergeMaxCtas / 32];
#pragma unroll
                for (int k = 0; k < kGridMergeMaxCtas / 32; ++k) {
                    const int c = lane + 32 * k;
                    f[k] = c < n_ctas ? ld_relaxed_u64(bar + 1 + c) : token;
                }
                bool mine = true;
#pragma unroll
                for (int k = 0; k < kGridMergeMaxCtas / 32; ++k) mine &= f[k] == token;
                all = __all_sync(0xffffffffu, mine);
            }
            __threadfence();   // the other CTAs' rows after their flags
            if (lane == 0) *s_ok = all ? 1 : 0;
        }
        __syncthreads();
        if (!*s_ok) {
            if (tid == 0) record_error(TQ_ERR_DEVICE_TIMEOUT);
            if (me == 0 && tid == 0) st_relaxed_u64(bar, ((uint64_t)kEpochMark << 32) | (e + 1u));
            return;
        }
    }
    if (tid == 0) TQ_PHASE(trace_slot, 8);
    constexpr int kRowsPerWarp = kGridMergeMaxCtas / kConsumers;
    const int SL = D / 32, R = n_splits;   // slices per head: (block, c) pairs
    const int n_items = Hq * SL;
    bool advanced = false;
    for (int item = me; item < n_items; item += n_ctas) {
        // slice sl: coordinates 4 lane + (sl & 3) of block sl >> 2, stored at words 32 sl + lane
        const int sl = item % SL, hh = item / SL;
        const uint64_t *base = reinterpret_cast<const uint64_t *>(part) + (int64_t)hh * PS;
        // warp w sums rows w, w + kConsumers, ... (lane = coordinate); thread t < R
        // brings row t's (m, l): every load of one reading is in flight at once
        float ov[kRowsPerWarp];
        float2 ml = make_float2(-INFINITY, 0.f);
        bool done = false;
        for (uint32_t it = 0; it < wait_limit && !done; ++it) {
            bool mine = true;
#pragma unroll
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int r = warp + kConsumers * k;
                const uint64_t wv = r < R ? ld_relaxed_u64(base + r * rw + 32 * sl + lane)
                                          : (uint64_t)tag << 32;
                mine &= (uint32_t)(wv >> 32) == tag;
                ov[k] = __uint_as_float((uint32_t)wv);
            }
            if (tid < R) {
                const uint64_t wm = ld_relaxed_u64(base + tid * rw + D);
                const uint64_t wl = ld_relaxed_u64(base + tid * rw + D + 1);
                mine &= (uint32_t)(wm >> 32) == tag && (uint32_t)(wl >> 32) == tag;
                ml = make_float2(__uint_as_float((uint32_t)wm), __uint_as_float((uint32_t)wl));
            }
            done = __syncthreads_and(mine) != 0;
        }
        if (!done) {
            if (tid == 0) record_error(TQ_ERR_DEVICE_TIMEOUT);
            break;
        }
        if (me == 0 && tid == 0 && !advanced) {
            st_relaxed_u64(bar, ((uint64_t)kEpochMark << 32) | (e + 1u));
            advanced = true;
        }
        if (tid == 0 && item == me) TQ_PHASE(trace_slot, 9);
        float mx = ml.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[warp] = mx;
        __syncthreads();
        float M = s_red[0];
        for (int w = 1; w < kConsumers; ++w) M = fmaxf(M, s_red[w]);
        const float wr = ml.x == -INFINITY ? 0.f : __expf(ml.x - M);
        if (tid < R) s_w[tid] = wr;
        float lw = wr * ml.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        if (lane == 0) s_red[kConsumers + warp] = lw;
        __syncthreads();
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kRowsPerWarp; ++k) {
            const int r = warp + kConsumers * k;
            if (r < R) acc = fmaf(s_w[r], ov[k], acc);
        }
        s_acc[warp * 32 + lane] = acc;
        __syncthreads();
        if (warp == 0) {
            float L = 0.f, o = 0.f;
            for (int w = 0; w < kConsumers; ++w) {
                L += s_red[kConsumers + w];
                o += s_acc[w * 32 + lane];
            }
            const float inv = L > 0.f ? kInvSqrt128 / L : 0.f;
            out[(int64_t)hh * D + kBlock * (sl >> 2) + 4 * lane + (sl & 3)] = o * inv;
        }
        __syncthreads();   // the scratch is reused by the next item
    }
    if (me == 0 && tid == 0 && !advanced) st_relaxed_u64(bar, ((uint64_t)kEpochMark << 32) | (e + 1u));
    if (tid == 0) TQ_PHASE(trace_slot, 10);
}

// APPEND: the decode-step form (p.k_new set); a separate instantiation, so that the plain
// attention carries none of its code.  QLO2: more than four query heads per KV head, so the
// low parts of the query take a second MMA per k-step instead of the spare columns.
template <int TK, int TV, int NB, bool APPEND, bool QLO2>
__global__ void __launch_bounds__(32 * consumers(NB), 1) attn_mma_kernel(const MmaParams p) {
    constexpr int kConsumers = consumers(NB);
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int BK = block_bytes(TK), BV = block_bytes(TV);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, q4 = lane & 3;
    const int Hq = p.n_q_heads, D = p.head_dim, G = p.group, Hkv = p.n_kv_heads;
    const int Rk = p.kc.row_bytes, Rv = p.vc.row_bytes;
    const int TT = p.tile_tokens;
    const int seq = blockIdx.y, split = blockIdx.x;
    const int trace_slot = blockIdx.y * gridDim.x + blockIdx.x;   // phase trace only
    (void)trace_slot;
    if (tid == 0) TQ_PHASE(trace_slot, 0);

    constexpr int QS = q_stride(NB);
    __half *qh = reinterpret_cast<__half *>(smem);                          // [Hq][QS]
    const size_t qbytes = ((size_t)(2 * Hq + 1) * QS * 2 + 127) & ~size_t(127);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + qbytes);          // [stages]
    uint64_t *empty = full + 4;                                            // [stages]
    uint8_t *stage0 = smem + qbytes + 128;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    // Before the dependency wait, warm L2 with this CTA's first reads: the sequence length,
    // the query row, the new token's rows and the first tile's rows of a contiguous cache.
    // An L2 prefetch puts nothing into the SM and L2 is where the GPU's memory is coherent,
    // so whatever the kernel before this one writes, the loads after the wait see it; the
    // prefetch only moves the DRAM latency of those first loads under that kernel's tail
    // (at a 32K context the length and query loads took about 2 us after the wait).
    // Tile 0 holds TT / 2 tokens, the others TT: with every CTA requesting its first tile
    // at once, a short first tile arrives sooner and the compute starts while the rest of
    // the split streams in.
    const int TF = TT / 2;
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    // In a contiguous cache the first tile's rows are known before the length: their
    // addresses are formed here, and the copy is requested right after the length load
    // when the tile turns out full and free of the new row (every CTA but the last ones).
    const uint8_t *pre_k = nullptr, *pre_v = nullptr;
    if (tid == 0) {
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.seq_lens + seq));
        l2_prefetch(p.q + (int64_t)seq * Hq * D, (uint32_t)(Hq * D * 2));
        if (APPEND) {
            l2_prefetch(p.k_new + (int64_t)seq * Hkv * D, (uint32_t)(Hkv * D * 2));
            l2_prefetch(p.v_new + (int64_t)seq * Hkv * D, (uint32_t)(Hkv * D * 2));
        }
        const int64_t t1 = min64(min64(t_begin + TF, t_begin + p.tokens_per_split), p.max_len);
        if (!p.kc.page_tokens && !p.vc.page_tokens && seq < p.kc.n_seqs && seq < p.vc.n_seqs) {
            const int64_t e = min64(t1, min64(p.kc.capacity, p.vc.capacity));
            if (e > t_begin) {
                const uint8_t *k0 = p.kc.base + (seq * p.kc.capacity + t_begin) * (int64_t)Rk;
                const uint8_t *v0 = p.vc.base + (seq * p.vc.capacity + t_begin) * (int64_t)Rv;
                l2_prefetch(k0, (uint32_t)((e - t_begin) * Rk));
                l2_prefetch(v0, (uint32_t)((e - t_begin) * Rv));
                if (e == t_begin + TF) {
                    pre_k = k0;
                    pre_v = v0;
                }
            }
        }
    }
    // The fp16 codebook tables and the last parameters, from the constant cache: their first
    // reads miss it, so they are made here, while the previous kernel runs (the codebook is
    // written by host copies only, never by a kernel).
    const HalfTables tk = make_tables<TK>(), tv = make_tables<TV>();
    asm volatile("" ::"r"(tk.l0), "r"(tk.l1), "r"(tk.h0), "r"(tk.h1), "r"(tv.l0), "r"(tv.l1),
                 "r"(tv.h0), "r"(tv.h1), "r"(p.mul2), "r"(p.hi31));
    // everything above touches only shared memory (and L2 prefetches); inputs may come from
    // the kernel launched before this one
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) TQ_PHASE(trace_slot, 1);

    // The query blocks of the rotation's first pass are requested first: the first tile's
    // copies, which all CTAs request right after the length load, then fill the memory
    // system for about a microsecond.
    constexpr int kRot = kConsumers - 1;
    uint2 qraw[5];
#pragma unroll
    for (int k = 0; k < 5; ++k) {
        const int hb = warp - 1 + k * kRot;
        const int h = hb / NB, b = hb - h * NB;
        qraw[k] = warp > 0 && hb < Hq * NB
                      ? *reinterpret_cast<const uint2 *>(p.q + ((int64_t)seq * Hq + h) * D + b * kBlock + 4 * lane)
                      : make_uint2(0u, 0u);
    }

    // grid merge: the workspace's epoch word, read now by the last warp's lane 0 and parked
    // in shared memory after the rotation (its L2 latency stays off the epilogue)
    uint64_t epoch_word = 0;
    if (p.out && tid == 32 * (kConsumers - 1)) epoch_word = ld_relaxed_u64(p.bar);

    int64_t len = p.seq_lens[seq];
    if (len < 0 || len > p.max_len) {
        if (tid == 0) record_error(TQ_ERR_OUT_OF_RANGE);
        len = len < 0 ? 0 : p.max_len;
    }
    // the first tile is full (TF rows) and does not hold the new row (position len - 1)
    const bool early0 = pre_k && len - (APPEND ? 1 : 0) >= t_begin + TF;
    if (tid == 0 && early0 && !p.withhold_tiles) {
        const uint32_t bar = smem_u32(&full[0]);
        asm volatile("mbarrier.expect_tx.shared.b64 [%0], %1;\n" ::"r"(bar), "r"((uint32_t)TF * (uint32_t)(Rk + Rv))
                     : "memory");
        bulk_g2s(smem_u32(stage0), pre_k, (uint32_t)TF * (uint32_t)Rk, bar);
        bulk_g2s(smem_u32(stage0 + (size_t)TT * Rk), pre_v, (uint32_t)TF * (uint32_t)Rv, bar);
        asm volatile("mbarrier.arrive.shared.b64 _, [%0];\n" ::"r"(bar) : "memory");
    }
    if (tid == 0) TQ_PHASE(trace_slot, 2);
    const int64_t t_end = min64(len, t_begin + p.tokens_per_split);
    // 32-bit from here: a split is at most tokens_per_split rows
    const int span = (int)max64(t_end - t_begin, 0);
    const int n_tiles = span == 0 ? 0 : span <= TF ? 1 : 1 + (span - TF + TT - 1) / TT;
    auto tile_start = [&](int i) -> int64_t { return t_begin + (i == 0 ? 0 : TF + (int64_t)(i - 1) * TT); };
    auto tile_len = [&](int i) -> int { return (int)min64(i == 0 ? TF : TT, t_end - tile_start(i)); };
    // ---- decode-step append (k_new set): the CTA whose split holds the new row (position
    // len - 1, the last row of its last tile) encodes the token's K and V blocks, one warp
    // per block, after the query rotation, and stores them in the caches.  When that tile's
    // stage is filled for the first time (the usual case), the blocks are also written
    // straight into the stage and the tile's TMA copy stops one row short, so the new row
    // costs no round trip through memory.  Otherwise an async-proxy fence and the barrier
    // below order the stores before the refill that copies the row; no other CTA reads it.
    const bool owner = APPEND && len > 0 && len - 1 >= t_begin && len - 1 < t_begin + p.tokens_per_split;
    const int i_new = owner ? n_tiles - 1 : -1;            // the tile holding the new row
    const bool new_in_stage = owner && i_new < p.stages;
    const int bpr = Hkv * NB;
    auto enc_src = [&](int bi) -> const __half * {
        const int c = bi >= bpr ? 1 : 0;
        return (c ? p.v_new : p.k_new) + ((int64_t)seq * bpr + (bi - c * bpr)) * kBlock;
    };
    uint2 enc_raw = make_uint2(0u, 0u);   // this warp's first block, loaded with the query
    if (owner && warp < 2 * bpr) enc_raw = warp_block_load(enc_src(warp), lane);
    // Thread 0 requests the first tile as soon as the sequence length is known and the rest
    // of the ring once that tile has landed; warps 1-15 rotate the query meanwhile, so the
    // query loads and the length load are in flight together.
    auto issue = [&](int i) {
        if (p.withhold_tiles) return;   // injected fault: nothing is copied, no copy in flight
        const int64_t t0 = tile_start(i);
        const int nt = tile_len(i) - (i == i_new && new_in_stage ? 1 : 0);
        uint8_t *dk = stage0 + (size_t)(i % p.stages) * p.stage_bytes;
        issue_tile(p, seq, t0, nt, dk, dk + (size_t)TT * Rk, smem_u32(&full[i % p.stages]));
    };
    if (tid == 0 && n_tiles > 0 && !early0) issue(0);
    if (tid == 0) TQ_PHASE(trace_slot, 3);
    if (warp == 0)   // the zero row of lanes without a head (warp 0 rotates nothing)
        for (int i = lane; i < QS / 8; i += 32)
            reinterpret_cast<uint4 *>(qh + 2 * Hq * QS)[i] = make_uint4(0u, 0u, 0u, 0u);
    // ---- rotate q once per call: y = W q_b * score_scale, stored as hi = fp16(y) and
    // lo = fp16(y - hi), by warps 1-15; a warp loads its (up to five) query blocks at once
    // (those of the first pass above), then rotates them
    if (warp > 0)
    for (int hb0 = warp - 1; hb0 < Hq * NB; hb0 += 5 * kRot) {
        if (hb0 != warp - 1) {
#pragma unroll
            for (int k = 0; k < 5; ++k) {
                const int hb = hb0 + k * kRot;
                const int h = hb / NB, b = hb - h * NB;
                qraw[k] = hb < Hq * NB
                              ? *reinterpret_cast<const uint2 *>(p.q + ((int64_t)seq * Hq + h) * D + b * kBlock + 4 * lane)
                              : make_uint2(0u, 0u);
            }
        }
#pragma unroll
        for (int k = 0; k < 5; ++k) {
            const int hb = hb0 + k * kRot;
            if (hb >= Hq * NB) break;
            const int h = hb / NB, b = hb - h * NB;
            const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&qraw[k].x));
            const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&qraw[k].y));
            float v[4] = {f01.x, f01.y, f23.x, f23.y};
            apply_signs4(v, p.kc, 4 * lane);   // rotation W D of the K cache
            warp_fwht4(v, lane);
            uint2 hi, lo;
            split_half2(v[0] * p.score_scale, v[1] * p.score_scale, hi.x, lo.x);
            split_half2(v[2] * p.score_scale, v[3] * p.score_scale, hi.y, lo.y);
            // lane = 8 q4 + j holds values 4 lane .. 4 lane + 3 = 32 q4 + 4 j ..
            __half *dst = qh + h * QS + b * kBlock + 16 * (lane & 7) + 4 * (lane >> 3);
            *reinterpret_cast<uint2 *>(dst) = hi;
            *reinterpret_cast<uint2 *>(dst + Hq * QS) = lo;
        }
    }
    if (owner) {
        // the new row's slot in its stage (used when new_in_stage)
        uint8_t *sk = stage0 + (size_t)(i_new % p.stages) * p.stage_bytes;
        const int r_new = tile_len(i_new) - 1;
        for (int bi = warp; bi < 2 * bpr; bi += kConsumers) {
            const int c = bi >= bpr ? 1 : 0, jb = bi - c * bpr;
            const CacheView &cv = c ? p.vc : p.kc;
            const uint2 raw = bi == warp ? enc_raw : warp_block_load(enc_src(bi), lane);
            uint8_t *row = nullptr;
            if (lane == 0) row = row_ptr(cv, seq, len - 1);   // records an out-of-range row once
            row = reinterpret_cast<uint8_t *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row), 0));
            if (TK == TV) {   // one call site: the second copy of the encoder slowed the main loop
                const WarpBlock wb = warp_encode_raw<TK>(raw, cv, lane);
                uint8_t *srow = c ? sk + (size_t)TT * Rk + (size_t)r_new * Rv : sk + (size_t)r_new * Rk;
                const int bb = c ? BV : BK;
                if (row) warp_store_block<TK>(row + jb * bb, wb, lane);
                if (new_in_stage) warp_store_block<TK>(srow + jb * bb, wb, lane);
            } else if (c) {
                const WarpBlock wb = warp_encode_raw<TV>(raw, cv, lane);
                if (row) warp_store_block<TV>(row + jb * BV, wb, lane);
                if (new_in_stage) warp_store_block<TV>(sk + (size_t)TT * Rk + (size_t)r_new * Rv + jb * BV, wb, lane);
            } else {
                const WarpBlock wb = warp_encode_raw<TK>(raw, cv, lane);
                if (row) warp_store_block<TK>(row + jb * BK, wb, lane);
                if (new_in_stage) warp_store_block<TK>(sk + (size_t)r_new * Rk + jb * BK, wb, lane);
            }
        }
        if (!new_in_stage) asm volatile("fence.proxy.async.global;\n" ::: "memory");
    }
    if (p.out && tid == 32 * (kConsumers - 1)) full[8] = epoch_word;   // past the barriers
    __syncthreads();
    // (a read of another warp's store keeps the stamp after the barrier)
    if (tid == 0 && __half_as_ushort(qh[0]) != 0x7e01u) TQ_PHASE(trace_slot, 4);

    bool timed_out = false;

    // ================= consumer warps
    const int g = warp % Hkv, sub = warp / Hkv;
    float m_run[2] = {-INFINITY, -INFINITY};  // log2 domain, heads 2q4, 2q4+1
    float l_run[2] = {0.f, 0.f};
    float oacc[NB][8][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[b][j][e] = 0.f;

    {
        // B fragments of the rotated query (column n = g8, values 32q4 + 4j + e) are read
        // from shared memory at each use: one 8-byte load per k-step and part.  Without
        // QLO2, column n < 4 holds the high part of head n and column 4 + n its low part;
        // with QLO2, column n holds head n, high part in the first MMA, low in the second.
        const int qhead = QLO2 ? g8 : (g8 & 3);
        const __half *qrow = qhead < G
            ? qh + ((QLO2 || g8 < 4 ? 0 : Hq) + g * G + qhead) * QS + 4 * q4
            : qh + 2 * Hq * QS + 4 * q4;                                  // the zero row
        const __half *qrow_lo = qhead < G ? qrow + Hq * QS : qrow;
        auto bq = [&](int b, int j) -> uint2 {
            return *reinterpret_cast<const uint2 *>(qrow + b * kBlock + 16 * j);
        };
        auto bq_lo = [&](int b, int j) -> uint2 {
            return *reinterpret_cast<const uint2 *>(qrow_lo + b * kBlock + 16 * j);
        };
        // word alignment of this warp's blocks (same for every row: rows are 16-byte
        // multiples) and the word-aligned offsets of this lane's quarter within a row
        uint32_t shk[NB], shv[NB];
        int owk[NB], ovk[NB], owv[NB], ovv[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int bk = (g * NB + b) * BK, bv = (g * NB + b) * BV;
            shk[b] = (uint32_t)((bk + 2) & 3) * 8u;
            shv[b] = (uint32_t)((bv + 2) & 3) * 8u;
            owk[b] = (bk + 2 + 8 * q4) & ~3;
            ovk[b] = (bk + 34 + 4 * q4) & ~3;
            owv[b] = (bv + 2 + 8 * q4) & ~3;
            ovv[b] = (bv + 34 + 4 * q4) & ~3;
        }
        const Shifts ks = {p.mul2, p.mul4, p.hi16, p.hi30, p.hi31};

        for (int i = 0; i < n_tiles; ++i) {
            const int s = i % p.stages;
            if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((i / p.stages) & 1), p.wait_limit)) {
                record_error(TQ_ERR_DEVICE_TIMEOUT);
                timed_out = true;
                break;
            }
            // the rest of the ring once the first tile has landed, so that the first tiles of
            // all CTAs do not share the HBM with the second ones (no copy of these reads the
            // new row: see above)
            if (i == 0 && tid == 0) TQ_PHASE(trace_slot, 5);
            if (i == 0 && tid == 0)
                for (int k = 1; k < n_tiles && k < p.stages; ++k) issue(k);
            const int nt = tile_len(i);
            const uint8_t *Kt = stage0 + (size_t)s * p.stage_bytes;
            const uint8_t *Vt = Kt + (size_t)TT * Rk;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
            // first row of these two m-tiles: the warps of a KV head take consecutive
            // 32-row slices of each half of the tile (a first tile is one half)
            const int hr0 = 32 * (half * p.wph + sub);
            if (hr0 < nt) {
                // ---------------- scores S^T[token, head] of two m-tiles (32 tokens)
                float sc[2][4];
                // all code words and norms of the phase first, so the loads overlap
                Quarter<TK> kq[2][NB][2];
                float kn[2][NB][2];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint8_t *rk = Kt + (size_t)(hr0 + 16 * mt + g8 + 8 * t) * Rk;
                            kq[mt][b][t] = load_quarter<TK>(rk, owk[b], ovk[b], shk[b]);
                            kn[mt][b][t] = ld_norm(rk + (g * NB + b) * BK);
                        }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int rA = hr0 + 16 * mt + g8, rB = rA + 8;
                    float acc[2][4];   // the first k-step of each block writes it (zero C)
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const Quarter<TK> &qa = kq[mt][b][0];
                        const Quarter<TK> &qb = kq[mt][b][1];
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww)
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                uint32_t xa[4], xb[4];
                                group_pairs<TK>(qa, ww, r, tk, ks, xa);
                                group_pairs<TK>(qb, ww, r, tk, ks, xb);
                                const int j = 4 * ww + 2 * r;
                                const uint2 q0 = bq(b, j), q1 = bq(b, j + 1);
                                if (ww == 0 && r == 0) {
                                    mma16816_z(acc[0], xa[0], xb[0], xa[1], xb[1], q0.x, q0.y);
                                    mma16816_z(acc[1], xa[2], xb[2], xa[3], xb[3], q1.x, q1.y);
                                } else {
                                    mma16816(acc[0], xa[0], xb[0], xa[1], xb[1], q0.x, q0.y);
                                    mma16816(acc[1], xa[2], xb[2], xa[3], xb[3], q1.x, q1.y);
                                }
                                if (QLO2) {
                                    const uint2 l0 = bq_lo(b, j), l1 = bq_lo(b, j + 1);
                                    mma16816(acc[0], xa[0], xb[0], xa[1], xb[1], l0.x, l0.y);
                                    mma16816(acc[1], xa[2], xb[2], xa[3], xb[3], l1.x, l1.y);
                                }
                            }
                        const float nA = kn[mt][b][0], nB = kn[mt][b][1];
                        s0 = fmaf(nA, acc[0][0] + acc[1][0], s0);
                        s1 = fmaf(nA, acc[0][1] + acc[1][1], s1);
                        s2 = fmaf(nB, acc[0][2] + acc[1][2], s2);
                        s3 = fmaf(nB, acc[0][3] + acc[1][3], s3);
                    }
                    if (!QLO2) {   // add the low parts' columns 4 + n (lane q4 ^ 2)
                        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
                        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
                        s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
                        s3 += __shfl_xor_sync(0xffffffffu, s3, 2);
                    }
                    // rows past the tile's valid tokens hold stale bytes: masked here
                    const bool okA = rA < nt, okB = rB < nt;
                    sc[mt][0] = okA ? s0 : -INFINITY;
                    sc[mt][1] = okA ? s1 : -INFINITY;
                    sc[mt][2] = okB ? s2 : -INFINITY;
                    sc[mt][3] = okB ? s3 : -INFINITY;
                }
                // ---------------- online softmax over the 32 tokens (log2 domain)
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
                    mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
                }
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
                const float al0 = mn0 == -INFINITY ? 1.f : ex2(m_run[0] - mn0);
                const float al1 = mn1 == -INFINITY ? 1.f : ex2(m_run[1] - mn1);
                m_run[0] = mn0;
                m_run[1] = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {   // masked: ex2(-inf) = 0
                    sc[mt][0] = ex2(sc[mt][0] - mn0);
                    sc[mt][1] = ex2(sc[mt][1] - mn1);
                    sc[mt][2] = ex2(sc[mt][2] - mn0);
                    sc[mt][3] = ex2(sc[mt][3] - mn1);
                    ps0 += sc[mt][0] + sc[mt][2];
                    ps1 += sc[mt][1] + sc[mt][3];
                }
                l_run[0] = l_run[0] * al0 + ps0;
                l_run[1] = l_run[1] * al1 + ps1;
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            oacc[b][j][0] *= al0;
                            oacc[b][j][1] *= al1;
                            oacc[b][j][2] *= al0;
                            oacc[b][j][3] *= al1;
                        }
                }
                // ---------------- values O^T[coord, head] += C_v^T[coord, token] (p|v|)^T
                Quarter<TV> vq[2][NB][2];
                float vn[2][NB][2];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const int row = hr0 + 16 * mt + g8 + 8 * t;
                            const uint8_t *rv = Vt + (size_t)row * Rv;
                            vq[mt][b][t] = load_quarter<TV>(rv, owv[b], ovv[b], shv[b]);
                            // masked rows may hold stale bytes: their weight is forced to 0;
                            // 1 / h_scale undoes the scaled V table
                            vn[mt][b][t] = row < nt ? ld_norm(rv + (g * NB + b) * BV) * p.v_unscale : 0.f;
                        }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float nvA = vn[mt][b][0], nvB = vn[mt][b][1];
                        const uint32_t b0 = movtrans(pack_half2(sc[mt][0] * nvA, sc[mt][1] * nvA));
                        const uint32_t b1 = movtrans(pack_half2(sc[mt][2] * nvB, sc[mt][3] * nvB));
                        const Quarter<TV> &qa = vq[mt][b][0];
                        const Quarter<TV> &qb = vq[mt][b][1];
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww)
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                uint32_t ya[4], yb[4];
                                group_pairs<TV>(qa, ww, r, tv, ks, ya);
                                group_pairs<TV>(qb, ww, r, tv, ks, yb);
                                const int j = 4 * ww + 2 * r;   // m-tiles j, j+1: pairs 2j..2j+3
                                mma16816(oacc[b][j], movtrans(ya[0]), movtrans(ya[1]),
                                         movtrans(yb[0]), movtrans(yb[1]), b0, b1);
                                mma16816(oacc[b][j + 1], movtrans(ya[2]), movtrans(ya[3]),
                                         movtrans(yb[2]), movtrans(yb[3]), b0, b1);
                            }
                    }
                }
            }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            // refill: once every warp has released stage s, bring in tile i + stages
            if (tid == 0 && i + p.stages < n_tiles) {
                if (!mbar_wait(smem_u32(&empty[s]), (uint32_t)((i / p.stages) & 1), p.wait_limit)) {
                    record_error(TQ_ERR_DEVICE_TIMEOUT);
                } else {
                    uint8_t *dk = stage0 + (size_t)s * p.stage_bytes;
                    issue_tile(p, seq, tile_start(i + p.stages), tile_len(i + p.stages), dk,
                               dk + (size_t)TT * Rk, smem_u32(&full[s]));
                }
            }
        }
    }

    if (lane == 0) TQ_PHASE_MAX(trace_slot, 6);
    // ---------------- epilogue: combine the lanes' sums, the warps of one KV head, write
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], o);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], o);
    }
    if (timed_out) {
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
    }
    if (p.wph > 1) {
        // warps sub > 0 hand (m, l, O) to warp sub == 0 of the same KV head through the
        // (now idle) stage buffers; every lane keeps the same (coord, head) positions.
        // 16-byte stores and loads: a quarter-warp's 8 lanes, 144 bytes apart, cover the 32
        // banks once
        __syncthreads();
        float4 *xch = reinterpret_cast<float4 *>(stage0);
        constexpr int kPer4 = 1 + NB * 8;   // float4 per lane
        if (warp < kConsumers && sub > 0) {
            float4 *d = xch + ((size_t)warp * 32 + lane) * kPer4;
            d[0] = make_float4(m_run[0], m_run[1], l_run[0], l_run[1]);
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    d[1 + b * 8 + j] = make_float4(oacc[b][j][0], oacc[b][j][1], oacc[b][j][2], oacc[b][j][3]);
        }
        __syncthreads();
        if (warp < kConsumers && sub == 0) {
            for (int s2 = 1; s2 < p.wph; ++s2) {
                const float4 *d = xch + ((size_t)(s2 * Hkv + g) * 32 + lane) * kPer4;
                const float4 ml = d[0];
                const float mo[2] = {ml.x, ml.y}, lo[2] = {ml.z, ml.w};
                float sa[2], sb[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mn = fmaxf(m_run[e], mo[e]);
                    sa[e] = mn == -INFINITY ? 0.f : ex2(m_run[e] - mn);
                    sb[e] = mn == -INFINITY ? 0.f : ex2(mo[e] - mn);
                    l_run[e] = l_run[e] * sa[e] + lo[e] * sb[e];
                    m_run[e] = mn;
                }
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 o = d[1 + b * 8 + j];
                        oacc[b][j][0] = oacc[b][j][0] * sa[0] + o.x * sb[0];
                        oacc[b][j][1] = oacc[b][j][1] * sa[1] + o.y * sb[1];
                        oacc[b][j][2] = oacc[b][j][2] * sa[0] + o.z * sb[0];
                        oacc[b][j][3] = oacc[b][j][3] * sa[1] + o.w * sb[1];
                    }
            }
        }
    }
    // (a test of the last combined value keeps the stamp after the combine)
    if (tid == 0 && __float_as_uint(oacc[NB - 1][7][3]) != 0x7fc00001u) TQ_PHASE(trace_slot, 11);
    // ---------------- this CTA's partial rows [Hq][part_stride(D)] into shared memory
    // (the end of the stage ring, past the warp exchange area)
    const int PS = part_stride(D);
    float *cpart = reinterpret_cast<float *>(stage0 + p.cpart_offset);
    __syncthreads();
    if (sub == 0) {
        // O^T row g8 of m-tile j is value 32(g8/2) + 4j + (g8 & 1) of the block, row g8+8
        // the value two above it (pairs 2j and 2j+1 after the movmatrix transposes).
        const int cbase = 32 * (g8 >> 1) + (g8 & 1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int hl = 2 * q4 + e;
            if (hl >= G) continue;
            float *dst = cpart + (g * G + hl) * PS;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dst[b * kBlock + cpart_pos(cbase + 4 * j)] = oacc[b][j][e];
                    dst[b * kBlock + cpart_pos(cbase + 4 * j + 2)] = oacc[b][j][2 + e];
                }
            if (g8 == 0) {
                dst[D] = m_run[e] == -INFINITY ? -INFINITY : m_run[e] * kLn2;
                dst[D + 1] = l_run[e];
            }
        }
    }
    if (p.out) {
        // ---------------- grid merge (one sequence whose splits run as one wave, launched
        // cooperatively).  Each CTA writes its partial rows turned back from the rotated
        // basis (o = D W o~; W is its own inverse up to 1/sqrt(128), applied with the
        // normalisation) as 64-bit words (value, tag), the tag a hash of the epoch word at
        // the start of the workspace.  The CTAs then merge the (head, 32-coordinate) slices
        // assigned to them (coordinates 4 l + c, l = 0..31, of one block: one contiguous run
        // of words), re-reading a slice until every word carries this call's tag: a
        // word is written and read whole, so a matching tag means a current value, and no
        // barrier is needed (words left by earlier calls carry other tags).  The first CTA
        // advances the epoch once its slice is complete, that is once every CTA has read
        // the epoch.  A workspace whose epoch word lacks kEpochMark (not yet used by this
        // form: its words may hold anything) first passes a barrier of per-CTA flags with
        // 64-bit tokens.
        const uint64_t E = full[8];
        const bool marked = (uint32_t)(E >> 32) == kEpochMark;
        const uint32_t e = marked ? (uint32_t)E : 0u;
        const uint32_t tag = (e + 1u) * 0x9E3779B9u;
        const int64_t rw = (int64_t)Hq * PS;    // 64-bit words between consecutive splits' rows
        uint64_t *prow = reinterpret_cast<uint64_t *>(p.part) + (int64_t)split * rw;
        __syncthreads();   // cpart complete
        for (int hb = warp; hb < Hq * NB; hb += kConsumers) {
            const int h = hb / NB, b = hb - h * NB;
            const float4 x = cpart_fix4(
                *reinterpret_cast<const float4 *>(cpart + h * PS + b * kBlock + cpart_off4(lane)), lane);
            float v[4] = {x.x, x.y, x.z, x.w};
            warp_fwht4(v, lane);
            apply_signs4(v, p.vc, 4 * lane);
            // coordinate 4 lane + c of the block at word 32 c + lane: each store is one
            // contiguous 256-byte run
            uint64_t *dst = prow + (int64_t)h * PS + b * kBlock + lane;
#pragma unroll
            for (int c = 0; c < 4; ++c) st_relaxed_u64(dst + 32 * c, tagged(v[c], tag));
        }
        for (int h = tid; h < Hq; h += 32 * kConsumers) {
            st_relaxed_u64(prow + (int64_t)h * PS + D, tagged(cpart[h * PS + D], tag));
            st_relaxed_u64(prow + (int64_t)h * PS + D + 1, tagged(cpart[h * PS + D + 1], tag));
        }
        __syncthreads();
        if (tid == 0) TQ_PHASE(trace_slot, 7);
        grid_merge<kConsumers>(p.part, p.bar, p.out, stage0, E, marked, e, tag, Hq, D, p.n_splits,
                               p.grid_wait_limit, trace_slot);
        return;
    }
    // ---------------- the CTAs of a cluster (consecutive splits) merge their partials
    // through distributed shared memory: CTA rank r owns heads r, r + CL, ...  (a cluster of
    // one CTA writes its own partial rows)
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
    if (tid == 0) TQ_PHASE(trace_slot, 7);
    {
        uint32_t rank;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
        constexpr int CLM = kClusterSplits;   // the most CTAs a cluster has
        const int CL = p.cl;
        const uint32_t local = smem_u32(cpart);
        const int group = split / CL;
        const int n_groups = p.n_splits / CL;
        // a warp takes its heads two at a time and issues every remote load of both
        // before using any
        constexpr int HW = 2;
        for (int h0 = (int)rank + CL * warp; h0 < Hq; h0 += HW * CL * kConsumers) {
            float mc[HW][CLM], lc[HW][CLM];
            float4 v[HW][CLM][NB];
#pragma unroll
            for (int k = 0; k < HW; ++k) {
                const int h = min(h0 + k * CL * kConsumers, Hq - 1);
#pragma unroll
                for (int c = 0; c < CLM; ++c) {
                    if (c >= CL) break;
                    uint32_t ra;
                    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                                 : "=r"(ra) : "r"(local + (uint32_t)(h * PS + D) * 4u), "r"(c));
                    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                                 : "=f"(mc[k][c]), "=f"(lc[k][c]) : "r"(ra) : "memory");
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                                     : "=r"(ra) : "r"(local + (uint32_t)(h * PS + 128 * b + cpart_off4(lane)) * 4u), "r"(c));
                        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(v[k][c][b].x), "=f"(v[k][c][b].y), "=f"(v[k][c][b].z), "=f"(v[k][c][b].w) : "r"(ra) : "memory");
                        v[k][c][b] = cpart_fix4(v[k][c][b], lane);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < HW; ++k) {
                const int h = h0 + k * CL * kConsumers;
                if (h >= Hq) break;
                float M = -INFINITY, L = 0.f, wgt[CLM];
#pragma unroll
                for (int c = 0; c < CLM; ++c)
                    if (c < CL) M = fmaxf(M, mc[k][c]);
#pragma unroll
                for (int c = 0; c < CLM; ++c) {
                    if (c >= CL) {
                        wgt[c] = 0.f;
                        continue;
                    }
                    wgt[c] = mc[k][c] == -INFINITY ? 0.f : __expf(mc[k][c] - M);
                    L += wgt[c] * lc[k][c];
                }
                float *dst = p.part + (((int64_t)seq * n_groups + group) * Hq + h) * PS;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < CLM; ++c) {
                        if (c >= CL) break;
                        a.x = fmaf(wgt[c], v[k][c][b].x, a.x);
                        a.y = fmaf(wgt[c], v[k][c][b].y, a.y);
                        a.z = fmaf(wgt[c], v[k][c][b].z, a.z);
                        a.w = fmaf(wgt[c], v[k][c][b].w, a.w);
                    }
                    *reinterpret_cast<float4 *>(dst + 128 * b + 4 * lane) = a;
                }
                if (lane == 0) {
                    dst[D] = M;
                    dst[D + 1] = L;
                }
            }
        }
    }
    if (tid == 0) TQ_PHASE(trace_slot, 8);
    // nobody leaves while a peer may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

template <int TK, int TV, int NB, bool APPEND, bool QLO2>
tq_status launch_tt(const MmaParams &p, int n_seqs, cudaStream_t stream) {
    static_assert(kGridMergeMaxCtas % (32 * 1) == 0 && kGridMergeMaxCtas <= 32 * consumers(NB),
                  "one (m, l) load per thread in the grid merge");
    const size_t qbytes = q_bytes(p.n_q_heads, NB);
    const size_t smem = qbytes + 128 + (size_t)p.stages * p.stage_bytes;
    // the most any shape asks for, so the attribute is set once per device
    (void)smem;
    const tq_status st = kernel_setup(reinterpret_cast<const void *>(attn_mma_kernel<TK, TV, NB, APPEND, QLO2>),
                                      (int)kSmemBudget, 32 * consumers(NB), nullptr);
    if (st != TQ_OK) return st;
    PdlConfig lc(dim3(p.n_splits, n_seqs), dim3(32 * consumers(NB)), smem, stream);
    if (p.out) {   // the grid merge: every CTA resident at once (one per SM)
        lc.attrs[1].id = cudaLaunchAttributeCooperative;
        lc.attrs[1].val.cooperative = 1;
    } else {
        lc.attrs[1].id = cudaLaunchAttributeClusterDimension;
        lc.attrs[1].val.clusterDim.x = (unsigned)p.cl;
        lc.attrs[1].val.clusterDim.y = 1;
        lc.attrs[1].val.clusterDim.z = 1;
    }
    lc.cfg.numAttrs = 2;
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, attn_mma_kernel<TK, TV, NB, APPEND, QLO2>, p));
}

template <int TK, int TV, int NB>
tq_status launch_t(const MmaParams &p, int n_seqs, cudaStream_t stream) {
    if (p.group > 4)
        return p.k_new ? launch_tt<TK, TV, NB, true, true>(p, n_seqs, stream)
                       : launch_tt<TK, TV, NB, false, true>(p, n_seqs, stream);
    return p.k_new ? launch_tt<TK, TV, NB, true, false>(p, n_seqs, stream)
                   : launch_tt<TK, TV, NB, false, false>(p, n_seqs, stream);
}

template <int NB>
tq_status launch_nb(int tk, int tv, const MmaParams &p, int n_seqs, cudaStream_t stream) {
    if (tk == TQ_TURBO3 && tv == TQ_TURBO3) return launch_t<3, 3, NB>(p, n_seqs, stream);
    if (tk == TQ_TURBO2 && tv == TQ_TURBO2) return launch_t<2, 2, NB>(p, n_seqs, stream);
    if (tk == TQ_TURBO3 && tv == TQ_TURBO2) return launch_t<3, 2, NB>(p, n_seqs, stream);
    return launch_t<2, 3, NB>(p, n_seqs, stream);
}

size_t stage_bytes_for(int tile_tokens, size_t rk, size_t rv) {
    return ((size_t)tile_tokens * (rk + rv) + 16 + 127) & ~size_t(127);
}

}  // namespace

bool grid_merge_fits(int n_seqs, int n_splits) {
    return n_seqs == 1 && n_splits <= std::min(device_sm_count(), kGridMergeMaxCtas);
}

bool attn_mma_supported(const tq_cache &k, const tq_cache &v, int n_q_heads) {
    const int hkv = k.n_kv_heads, nb = k.head_dim / kBlock, G = n_q_heads / hkv;
    if (nb < 1 || nb > 2 || G > 8) return false;
    if (hkv < 1 || hkv > consumers(nb) || consumers(nb) % hkv) return false;
    const size_t rk = tq_row_bytes(k.type, hkv, k.head_dim), rv = tq_row_bytes(v.type, hkv, v.head_dim);
    if (rk % 16 || rv % 16) return false;
    const int TT = kWarpTokens * (consumers(nb) / hkv);
    if (k.page_tokens && k.page_tokens % 16) return false;
    if (v.page_tokens && v.page_tokens % 16) return false;
    const size_t qbytes = q_bytes(n_q_heads, nb);
    return qbytes + 128 + 2 * stage_bytes_for(TT, rk, rv) <= kSmemBudget;
}

tq_status launch_attn_mma(const tq_cache &k, const tq_cache &v, const void *q, int n_seqs,
                          int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len, float scale,
                          float *part, int n_splits, int tokens_per_split, int cluster,
                          const void *k_new, const void *v_new, float *out, uint64_t *bar,
                          cudaStream_t stream) {
    MmaParams p;
    p.kc = make_view(k);
    p.vc = make_view(v);
    p.q = static_cast<const __half *>(q);
    p.k_new = static_cast<const __half *>(k_new);
    p.v_new = static_cast<const __half *>(v_new);
    p.seq_lens = seq_lens;
    p.part = part;
    p.score_scale = scale * kLog2e * kInvSqrt128 / centroid_h_scale(k.type);
    p.v_unscale = 1.0f / centroid_h_scale(v.type);
    p.max_len = max_seq_len;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = k.n_kv_heads;
    p.group = n_q_heads / k.n_kv_heads;
    p.head_dim = k.head_dim;
    p.n_splits = n_splits;
    p.tokens_per_split = tokens_per_split;
    const int nb = k.head_dim / kBlock;
    p.wph = consumers(nb) / k.n_kv_heads;
    p.tile_tokens = kWarpTokens * p.wph;
    p.wait_limit = kWaitLimit;
    p.withhold_tiles = 0;
    p.out = out;
    p.bar = bar;
    p.grid_wait_limit = kGridWaitLimit;
    if (out && (cluster != 1 || !bar || !grid_merge_fits(n_seqs, n_splits))) return TQ_ERR_UNSUPPORTED;
    for (int n = g_inject_timeouts.load(); n > 0;)
        if (g_inject_timeouts.compare_exchange_weak(n, n - 1)) {
            p.wait_limit = kInjectedWaitLimit;
            p.withhold_tiles = 1;
            break;
        }
    p.mul2 = 2u;
    p.mul4 = 4u;
    p.hi16 = 1u << 16;
    p.hi30 = 1u << 30;
    p.hi31 = 1u << 31;
    const size_t stage = stage_bytes_for(p.tile_tokens, p.kc.row_bytes, p.vc.row_bytes);
    p.stage_bytes = (int)stage;
    const size_t qbytes = q_bytes(n_q_heads, nb);
    p.stages = (int)std::min<size_t>(4, (kSmemBudget - qbytes - 128) / stage);
    if (p.stages < 2) return TQ_ERR_UNSUPPORTED;
    if (cluster < 1 || cluster > kClusterSplits || n_splits % cluster) return TQ_ERR_UNSUPPORTED;
    p.cl = cluster;
    const size_t cpart = (size_t)n_q_heads * part_stride(k.head_dim) * sizeof(float);
    if (cpart > (size_t)p.stages * stage) return TQ_ERR_UNSUPPORTED;
    p.cpart_offset = (int)(((size_t)p.stages * stage - cpart) & ~size_t(15));
    return nb == 1 ? launch_nb<1>(k.type, v.type, p, n_seqs, stream)
                   : launch_nb<2>(k.type, v.type, p, n_seqs, stream);
}

tq_status inject_wait_timeout(int n_calls) {
    if (n_calls < 0) return TQ_ERR_INVALID_ARGUMENT;
    g_inject_timeouts.store(n_calls);
    return TQ_OK;
}

}  // namespace tq

extern "C" tq_status tq_inject_wait_timeout(int n_calls) { return tq::inject_wait_timeout(n_calls); }
