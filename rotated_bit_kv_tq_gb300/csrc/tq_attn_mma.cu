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
// Data movement: one CTA per (split, sequence), 8 warps; warp w owns KV head w % Hkv and a
// 64-token slice of every tile.  Tiles of whole packed rows (all KV heads) are copied by
// TMA bulk copies (one per contiguous run of rows, split at page boundaries) into a ring
// of shared-memory stages completed through mbarriers; waits are bounded.
#include <cmath>

#include "tq_internal.cuh"
#include "tq_simd.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kWarpTokens = 64;            // 4 m-tiles of 16 tokens per warp per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kWaitLimit = 1u << 26;  // bounded mbarrier wait (tens of ms)

struct MmaParams {
    CacheView kc, vc;
    const __half *q;
    const int32_t *seq_lens;
    float *part;        // [n_seqs][n_splits][Hq][D + 2]
    float score_scale;  // softmax scale * log2(e) / sqrt(128)
    int64_t max_len;
    int32_t n_q_heads, n_kv_heads, group, head_dim;
    int32_t n_splits, tokens_per_split;
    int32_t wph;        // warps per KV head (8 / n_kv_heads)
    int32_t tile_tokens;
    int32_t stages;
    int32_t stage_bytes;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 32-bit little-endian word at a 2-byte-aligned shared address.
__device__ __forceinline__ uint32_t ld_u32_2a(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *b = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    return __funnelshift_r(b[0], b[1], (uint32_t)(a & 3) * 8u);
}

__device__ __forceinline__ float ld_norm(const uint8_t *blk) {
    return __half2float(*reinterpret_cast<const __half *>(blk));
}

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

// ------------------------------------------------------------------ code -> fp16 lookup
// Byte tables of the fp16 codebook: L = low bytes, H = high bytes of entries 0..7.
struct HalfTables {
    uint32_t l0, l1, h0, h1;
};

// Selector of 8 codes: nibble k = code of value (16w + 8r + k) of a block whose low-plane
// word is W and high-plane word is V (bit 4k+p), per the layout of tq.h.
template <int TYPE>
__device__ __forceinline__ uint32_t sel8(uint32_t W, uint32_t V, int r, int p) {
    uint32_t x = (r ? (W >> 2) : W) & 0x33333333u;
    if (TYPE == TQ_TURBO3) {
        const uint32_t hv = (p <= 2) ? (V << (2 - p)) : (V >> (p - 2));
        x |= hv & 0x44444444u;
    }
    return x;
}

// Low and high bytes of the fp16 centroids of 4 codes (selector nibbles 0..3).
__device__ __forceinline__ void lookup4(const HalfTables &t, uint32_t sel, uint32_t &L,
                                        uint32_t &H) {
    L = prmt(t.l0, t.l1, sel);
    H = prmt(t.h0, t.h1, sel);
}

// Rotate the query of one (head, block) pair held by a warp, four values per lane
// (butterfly stages h = 1, 2 in-lane, 4 .. 64 across lanes).
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

template <int TK, int TV, int NB>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(const MmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int BK = block_bytes(TK), BV = block_bytes(TV);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, q4 = lane & 3;
    const int Hq = p.n_q_heads, D = p.head_dim, G = p.group, Hkv = p.n_kv_heads;
    const int Rk = p.kc.row_bytes, Rv = p.vc.row_bytes;
    const int TT = p.tile_tokens;
    const int seq = blockIdx.y, split = blockIdx.x;
    const int g = warp % Hkv, sub = warp / Hkv;

    __half *qh = reinterpret_cast<__half *>(smem);                          // [Hq][D]
    const size_t qbytes = ((size_t)Hq * D * 2 + 127) & ~size_t(127);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + qbytes);          // [stages]
    uint8_t *stage0 = smem + qbytes + 128;

    int64_t len = p.seq_lens[seq];
    if (len < 0 || len > p.max_len) {
        if (tid == 0) record_error(TQ_ERR_OUT_OF_RANGE);
        len = len < 0 ? 0 : p.max_len;
    }
    const int64_t t_begin = (int64_t)split * p.tokens_per_split;
    const int64_t t_end = min64(len, t_begin + p.tokens_per_split);
    const int n_tiles = t_end > t_begin ? (int)((t_end - t_begin + TT - 1) / TT) : 0;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) mbar_init(smem_u32(&bars[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        for (int i = 0; i < n_tiles && i < p.stages; ++i) {
            const int64_t t0 = t_begin + (int64_t)i * TT;
            const int nt = (int)min64(TT, t_end - t0);
            uint8_t *dk = stage0 + (size_t)i * p.stage_bytes;
            issue_tile(p, seq, t0, nt, dk, dk + (size_t)TT * Rk, smem_u32(&bars[i]));
        }
    }

    // ---- rotate q once per call: qh = fp16(W q_b * scale * log2(e) / sqrt(128))
    for (int hb = warp; hb < Hq * NB; hb += kWarps) {
        const int h = hb / NB, b = hb - h * NB;
        const __half *qp = p.q + ((int64_t)seq * Hq + h) * D + b * kBlock + 4 * lane;
        const uint2 raw = *reinterpret_cast<const uint2 *>(qp);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
        float v[4] = {f01.x, f01.y, f23.x, f23.y};
        warp_fwht4(v, lane);
        uint2 o;
        o.x = pack_half2(v[0] * p.score_scale, v[1] * p.score_scale);
        o.y = pack_half2(v[2] * p.score_scale, v[3] * p.score_scale);
        *reinterpret_cast<uint2 *>(qh + h * D + b * kBlock + 4 * lane) = o;
    }
    __syncthreads();

    // B fragments of the rotated query: head n = g8 of KV head g, coords 32 q4 + 4 j + e.
    uint32_t bq[NB][8][2];
    {
        const bool hv = g8 < G;
        const __half *qrow = qh + (g * G + (hv ? g8 : 0)) * D;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half *c = qrow + b * kBlock + 32 * q4 + 4 * j;
                bq[b][j][0] = hv ? *reinterpret_cast<const uint32_t *>(c) : 0u;
                bq[b][j][1] = hv ? *reinterpret_cast<const uint32_t *>(c + 2) : 0u;
            }
    }
    HalfTables tk, tv;
    {
        const __half *ck = c_codebook[cb_index(TK)].centroid_h;
        const __half *cv = c_codebook[cb_index(TV)].centroid_h;
        uint32_t lk[2] = {0, 0}, hk[2] = {0, 0}, lv[2] = {0, 0}, hv[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint16_t a = e < (1 << TK) ? __half_as_ushort(ck[e]) : 0;
            const uint16_t c = e < (1 << TV) ? __half_as_ushort(cv[e]) : 0;
            lk[e >> 2] |= (uint32_t)(a & 0xff) << (8 * (e & 3));
            hk[e >> 2] |= (uint32_t)(a >> 8) << (8 * (e & 3));
            lv[e >> 2] |= (uint32_t)(c & 0xff) << (8 * (e & 3));
            hv[e >> 2] |= (uint32_t)(c >> 8) << (8 * (e & 3));
        }
        tk = {lk[0], lk[1], hk[0], hk[1]};
        tv = {lv[0], lv[1], hv[0], hv[1]};
    }

    float m_run[2] = {-INFINITY, -INFINITY};  // log2 domain, heads 2q4, 2q4+1
    float l_run[2] = {0.f, 0.f};
    float oacc[NB][8][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[b][j][e] = 0.f;

    // V-side per-thread constants: low-plane word g8, high-plane word g8/2, bit offset p.
    const int vp = 2 * (g8 & 1);
    bool timed_out = false;

    for (int i = 0; i < n_tiles; ++i) {
        const int s = i % p.stages;
        const uint32_t bar = smem_u32(&bars[s]);
        {
            uint32_t it = 0;
            while (!mbar_try_wait(bar, (uint32_t)((i / p.stages) & 1))) {
                if (++it > kWaitLimit) {
                    timed_out = true;
                    break;
                }
            }
        }
        // one decision for the whole CTA, so that no thread is left at a barrier
        timed_out = __syncthreads_or(timed_out) != 0;
        if (timed_out) {
            if (tid == 0) record_error(TQ_ERR_DEVICE_TIMEOUT);
            break;
        }
        const int64_t t0 = t_begin + (int64_t)i * TT;
        const int nt = (int)min64(TT, t_end - t0);
        const uint8_t *Kt = stage0 + (size_t)s * p.stage_bytes;
        const uint8_t *Vt = Kt + (size_t)TT * Rk;
        const int wr0 = sub * kWarpTokens;   // this warp's first row in the tile

        if (wr0 < nt) {
            // ---------------- scores: S^T[token, head] for 4 m-tiles of 16 tokens
            float sc[4][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int rA = wr0 + 16 * mt + g8, rB = rA + 8;
                if (wr0 + 16 * mt < nt) {
                    float acc[NB][4];
                    float nA[NB], nB[NB];
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[b][e] = 0.f;
                        const uint8_t *bA = Kt + (size_t)rA * Rk + (g * NB + b) * BK;
                        const uint8_t *bB = Kt + (size_t)rB * Rk + (g * NB + b) * BK;
                        nA[b] = ld_norm(bA);
                        nB[b] = ld_norm(bB);
                        const uint32_t WA[2] = {ld_u32_2a(bA + 2 + 8 * q4), ld_u32_2a(bA + 6 + 8 * q4)};
                        const uint32_t WB[2] = {ld_u32_2a(bB + 2 + 8 * q4), ld_u32_2a(bB + 6 + 8 * q4)};
                        const uint32_t VA = TK == TQ_TURBO3 ? ld_u32_2a(bA + 34 + 4 * q4) : 0u;
                        const uint32_t VB = TK == TQ_TURBO3 ? ld_u32_2a(bB + 34 + 4 * q4) : 0u;
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww)
#pragma unroll
                            for (int r = 0; r < 2; ++r) {
                                const int j0 = 4 * ww + 2 * r;
                                const uint32_t sA = sel8<TK>(WA[ww], VA, r, 2 * ww + r);
                                const uint32_t sB = sel8<TK>(WB[ww], VB, r, 2 * ww + r);
                                uint32_t LA, HA, LB, HB;
                                lookup4(tk, sA, LA, HA);
                                lookup4(tk, sB, LB, HB);
                                mma16816(acc[b], prmt(LA, HA, 0x5140), prmt(LB, HB, 0x5140),
                                         prmt(LA, HA, 0x7362), prmt(LB, HB, 0x7362), bq[b][j0][0],
                                         bq[b][j0][1]);
                                lookup4(tk, sA >> 16, LA, HA);
                                lookup4(tk, sB >> 16, LB, HB);
                                mma16816(acc[b], prmt(LA, HA, 0x5140), prmt(LB, HB, 0x5140),
                                         prmt(LA, HA, 0x7362), prmt(LB, HB, 0x7362),
                                         bq[b][j0 + 1][0], bq[b][j0 + 1][1]);
                            }
                    }
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        s0 = fmaf(nA[b], acc[b][0], s0);
                        s1 = fmaf(nA[b], acc[b][1], s1);
                        s2 = fmaf(nB[b], acc[b][2], s2);
                        s3 = fmaf(nB[b], acc[b][3], s3);
                    }
                    const bool okA = t0 + rA < t_end, okB = t0 + rB < t_end;
                    sc[mt][0] = okA ? s0 : -INFINITY;
                    sc[mt][1] = okA ? s1 : -INFINITY;
                    sc[mt][2] = okB ? s2 : -INFINITY;
                    sc[mt][3] = okB ? s3 : -INFINITY;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[mt][e] = -INFINITY;
                }
            }
            // ---------------- online softmax (log2 domain), heads 2q4 and 2q4+1
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
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
            for (int mt = 0; mt < 4; ++mt) {
                sc[mt][0] = mn0 == -INFINITY ? 0.f : ex2(sc[mt][0] - mn0);
                sc[mt][1] = mn1 == -INFINITY ? 0.f : ex2(sc[mt][1] - mn1);
                sc[mt][2] = mn0 == -INFINITY ? 0.f : ex2(sc[mt][2] - mn0);
                sc[mt][3] = mn1 == -INFINITY ? 0.f : ex2(sc[mt][3] - mn1);
                ps0 += sc[mt][0] + sc[mt][2];
                ps1 += sc[mt][1] + sc[mt][3];
            }
            l_run[0] = l_run[0] * al0 + ps0;
            l_run[1] = l_run[1] * al1 + ps1;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    oacc[b][j][0] *= al0;
                    oacc[b][j][1] *= al1;
                    oacc[b][j][2] *= al0;
                    oacc[b][j][3] *= al1;
                }
            // ---------------- values: O^T[coord, head] += C_v^T[coord, token] (p|v|)^T
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                if (wr0 + 16 * mt >= nt) continue;
                const int rA = wr0 + 16 * mt + g8, rB = rA + 8;
                const int rt = wr0 + 16 * mt + 2 * q4;   // first token row of this lane's A pairs
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int boff = (g * NB + b) * BV;
                    const float nvA = ld_norm(Vt + (size_t)rA * Rv + boff);
                    const float nvB = ld_norm(Vt + (size_t)rB * Rv + boff);
                    // probabilities of masked tokens are exactly 0; keep stale norms out
                    const uint32_t x1 = pack_half2(sc[mt][0] == 0.f ? 0.f : sc[mt][0] * nvA,
                                                   sc[mt][1] == 0.f ? 0.f : sc[mt][1] * nvA);
                    const uint32_t x2 = pack_half2(sc[mt][2] == 0.f ? 0.f : sc[mt][2] * nvB,
                                                   sc[mt][3] == 0.f ? 0.f : sc[mt][3] * nvB);
                    const uint32_t b0 = movtrans(x1), b1 = movtrans(x2);
                    uint32_t A[2][2][8];   // [token pair][r][m-tile j]
#pragma unroll
                    for (int tp = 0; tp < 2; ++tp) {
                        const uint8_t *v0 = Vt + (size_t)(rt + 8 * tp) * Rv + boff;
                        const uint8_t *v1 = v0 + Rv;
                        const uint32_t W0 = ld_u32_2a(v0 + 2 + 4 * g8);
                        const uint32_t W1 = ld_u32_2a(v1 + 2 + 4 * g8);
                        uint32_t V0 = 0, V1 = 0;
                        if (TV == TQ_TURBO3) {
                            // bit 4k+vp of the high-plane word moved to bit 4k+2
                            const uint32_t h0 = ld_u32_2a(v0 + 34 + 4 * (g8 >> 1));
                            const uint32_t h1 = ld_u32_2a(v1 + 34 + 4 * (g8 >> 1));
                            V0 = __funnelshift_r(h0 << 2, h0 >> 30, vp);
                            V1 = __funnelshift_r(h1 << 2, h1 >> 30, vp);
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            uint32_t s0 = (r ? (W0 >> 2) : W0) & 0x33333333u;
                            uint32_t s1 = (r ? (W1 >> 2) : W1) & 0x33333333u;
                            if (TV == TQ_TURBO3) {
                                s0 |= (r ? (V0 >> 1) : V0) & 0x44444444u;
                                s1 |= (r ? (V1 >> 1) : V1) & 0x44444444u;
                            }
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                uint32_t L0, H0, L1, H1;
                                lookup4(tv, half ? s0 >> 16 : s0, L0, H0);
                                lookup4(tv, half ? s1 >> 16 : s1, L1, H1);
                                const uint32_t LL = prmt(L0, L1, 0x5140), HH = prmt(H0, H1, 0x5140);
                                const uint32_t LL2 = prmt(L0, L1, 0x7362), HH2 = prmt(H0, H1, 0x7362);
                                A[tp][r][4 * half + 0] = prmt(LL, HH, 0x5140);
                                A[tp][r][4 * half + 1] = prmt(LL, HH, 0x7362);
                                A[tp][r][4 * half + 2] = prmt(LL2, HH2, 0x5140);
                                A[tp][r][4 * half + 3] = prmt(LL2, HH2, 0x7362);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        mma16816(oacc[b][j], A[0][0][j], A[0][1][j], A[1][0][j], A[1][1][j], b0, b1);
                }
            }
        }
        __syncthreads();   // every warp is done with stage s
        if (tid == 0 && i + p.stages < n_tiles) {
            const int64_t tn = t_begin + (int64_t)(i + p.stages) * TT;
            const int ntn = (int)min64(TT, t_end - tn);
            uint8_t *dk = stage0 + (size_t)s * p.stage_bytes;
            issue_tile(p, seq, tn, ntn, dk, dk + (size_t)TT * Rk, bar);
        }
    }

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
        __syncthreads();
        float *xch = reinterpret_cast<float *>(stage0);
        constexpr int kPer = 4 + NB * 32;   // floats per lane
        if (sub > 0) {
            float *d = xch + ((size_t)warp * 32 + lane) * kPer;
            d[0] = m_run[0];
            d[1] = m_run[1];
            d[2] = l_run[0];
            d[3] = l_run[1];
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[4 + b * 32 + j * 4 + e] = oacc[b][j][e];
        }
        __syncthreads();
        if (sub == 0) {
            for (int s2 = 1; s2 < p.wph; ++s2) {
                const float *d = xch + ((size_t)(s2 * Hkv + g) * 32 + lane) * kPer;
                float sa[2], sb[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mo = d[e];
                    const float mn = fmaxf(m_run[e], mo);
                    sa[e] = mn == -INFINITY ? 0.f : ex2(m_run[e] - mn);
                    sb[e] = mn == -INFINITY ? 0.f : ex2(mo - mn);
                    l_run[e] = l_run[e] * sa[e] + d[2 + e] * sb[e];
                    m_run[e] = mn;
                }
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            oacc[b][j][e] = oacc[b][j][e] * sa[e & 1] + d[4 + b * 32 + j * 4 + e] * sb[e & 1];
            }
        }
    }
    if (sub == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int hl = 2 * q4 + e;
            if (hl >= G) continue;
            float *dst = p.part + (((int64_t)seq * p.n_splits + split) * Hq + g * G + hl) * (D + 2);
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dst[b * kBlock + 16 * g8 + j] = oacc[b][j][e];
                    dst[b * kBlock + 16 * g8 + 8 + j] = oacc[b][j][2 + e];
                }
            if (g8 == 0) {
                dst[D] = m_run[e] == -INFINITY ? -INFINITY : m_run[e] * kLn2;
                dst[D + 1] = l_run[e];
            }
        }
    }
}

template <int TK, int TV, int NB>
tq_status launch_t(const MmaParams &p, int n_seqs, cudaStream_t stream) {
    const size_t qbytes = ((size_t)p.n_q_heads * p.head_dim * 2 + 127) & ~size_t(127);
    const size_t smem = qbytes + 128 + (size_t)p.stages * p.stage_bytes;
    if (cudaFuncSetAttribute(attn_mma_kernel<TK, TV, NB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return TQ_ERR_CUDA;
    attn_mma_kernel<TK, TV, NB><<<dim3(p.n_splits, n_seqs), kThreads, smem, stream>>>(p);
    return check_cuda(cudaGetLastError());
}

template <int NB>
tq_status launch_nb(int tk, int tv, const MmaParams &p, int n_seqs, cudaStream_t stream) {
    if (tk == TQ_TURBO3 && tv == TQ_TURBO3) return launch_t<3, 3, NB>(p, n_seqs, stream);
    if (tk == TQ_TURBO2 && tv == TQ_TURBO2) return launch_t<2, 2, NB>(p, n_seqs, stream);
    if (tk == TQ_TURBO3 && tv == TQ_TURBO2) return launch_t<3, 2, NB>(p, n_seqs, stream);
    return launch_t<2, 3, NB>(p, n_seqs, stream);
}

}  // namespace

bool attn_mma_supported(const tq_cache &k, const tq_cache &v, int n_q_heads) {
    const int hkv = k.n_kv_heads, nb = k.head_dim / kBlock, G = n_q_heads / hkv;
    if (hkv < 1 || hkv > 8 || 8 % hkv) return false;
    if (nb < 1 || nb > 2 || G > 8) return false;
    const size_t rk = tq_row_bytes(k.type, hkv, k.head_dim), rv = tq_row_bytes(v.type, hkv, v.head_dim);
    if (rk % 16 || rv % 16) return false;
    const int wph = 8 / hkv, TT = kWarpTokens * wph;
    if (k.page_tokens && k.page_tokens % 16) return false;
    if (v.page_tokens && v.page_tokens % 16) return false;
    const size_t stage = ((size_t)TT * (rk + rv) + 16 + 127) & ~size_t(127);
    const size_t qbytes = ((size_t)n_q_heads * k.head_dim * 2 + 127) & ~size_t(127);
    return qbytes + 128 + 2 * stage <= 220 * 1024;
}

tq_status launch_attn_mma(const tq_cache &k, const tq_cache &v, const void *q, int n_seqs,
                          int n_q_heads, const int32_t *seq_lens, int64_t max_seq_len, float scale,
                          float *part, int n_splits, int tokens_per_split, cudaStream_t stream) {
    MmaParams p;
    p.kc = make_view(k);
    p.vc = make_view(v);
    p.q = static_cast<const __half *>(q);
    p.seq_lens = seq_lens;
    p.part = part;
    p.score_scale = scale * kLog2e * kInvSqrt128;
    p.max_len = max_seq_len;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = k.n_kv_heads;
    p.group = n_q_heads / k.n_kv_heads;
    p.head_dim = k.head_dim;
    p.n_splits = n_splits;
    p.tokens_per_split = tokens_per_split;
    p.wph = 8 / k.n_kv_heads;
    p.tile_tokens = kWarpTokens * p.wph;
    const size_t stage = ((size_t)p.tile_tokens * (p.kc.row_bytes + p.vc.row_bytes) + 16 + 127) &
                         ~size_t(127);
    p.stage_bytes = (int)stage;
    const size_t qbytes = ((size_t)n_q_heads * k.head_dim * 2 + 127) & ~size_t(127);
    p.stages = (int)std::min<size_t>(4, (220 * 1024 - qbytes - 128) / stage);
    if (p.stages < 2) return TQ_ERR_UNSUPPORTED;
    const int nb = k.head_dim / kBlock;
    return nb == 1 ? launch_nb<1>(k.type, v.type, p, n_seqs, stream)
                   : launch_nb<2>(k.type, v.type, p, n_seqs, stream);
}

}  // namespace tq
