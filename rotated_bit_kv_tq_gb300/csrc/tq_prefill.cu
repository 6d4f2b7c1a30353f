// tq_prefill.cu -- causal attention of a prompt chunk over the packed cache.
//
// "llama.cpp に TurboQuant を実装": prompt processing runs over the compressed cache as well
// ("Numbers on real models"), and the roadmap fuses the dequantisation into the Flash-
// Attention tiles so that K is never materialised in FP16 in HBM ("Current implementation
// and what's next").  Query token j of the chunk sits at position pos0 + j and attends to
// rows 0 .. pos0 + j (TinyLLaMA article, section 7, at every position of the chunk).
//
// Here the work is a dense contraction: one decoded K/V tile serves every query row of a
// CTA, so it runs on tensor cores in the Flash-Attention-2 arrangement.
//  - CTA = (block of query tokens, KV head g); its 128 rows are (query token, head of
//    the group) pairs, 16 per warp.  The rotated, scaled queries (fp16) stay in registers
//    as MMA A fragments.
//  - Keys come in tiles of 64: the bytes of head g's block of each row are staged with
//    cp.async (the covering 16-byte chunks), then decoded once into fp16 centroid values
//    in shared memory (the prmt lookups of tq_codes.cuh); norms are kept apart and applied
//    to the score columns (K) and to the probabilities (V).
//  - S = Q~ C_k^T (B fragments by ldmatrix), causal mask, online softmax in the log2 domain,
//    O += (p |v|) C_v (A = probabilities straight from the score accumulators, B by
//    ldmatrix.trans).  Everything stays in the rotated domain; each output row gets one
//    inverse FWHT at the end.
#include <cmath>

#include "tq_internal.cuh"
#include "tq_simd.cuh"
#include "tq_codes.cuh"

namespace tq {
namespace {

constexpr int kPfWarps = 8;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kPfRows = 16 * kPfWarps;      // (query token, head) rows per CTA
constexpr int kPfKeys = 64;                 // keys per tile
constexpr int kKs = 136;                    // halfs per decoded row (128 + 8: ldmatrix without bank conflicts)
constexpr int kSlot = 64;                   // staged bytes per key: the block's covering 16-byte chunks
constexpr int kOs = 132;                    // floats per output staging row
constexpr float kPfLog2e = 1.4426950408889634f;
// The 5th-generation tensor-core kernel (tq_prefill_tc.cu) takes every shape this one does.
constexpr bool kUseTcgen05 = true;

struct PrefillParams {
    CacheView kc, vc;
    const __half *q;        // [n_q][Hq][128] fp16
    float *out;             // [n_q][Hq][128] fp32
    int64_t pos0, n_q;
    int32_t seq, n_q_heads, group, bq;   // bq = query tokens per CTA (128 / group)
    int32_t chunked_k, chunked_v;        // row bytes a multiple of 16: cp.async of 16-byte chunks
    float score_scale;      // softmax scale * log2(e) / sqrt(128)
};

// Shared memory: the decoded tiles (the rotated-query tile overlays them before the first
// tile), the staged raw bytes (two buffers, K and V), the norms; the output staging of the
// epilogue overlays everything.
struct PrefillTiles {
    alignas(16) __half ks[kPfKeys * kKs];
    alignas(16) __half vs[kPfKeys * kKs];
    alignas(16) uint8_t raw[2][2][kPfKeys * kSlot];
    alignas(16) uint8_t raw_pad[16];   // a quarter's last word pair may read 4 bytes past a slot
    float kn[kPfKeys], vn[kPfKeys];
};
static_assert(sizeof(__half) * 2 * kPfKeys * kKs == sizeof(__half) * kPfRows * kKs,
              "the query tile overlays the two decoded tiles");
constexpr size_t kPfSmem = sizeof(PrefillTiles) > sizeof(float) * kPfWarps * 16 * kOs
                               ? sizeof(PrefillTiles)
                               : sizeof(float) * kPfWarps * 16 * kOs;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// Stage the bytes of head g's block of keys t0 .. t0+63 of both caches into raw[buf]; the
// block lands at offset (block offset in the row) mod 16 of its 64-byte slot.  Rows that
// are 16-byte multiples: thread (key kk = tid / 4, chunk c = tid % 4) copies the c-th
// 16-byte chunk covering the block with cp.async (the covering chunks stay inside the
// row).  Other rows (2-byte aligned): the same threads copy the block's 2-byte words
// c, c + 4, ... with plain loads.  ok[kk] records whether the row exists (keys past the
// last position any query of the CTA sees are not staged).
template <int TK, int TV>
__device__ __forceinline__ void stage_tile(const PrefillParams &p, int g, int64_t t0,
                                           int64_t n_keys, uint8_t *raw_k, uint8_t *raw_v,
                                           uint8_t *ok_k, uint8_t *ok_v) {
    const int kk = threadIdx.x >> 2, c = threadIdx.x & 3;
    const int64_t t = t0 + kk;
    const CacheView *cs[2] = {&p.kc, &p.vc};
    uint8_t *raw[2] = {raw_k, raw_v};
    uint8_t *ok[2] = {ok_k, ok_v};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const CacheView &cv = *cs[i];
        const uint8_t *row = t < n_keys ? row_ptr(cv, p.seq, t) : nullptr;
        const int bb = i == 0 ? block_bytes(TK) : block_bytes(TV);
        const int bo = g * bb;
        const int c0 = bo & ~15, end = (bo + bb + 15) & ~15;
        if (row) {
            if (i == 0 ? p.chunked_k : p.chunked_v) {
                if (c0 + 16 * c < end)
                    cp_async16(smem_u32(raw[i] + kk * kSlot + 16 * c), row + c0 + 16 * c);
            } else {
                const uint16_t *src = reinterpret_cast<const uint16_t *>(row + bo);
                uint16_t *dst = reinterpret_cast<uint16_t *>(raw[i] + kk * kSlot + (bo - c0));
                for (int w = c; w < bb / 2; w += 4) dst[w] = src[w];
            }
        }
        if (c == 0) ok[i][kk] = row ? 1 : 0;
    }
}

// Decode one cache's staged tile into fp16 centroid values dst[key][coord] and norms:
// thread (key kk = tid / 4, quarter q4 = tid % 4) does values 32 q4 .. 32 q4 + 31.
template <int TYPE>
__device__ __forceinline__ void decode_tile(const uint8_t *raw, const uint8_t *ok, int g,
                                            const HalfTables &tab, __half *dst, float *norm) {
    constexpr int B = block_bytes(TYPE);
    const int kk = threadIdx.x >> 2, q4 = threadIdx.x & 3;
    const uint8_t *slot = raw + kk * kSlot;
    const int off = (g * B) & 15;   // the block's offset in its first chunk
    const Shifts sh = {2u, 4u, 1u << 16, 1u << 30, 1u << 31};
    const Quarter<TYPE> qw = load_quarter<TYPE>(slot, (off + 2 + 8 * q4) & ~3,
                                                (off + 34 + 4 * q4) & ~3,
                                                (uint32_t)((off + 2) & 3) * 8u);
    __half *d = dst + kk * kKs + 32 * q4;
#pragma unroll
    for (int ww = 0; ww < 2; ++ww)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            uint32_t o[4];
            group_pairs<TYPE>(qw, ww, r, tab, sh, o);
            *reinterpret_cast<uint4 *>(d + 16 * ww + 8 * r) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    if (q4 == 0) norm[kk] = ok[kk] ? ld_norm(slot + off) : 0.f;
}

template <int TK, int TV>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const PrefillParams p) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(128) uint8_t smem[];
    PrefillTiles &sm = *reinterpret_cast<PrefillTiles *>(smem);
    __shared__ uint8_t ok[2][2][kPfKeys];   // [buffer][K/V][key]: row present
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, q4 = lane & 3;
    const int g = blockIdx.y, G = p.group, Hq = p.n_q_heads;
    const int64_t j0 = (int64_t)blockIdx.x * p.bq;        // first query token of the CTA
    const int64_t j_end = min64(p.n_q, j0 + p.bq);
    const int64_t n_keys = p.pos0 + j_end;                 // rows the CTA's last query sees
    const int n_tiles = (int)((n_keys + kPfKeys - 1) / kPfKeys);

    stage_tile<TK, TV>(p, g, 0, n_keys, sm.raw[0][0], sm.raw[0][1], ok[0][0], ok[0][1]);
    cp_async_commit();

    // ---- rotated, scaled queries, row r = (query j0 + r / G, head g G + r % G), into the
    // A fragments of this warp's 16 rows (the query tile overlays the decoded K/V tiles)
    __half *qt = sm.ks;
    for (int r = warp; r < kPfRows; r += kPfWarps) {
        const int jl = r / G, hl = r - jl * G;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (jl < p.bq && j0 + jl < p.n_q) {
            const __half *src = p.q + ((j0 + jl) * Hq + g * G + hl) * (int64_t)kBlock + 4 * lane;
            const uint2 raw = *reinterpret_cast<const uint2 *>(src);
            const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
            const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
            v[0] = f01.x;
            v[1] = f01.y;
            v[2] = f23.x;
            v[3] = f23.y;
            apply_signs4(v, p.kc, 4 * lane);   // rotation W D of the K cache
            warp_fwht4(v, lane);
        }
        *reinterpret_cast<uint2 *>(qt + r * kKs + 4 * lane) =
            make_uint2(pack_half2(v[0] * p.score_scale, v[1] * p.score_scale),
                       pack_half2(v[2] * p.score_scale, v[3] * p.score_scale));
    }
    __syncthreads();
    uint32_t qa[8][4];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        ldsm_x4(smem_u32(qt + (16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1)) * kKs + 16 * ks +
                         8 * (lane >> 4)),
                qa[ks]);
    __syncthreads();   // the decoded tiles overwrite the query tile

    // positions of this thread's two rows (g8 and g8 + 8); rows past the chunk are never
    // masked and never written
    int64_t qpos[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int jl = (16 * warp + g8 + 8 * i) / G;
        qpos[i] = (jl < p.bq && j0 + jl < p.n_q) ? p.pos0 + j0 + jl : INT64_MAX;
    }
    const HalfTables tk = make_tables<TK>(), tv = make_tables<TV>();
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;

    for (int it = 0; it < n_tiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < n_tiles)
            stage_tile<TK, TV>(p, g, (int64_t)(it + 1) * kPfKeys, n_keys, sm.raw[buf ^ 1][0],
                               sm.raw[buf ^ 1][1], ok[buf ^ 1][0], ok[buf ^ 1][1]);
        cp_async_commit();
        cp_async_wait<1>();   // this tile's bytes have landed
        __syncthreads();
        decode_tile<TK>(sm.raw[buf][0], ok[buf][0], g, tk, sm.ks, sm.kn);
        decode_tile<TV>(sm.raw[buf][1], ok[buf][1], g, tv, sm.vs, sm.vn);
        __syncthreads();
        const int64_t t0 = (int64_t)it * kPfKeys;

        // ---- scores S[row, key] = Q~ . C_k (then times |k|), 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {   // k-steps 2 kp and 2 kp + 1
                uint32_t b[4];
                ldsm_x4(smem_u32(sm.ks + (8 * nt + (lane & 7)) * kKs + 32 * kp + 8 * (lane >> 3)), b);
                mma16816(s[nt], qa[2 * kp][0], qa[2 * kp][1], qa[2 * kp][2], qa[2 * kp][3], b[0], b[1]);
                mma16816(s[nt], qa[2 * kp + 1][0], qa[2 * kp + 1][1], qa[2 * kp + 1][2],
                         qa[2 * kp + 1][3], b[2], b[3]);
            }
        }
        // ---- |k|, causal mask, online softmax (log2 domain)
        float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kc = 8 * nt + 2 * q4 + (e & 1);
                const float v = s[nt][e] * sm.kn[kc];
                s[nt][e] = t0 + kc > qpos[e >> 1] ? -INFINITY : v;
                mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
            }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        }
        float alpha[2], psum[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            alpha[i] = m_run[i] == -INFINITY ? 0.f : ex2(m_run[i] - mx[i]);
            m_run[i] = mx[i];
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mm = mx[e >> 1];
                const float pr = mm == -INFINITY ? 0.f : ex2(s[nt][e] - mm);
                psum[e >> 1] += pr;
                s[nt][e] = pr * sm.vn[8 * nt + 2 * q4 + (e & 1)];   // weight of the value row
            }
#pragma unroll
        for (int i = 0; i < 2; ++i) l_run[i] = l_run[i] * alpha[i] + psum[i];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            o[nt][0] *= alpha[0];
            o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1];
            o[nt][3] *= alpha[1];
        }
        // ---- O[row, coord] += (p |v|) . C_v: A from the score accumulators, B by ldmatrix.trans
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // keys 16 kk .. 16 kk + 15
            const uint32_t a0 = pack_half2(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t a1 = pack_half2(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t a2 = pack_half2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t a3 = pack_half2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // coords 16 c .. 16 c + 15
                uint32_t b[4];
                ldsm_x4_trans(smem_u32(sm.vs + (16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7)) * kKs +
                                       16 * c + 8 * (lane >> 4)),
                              b);
                mma16816(o[2 * c], a0, a1, a2, a3, b[0], b[1]);
                mma16816(o[2 * c + 1], a0, a1, a2, a3, b[2], b[3]);
            }
        }
        __syncthreads();   // the next tile's decode overwrites ks / vs
    }
    cp_async_wait<0>();

    // ---- epilogue: divide by the row sums, inverse rotation per row, write
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
        l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
    }
    const float inv[2] = {l_run[0] > 0.f ? kInvSqrt128 / l_run[0] : 0.f,
                          l_run[1] > 0.f ? kInvSqrt128 / l_run[1] : 0.f};
    __syncthreads();   // the staging rows overlay the tiles
    float *os = reinterpret_cast<float *>(smem) + warp * 16 * kOs;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i)
            *reinterpret_cast<float2 *>(os + (g8 + 8 * i) * kOs + 8 * nt + 2 * q4) =
                make_float2(o[nt][2 * i] * inv[i], o[nt][2 * i + 1] * inv[i]);
    __syncwarp();
    for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * warp + rr, jl = r / G, hl = r - jl * G;
        if (jl >= p.bq || j0 + jl >= p.n_q) break;   // rows only grow from here
        float4 a = *reinterpret_cast<const float4 *>(os + rr * kOs + 4 * lane);
        float v[4] = {a.x, a.y, a.z, a.w};
        warp_fwht4(v, lane);   // (1/sqrt(128)) W o, the 1/sqrt(128) folded into inv
        apply_signs4(v, p.vc, 4 * lane);     // inverse D W of the V cache
        *reinterpret_cast<float4 *>(p.out + ((j0 + jl) * Hq + g * G + hl) * (int64_t)kBlock + 4 * lane) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

template <int TK, int TV>
tq_status launch_prefill_t(const PrefillParams &p, unsigned grid_x, unsigned n_kv_heads,
                           cudaStream_t stream) {
    if (cudaFuncSetAttribute(prefill_kernel<TK, TV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPfSmem) != cudaSuccess)
        return TQ_ERR_CUDA;
    PdlConfig lc(dim3(grid_x, n_kv_heads), dim3(kPfThreads), kPfSmem, stream);
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, prefill_kernel<TK, TV>, p));
}

}  // namespace

bool prefill_supported(const tq_cache &k, const tq_cache &v, int n_q_heads) {
    if (k.head_dim != kBlock || v.head_dim != kBlock) return false;
    return n_q_heads % k.n_kv_heads == 0 && n_q_heads / k.n_kv_heads <= kPfRows;
}

tq_status launch_prefill(const tq_cache &k, const tq_cache &v, const void *q, int32_t seq_id,
                         int64_t pos0, int64_t n_q, int n_q_heads, float scale, float *out,
                         cudaStream_t stream) {
    if (!prefill_supported(k, v, n_q_heads)) return TQ_ERR_UNSUPPORTED;
    if (n_q == 0) return TQ_OK;
    if (kUseTcgen05)
        return launch_prefill_tc(k, v, q, seq_id, pos0, n_q, n_q_heads, scale, out, stream);
    PrefillParams p;
    p.kc = make_view(k);
    p.vc = make_view(v);
    p.q = static_cast<const __half *>(q);
    p.out = out;
    p.pos0 = pos0;
    p.n_q = n_q;
    p.seq = seq_id;
    p.n_q_heads = n_q_heads;
    p.group = n_q_heads / k.n_kv_heads;
    p.bq = kPfRows / p.group;
    p.score_scale = scale * kPfLog2e * kInvSqrt128;
    p.chunked_k = p.kc.row_bytes % 16 == 0;
    p.chunked_v = p.vc.row_bytes % 16 == 0;
    const int64_t grid_x = (n_q + p.bq - 1) / p.bq;
    if (grid_x > 0x7fffffff) return TQ_ERR_UNSUPPORTED;
    const unsigned gx = (unsigned)grid_x, hk = (unsigned)k.n_kv_heads;
    if (k.type == TQ_TURBO3 && v.type == TQ_TURBO3) return launch_prefill_t<3, 3>(p, gx, hk, stream);
    if (k.type == TQ_TURBO2 && v.type == TQ_TURBO2) return launch_prefill_t<2, 2>(p, gx, hk, stream);
    if (k.type == TQ_TURBO3 && v.type == TQ_TURBO2) return launch_prefill_t<3, 2>(p, gx, hk, stream);
    return launch_prefill_t<2, 3>(p, gx, hk, stream);
}

}  // namespace tq
