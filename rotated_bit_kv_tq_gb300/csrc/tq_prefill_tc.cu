// tq_prefill_tc.cu -- causal prompt-chunk attention over the packed cache on the 5th-generation
// tensor cores (tcgen05: operands in shared memory, accumulators in tensor memory).
//
// "llama.cpp に TurboQuant を実装": prompt processing runs over the compressed cache as well
// ("Numbers on real models"), and the roadmap fuses the dequantisation into the Flash-
// Attention tiles so that K is never materialised in FP16 in HBM ("Current implementation
// and what's next").  Query token j of the chunk sits at position pos0 + j and attends to
// rows 0 .. pos0 + j (TinyLLaMA article, section 7, at every position of the chunk).
// Everything stays in the rotated domain; each output row gets one inverse FWHT at the end.
//
// One decoded K/V tile serves every query row of a CTA, so the products are a dense
// contraction and run on the tensor cores.  The work split follows the roles the
// tensor-memory model suggests:
//  - warps 0-7, two threads per row of the 128-row tile (row = TMEM lane, warps q and q + 4
//    share lanes 32q..32q+31), each thread owning 64 of a tile's 128 keys: rotate the
//    queries into shared memory; per key tile read the scores S from TMEM, scale by |k|,
//    mask on the diagonal tiles, exchange the row maximum with the partner thread, write P
//    (fp16) into tensor memory, rescale O there when the running maximum moved; at the
//    end read O, divide, inverse-FWHT the row (the last butterfly across the pair) and
//    store it;
//  - warps 8-11 (K) and 12-15 (V), one thread per key: stage the tile's block bytes
//    (cp.async) and decode them once into fp16 values laid out as the MMA operands (K:
//    centroids, keys x coords, K-major, norms apart; V: |v| times centroids, keys x coords
//    with coords contiguous, MN-major), double-buffered;
//  - warp 16: allocates TMEM and issues the MMAs from one thread, in whichever order their
//    inputs become ready: S[b] = Q~ K^T (M = 128 rows, N = 128 keys, K = 128 coords; Q~ is
//    an fp16 pair hi + lo, two MMAs per k-step, and the centroid table is scaled to be nearly
//    exact in fp16, Codebook::h_scale) into
//    one of two TMEM score buffers, and O += P V with P read from one of two TMEM buffers
//    (N = 128 coords, K = 128 keys); completions arrive on mbarriers through
//    tcgen05.commit.
// Shared-memory operands use the no-swizzle canonical layout: 8 x 16-byte core matrices,
// core matrices adjacent along K 128 bytes apart (LBO), 8-row groups along M/N 2048 bytes
// apart (SBO).  Every wait is bounded; a timeout records TQ_ERR_DEVICE_TIMEOUT and the CTA
// still releases its tensor memory.
#include <cmath>

#include "tq_internal.cuh"
#include "tq_simd.cuh"
#include "tq_codes.cuh"

namespace tq {
namespace {

constexpr int kTcRows = 128;          // (query token, head) rows per CTA = TMEM lanes
constexpr int kTcKeys = 128;          // keys per tile
constexpr int kTcSoftmax = 256;       // warps 0-7: two threads per row (one per 64-key half)
constexpr int kTcGroup = 128;         // threads of one producer group (warps 8-11 K, 12-15 V)
constexpr int kTcProducer = 2 * kTcGroup;
constexpr int kTcMmaWarp = (kTcSoftmax + kTcProducer) / 32;
constexpr int kTcThreads = kTcSoftmax + kTcProducer + 32;
constexpr uint32_t kTcWaitLimit = 1u << 20;
constexpr uint32_t kTcPollLimit = 1u << 24;   // polls without progress of the MMA thread
// tensor memory columns: S0 [0,128), S1 [128,256), O [256,384) fp32; P0 [384,448),
// P1 [448,512) fp16 pairs (the A operand of P V)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256, kTmemP = 384;
constexpr float kTcLog2e = 1.4426950408889634f;

// mbarriers
// Buffer b of a double-buffered resource serves tiles b, b + 2, ...; a waiter for tile i
// waits for phase i >> 1 of barrier b, which is safe because no barrier can run more than
// one phase ahead of (or behind) its waiters: each role waits for the previous use of a
// buffer before it arrives for the next.
enum {
    kBarQ = 0,          // queries written (128 arrivals)
    kBarKFull = 1,      // [2] K tile and its norms decoded (128 arrivals)
    kBarVFull = 3,      // [2] V tile decoded (128 arrivals)
    kBarPvFree = 5,     // [2] the tile's P V done: V tile and P buffer free (commit)
    kBarSFull = 7,      // [2] scores ready (commit)
    kBarSFree = 9,      // [2] scores and K norms read (128 arrivals); implies the S MMAs are done
    kBarPFull = 11,     // [2] P written, O rescaled (128 arrivals)
    kBarDrain = 13,     // every MMA of the CTA done (commit), before TMEM is released
    kBarCount = 14
};

struct TcParams {
    CacheView kc, vc;
    const __half *q;        // [n_q][Hq][128] fp16
    float *out;             // [n_q][Hq][128] fp32
    int64_t pos0, n_q;
    int32_t seq, n_q_heads, group, bq;
    int32_t n_kv_heads;
    int64_t n_qblocks;      // query blocks of bq tokens
    int32_t chunked_k, chunked_v;
    float score_scale;      // softmax scale * log2(e) / (sqrt(128) * h_scale of the K table)
    float out_scale;        // 1 / (sqrt(128) * h_scale of the V table)
    int32_t split;          // CTAs per query block: 1, or 2 (a cluster: key tiles cut in two halves)
};

struct TcSmem {
    alignas(1024) uint8_t q[32768];        // Q~ high fp16 parts [row][coord], K-major
    alignas(1024) uint8_t ql[32768];       // Q~ low parts (fp16 rounding of the remainder)
    alignas(1024) uint8_t k[2][32768];     // K tile [key][coord], K-major
    alignas(1024) uint8_t v[2][32768];     // V tile [key][coord], coords contiguous (MN-major)
    alignas(16) uint8_t raw[2][kTcKeys * 64];   // staged blocks of one tile (K, V), 64-byte key windows
    float kn[2][kTcKeys];                  // K norms of the two tile buffers
    float xch[2][2][kTcRows];              // [tile parity][half][row] row maxima, then sums
    uint8_t ok[2][kTcKeys];                // [K/V][key] row present
    alignas(8) uint64_t bar[kBarCount];
    uint32_t tmem;
};

// Byte offset of element (r, c) of a 128-column tile in the no-swizzle canonical layout with
// rows along M/N (8-row groups 2048 bytes apart) and columns along K (8-column groups 128
// bytes apart).
__device__ __forceinline__ uint32_t canon(int r, int c) {
    return (uint32_t)((r >> 3) * 2048 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}
// The MN-major V tile: keys are K (8-key groups 2048 bytes apart), coords are N (8-coord
// groups 128 bytes apart), coords contiguous inside a core matrix.
__device__ __forceinline__ uint32_t canon_mn(int key, int c) {
    return (uint32_t)((c >> 3) * 128 + (key >> 3) * 2048 + (key & 7) * 16 + (c & 7) * 2);
}

// Shared-memory matrix descriptor (no swizzle): start, leading (K) and stride (M/N) byte
// offsets in 16-byte units, descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, M = 128, N = 128.
constexpr uint32_t idesc_f16(bool b_mn_major) {
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// The same with A read from tensor memory (row m = lane m, two fp16 K values per column).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
          "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]),
          "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]),
          "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])),
          "r"(__float_as_uint(r[2])), "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])),
          "r"(__float_as_uint(r[5])), "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])),
          "r"(__float_as_uint(r[8])), "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])),
          "r"(__float_as_uint(r[11])), "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])),
          "r"(__float_as_uint(r[14])), "r"(__float_as_uint(r[15])), "r"(__float_as_uint(r[16])),
          "r"(__float_as_uint(r[17])), "r"(__float_as_uint(r[18])), "r"(__float_as_uint(r[19])),
          "r"(__float_as_uint(r[20])), "r"(__float_as_uint(r[21])), "r"(__float_as_uint(r[22])),
          "r"(__float_as_uint(r[23])), "r"(__float_as_uint(r[24])), "r"(__float_as_uint(r[25])),
          "r"(__float_as_uint(r[26])), "r"(__float_as_uint(r[27])), "r"(__float_as_uint(r[28])),
          "r"(__float_as_uint(r[29])), "r"(__float_as_uint(r[30])), "r"(__float_as_uint(r[31]))
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
          "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
          "r"(r[14]), "r"(r[15])
        : "memory");
}

// 64 consecutive fp32 columns of this thread's TMEM lane (two loads, one wait, in one
// statement so that no use of the values can be scheduled before the wait).
__device__ __forceinline__ void tc_ld64(uint32_t taddr, float (&r)[64]) {
    uint32_t u[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
        "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
          "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]),
          "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]),
          "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]),
          "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]), "=r"(u[37]),
          "=r"(u[38]), "=r"(u[39]), "=r"(u[40]), "=r"(u[41]), "=r"(u[42]), "=r"(u[43]),
          "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47]), "=r"(u[48]), "=r"(u[49]),
          "=r"(u[50]), "=r"(u[51]), "=r"(u[52]), "=r"(u[53]), "=r"(u[54]), "=r"(u[55]),
          "=r"(u[56]), "=r"(u[57]), "=r"(u[58]), "=r"(u[59]), "=r"(u[60]), "=r"(u[61]),
          "=r"(u[62]), "=r"(u[63])
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) r[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tc_bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void tc_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool tc_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait on a phase; false (and TQ_ERR_DEVICE_TIMEOUT recorded) on timeout.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kTcWaitLimit; ++it) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}\n"
                     : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
    }
    record_error(TQ_ERR_DEVICE_TIMEOUT);
    return false;
}
// Cluster-wide barrier, each thread on its own (not warp-aligned): every thread of both CTAs
// of a split query block passes it exactly twice (before and after the partial exchange).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local, uint32_t rank) {
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t local, uint32_t rank) {
    uint32_t ra;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra) : "memory");
    return v;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Staged tile bytes are key-major: key k owns the 64 bytes at k * 64 of the cache's staging
// area, a window of its row that starts at the 16-byte boundary at or below the block (the
// block sits at window byte (block offset in the row) mod 16, and 14 + 50 bytes fit).  The
// window's 16-byte chunk c is stored at chunk c ^ ((k >> 1) & 3), so that 8 consecutive keys'
// 16-byte accesses to one chunk cover the 32 banks once (the copies that fill it, and the
// decode threads, one per key, reading it back).
__device__ __forceinline__ uint32_t win_chunk(int key, int c) {
    return (uint32_t)(key * 64 + ((c ^ ((key >> 1) & 3)) << 4));
}

// Producer thread pt of a group stages key pt of tile [t0, t0 + keys) of its cache: the
// 16-byte chunks covering head g's block with cp.async when rows are 16-byte multiples (so
// the chunks are aligned and lie inside the row), else the block's 2-byte halves with plain
// loads.
template <int TYPE>
__device__ __forceinline__ void tc_stage(const CacheView &cv, int32_t seq, bool chunked,
                                         uint8_t *raw, uint8_t *ok, int g, int64_t t0,
                                         int64_t n_keys, int pt) {
    const int64_t t = t0 + pt;
    const uint8_t *row = t < n_keys ? row_ptr(cv, seq, t) : nullptr;
    constexpr int bb = block_bytes(TYPE);
    const int bo = g * bb, x0 = bo & ~15, lead = bo & 15;
    if (row) {
        if (chunked) {
            const int nc = (lead + bb + 15) >> 4;   // chunks up to the one holding the last byte
            for (int c = 0; c < nc; ++c) cp_async16(smem_u32(raw + win_chunk(pt, c)), row + x0 + 16 * c);
        } else {
            // 2-byte aligned rows: half h of the block goes to window byte lead + 2h
            const uint16_t *src = reinterpret_cast<const uint16_t *>(row + bo);
            for (int h = 0; h < bb / 2; ++h) {
                const int wb = lead + 2 * h;
                *reinterpret_cast<uint16_t *>(raw + win_chunk(pt, wb >> 4) + (wb & 15)) = src[h];
            }
        }
    }
    ok[pt] = row ? 1 : 0;
}

// Producer thread pt reads key pt's staged window and brings its block to byte 0:
// n[j] = block bytes 4j .. 4j + 3.  The block's offset in the window, lead (its offset in the
// row mod 16), is the same for all keys of a warp; one code path serves every head (a form
// templated on lead overflowed the instruction cache): a word shift by lead >> 2 in two
// select levels, then a funnel shift by the remaining 0 or 2 bytes.  The staging area is
// free again once this returns.
template <int TYPE>
__device__ __forceinline__ void tc_window(const uint8_t *raw, int g, int pt, uint32_t (&n)[13]) {
    constexpr int B = block_bytes(TYPE);
    uint32_t w[17];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(raw + win_chunk(pt, c));
        w[4 * c] = u.x;
        w[4 * c + 1] = u.y;
        w[4 * c + 2] = u.z;
        w[4 * c + 3] = u.w;
    }
    w[16] = 0u;
    const int lead = (g * B) & 15;
    const bool s1 = lead & 4, s2 = lead & 8;
    const uint32_t sh = 8u * (uint32_t)(lead & 3);
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = s1 ? w[j + 1] : w[j];
#pragma unroll
    for (int j = 0; j < 14; ++j) w[j] = s2 ? w[j + 2] : w[j];
#pragma unroll
    for (int j = 0; j < 13; ++j) n[j] = __funnelshift_r(w[j], w[j + 1], sh);
}

// Producer thread pt decodes key pt from its block bytes n (tc_window): K into fp16
// centroids at tile[key][coord] (K-major) and its norm into norm[key]; V into fp16 |v| c
// (MN-major).  Absent rows get norm 0.
// NC, c_off (MN only): the tile holds NC coordinates and this block fills coordinates
// c_off .. c_off + 127 (8-key groups NC * 16 bytes apart).
template <int TYPE, bool MN, int NC = 128>
__device__ __forceinline__ void tc_decode(const uint32_t (&n)[13], bool present,
                                          const HalfTables &tab, uint8_t *tile, float *norm,
                                          int pt, int c_off = 0) {
    const Shifts shifts = {2u, 4u, 1u << 16, 1u << 30, 1u << 31};
    // the norm: block bytes 0-1, 0 for an absent row.  V folds it into the tile values
    // (|v| c); K keeps it apart (norm[]) and the scores are scaled in fp32, which keeps one
    // fp16 rounding on the score path
    const __half nrm = present ? __ushort_as_half((uint16_t)(n[0] & 0xffffu)) : __ushort_as_half(0);
    const __half2 n2 = __halves2half2(nrm, nrm);
    if (!MN) norm[pt] = __half2float(nrm);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        // the quarter's low-plane bytes are block bytes 2 + 8 q4 .., its high-plane word
        // block bytes 34 + 4 q4 ..
        Quarter<TYPE> qw;
        qw.W0 = __funnelshift_r(n[2 * q4], n[2 * q4 + 1], 16);
        qw.W1 = __funnelshift_r(n[2 * q4 + 1], n[2 * q4 + 2], 16);
        if (TYPE == TQ_TURBO3) qw.V = __funnelshift_r(n[8 + q4], n[9 + q4], 16);
        else qw.V = 0u;
#pragma unroll
        for (int ww = 0; ww < 2; ++ww)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                uint32_t o[4];
                group_pairs<TYPE>(qw, ww, r, tab, shifts, o);
                if (MN) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __half2 h = __hmul2(*reinterpret_cast<const __half2 *>(&o[e]), n2);
                        o[e] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                }
                const int c0 = 32 * q4 + 16 * ww + 8 * r;
                const uint32_t at = MN ? (uint32_t)(((c_off + c0) >> 3) * 128 + (pt >> 3) * (NC * 16) + (pt & 7) * 16)
                                       : canon(pt, c0);
                *reinterpret_cast<uint4 *>(tile + at) = make_uint4(o[0], o[1], o[2], o[3]);
            }
    }
}

// In-thread Walsh-Hadamard butterflies over 64 values, h = 1 .. 32.
__device__ __forceinline__ void fwht64(float (&x)[64]) {
#pragma unroll
    for (int h = 1; h < 64; h <<= 1)
#pragma unroll
        for (int i = 0; i < 64; ++i)
            if (!(i & h)) {
                const float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

// One producer group: stage and decode every tile of its cache (K: centroids and norms;
// V: |v| c), double-buffered.  Each thread reads back only the bytes it staged itself, so
// the group needs no barrier of its own.  Tile i's bytes are read into registers first, and
// tile i + 1's copies go out before the wait for the tile buffer: tile buffer b is rewritten
// once the consumers of tile i - 2 are done with it (K: the softmax has read that tile's
// scores and norms; V: its P V has completed).
template <int TYPE, bool IS_V>
__device__ __forceinline__ void tc_produce(const TcParams &p, TcSmem &sm, int g, int64_t n_keys,
                                           int tile0, int n_tiles, int pt, volatile int *abort_v) {
    const CacheView &cv = IS_V ? p.vc : p.kc;
    const bool chunked = IS_V ? p.chunked_v : p.chunked_k;
    uint8_t *raw = sm.raw[IS_V ? 1 : 0];
    uint8_t *ok = sm.ok[IS_V ? 1 : 0];
    const HalfTables tab = make_tables<TYPE>();
    const int free_bar = IS_V ? kBarPvFree : kBarSFree, full_bar = IS_V ? kBarVFull : kBarKFull;
    if (n_tiles > 0) tc_stage<TYPE>(cv, p.seq, chunked, raw, ok, g, (int64_t)tile0 * kTcKeys, n_keys, pt);
    cp_async_commit();
    for (int i = 0; i < n_tiles; ++i) {
        const int b = i & 1;
        cp_async_wait<0>();   // this thread's bytes of tile i have landed
        uint32_t nb[13];
        tc_window<TYPE>(raw, g, pt, nb);
        const bool present = ok[pt] != 0;
        if (i + 1 < n_tiles) tc_stage<TYPE>(cv, p.seq, chunked, raw, ok, g, (int64_t)(tile0 + i + 1) * kTcKeys, n_keys, pt);
        cp_async_commit();
        if (i >= 2 && !*abort_v &&
            !tc_wait(smem_u32(&sm.bar[free_bar + b]), (uint32_t)(((i - 2) >> 1) & 1)))
            *abort_v = 1;
        if (IS_V) tc_decode<TYPE, true>(nb, present, tab, sm.v[b], nullptr, pt);
        else tc_decode<TYPE, false>(nb, present, tab, sm.k[b], sm.kn[b], pt);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_arrive(smem_u32(&sm.bar[full_bar + b]));
    }
    cp_async_wait<0>();
}

template <int TK, int TV>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const TcParams p) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem_raw[];   // 16: the runtime guarantees no more
    // the MMA operand tiles must start on a 1024-byte boundary of the shared window (the
    // dynamic block itself may start after static shared memory at a lower alignment)
    TcSmem &sm = *reinterpret_cast<TcSmem *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTAs run longest first: the last query block (the most keys) of every head first.  With
    // split = 2, the two CTAs of a cluster share a query block: rank 0 takes the first half of
    // its key tiles, rank 1 the rest, and they merge their partial outputs at the end.
    const unsigned qcta = p.split == 2 ? blockIdx.x >> 1 : blockIdx.x;
    const int rank = p.split == 2 ? (int)(blockIdx.x & 1u) : 0;   // the cluster rank
    const int g = (int)(qcta % (unsigned)p.n_kv_heads), G = p.group, Hq = p.n_q_heads;
    const int64_t j0 = (p.n_qblocks - 1 - (int64_t)(qcta / (unsigned)p.n_kv_heads)) * p.bq;
    const int64_t j_end = min64(p.n_q, j0 + p.bq);
    const int64_t n_keys = p.pos0 + j_end;                  // rows the CTA's last query sees
    const int64_t first_pos = p.pos0 + j0;                  // the CTA's first query position
    const int n_all = (int)((n_keys + kTcKeys - 1) / kTcKeys);
    const int half_tiles = (n_all + 1) / 2;
    const int tile0 = p.split == 2 && rank == 1 ? half_tiles : 0;          // first key tile
    const int n_tiles = p.split == 2 ? (rank == 0 ? half_tiles : n_all - half_tiles) : n_all;
    auto bar = [&](int i) { return smem_u32(&sm.bar[i]); };

    if (tid == 0) {
        abort_flag = 0;
        tc_bar_init(bar(kBarQ), kTcSoftmax);
        for (int b = 0; b < 2; ++b) {
            tc_bar_init(bar(kBarKFull + b), kTcGroup);
            tc_bar_init(bar(kBarVFull + b), kTcGroup);
            tc_bar_init(bar(kBarPvFree + b), 1);
            tc_bar_init(bar(kBarPFull + b), kTcSoftmax);
            tc_bar_init(bar(kBarSFull + b), 1);
            tc_bar_init(bar(kBarSFree + b), kTcSoftmax);
        }
        tc_bar_init(bar(kBarDrain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&sm.tmem)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    volatile int *abort_v = &abort_flag;

    if (warp < kTcSoftmax / 32) {
        // ================= softmax: thread (r, h) owns keys 64 h .. 64 h + 63 of every tile
        // for row r = TMEM lane r (warps quad and quad + 4 share the lanes of quad)
        const int quad = warp & 3, h = warp >> 2;
        const int r = 32 * quad + lane, jl = r / G, hl = r - jl * G;
        const bool valid = jl < p.bq && j0 + jl < p.n_q;
        const int64_t qpos = valid ? p.pos0 + j0 + jl : INT64_MAX;
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint32_t pair_bar = 3u + (uint32_t)quad;   // named barrier of the row's two threads
        {
            // coords 64 h .. 64 h + 63 of Q~ = H (D q) * scale: the stride-64 butterfly straight
            // from the loaded row, then strides 1 .. 32 inside the thread
            float x[64];
            if (valid) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.q + ((j0 + jl) * Hq + g * G + hl) * (int64_t)kBlock);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 ua = src[c], ub = src[c + 8];   // coords 8 c .. and 64 + 8 c ..
                    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = 8 * c + 2 * e;
                        const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[e]));
                        const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[e]));
                        float a0 = fa.x, a1 = fa.y, b0 = fb.x, b1 = fb.y;
                        if (p.kc.has_signs) {
                            a0 = __uint_as_float(__float_as_uint(a0) ^ sign_mask(p.kc, i0));
                            a1 = __uint_as_float(__float_as_uint(a1) ^ sign_mask(p.kc, i0 + 1));
                            b0 = __uint_as_float(__float_as_uint(b0) ^ sign_mask(p.kc, 64 + i0));
                            b1 = __uint_as_float(__float_as_uint(b1) ^ sign_mask(p.kc, 64 + i0 + 1));
                        }
                        x[i0] = h ? a0 - b0 : a0 + b0;
                        x[i0 + 1] = h ? a1 - b1 : a1 + b1;
                    }
                }
                fwht64(x);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) x[i] = 0.f;
            }
            // Q~ = hi + lo, both fp16: the scores take both (two MMAs per k-step), so the
            // query keeps about 22 bits
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t w[4], wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    split_half2(x[8 * c + 2 * e] * p.score_scale, x[8 * c + 2 * e + 1] * p.score_scale, w[e], wl[e]);
                *reinterpret_cast<uint4 *>(sm.q + canon(r, 64 * h + 8 * c)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(sm.ql + canon(r, 64 * h + 8 * c)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_arrive(bar(kBarQ));

        float m_run = -INFINITY, l_run = 0.f;   // l_run: this half's share of the row sum
        // every thread runs every tile (the TMEM accesses and the pair barrier are
        // collective); after a timeout the remaining waits are skipped
        for (int i = 0; i < n_tiles; ++i) {
            const int b = i & 1;
            if (!*abort_v && !tc_wait(bar(kBarSFull + b), (uint32_t)((i >> 1) & 1))) *abort_v = 1;
            tc_fence_after();
            float s[64];
            tc_ld64(tmem + lane_base + 128u * b + 64u * h, s);
            const float *kn = sm.kn[b] + 64 * h;
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = m_run;
            if ((int64_t)(tile0 + i) * kTcKeys + (kTcKeys - 1) <= first_pos) {
                // every key of the tile is visible to every row of the CTA
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s[j] *= kn[j];
                    mx8[j & 7] = fmaxf(mx8[j & 7], s[j]);
                }
            } else {
                // keys past this row's position are masked
                const int64_t t0 = (int64_t)(tile0 + i) * kTcKeys + 64 * h;
                const int lim = (int)max64(-1, min64(qpos - t0, 64));   // keys j > lim are masked
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    s[j] = j > lim ? -INFINITY : s[j] * kn[j];
                    mx8[j & 7] = fmaxf(mx8[j & 7], s[j]);
                }
            }
            // S buffer b and the K norms of tile buffer b are free for tile i + 2
            tc_fence_before();
            tc_arrive(bar(kBarSFree + b));
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            // the row's maximum over both halves (exchange slot b is reused two tiles on,
            // after the partner has passed the next pair barrier)
            sm.xch[b][h][r] = mx;
            named_sync(pair_bar, 64);
            mx = fmaxf(mx, sm.xch[b][h ^ 1][r]);
            // lazy rescaling: the reference maximum moves only when the row's maximum exceeds
            // it by more than 8 (log2 units), so p <= 2^8 (fp16-safe: |v| is in the V tile) and
            // O in tensor memory is rarely rewritten; both halves take the same decisions
            float alpha = 1.f;
            if (m_run == -INFINITY || mx > m_run + 8.f) {
                alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
                m_run = mx;
            }
            // P buffer b is free once tile i - 2's P V is done
            if (i >= 2 && !*abort_v && !tc_wait(bar(kBarPvFree + b), (uint32_t)(((i - 2) >> 1) & 1)))
                *abort_v = 1;
            tc_fence_after();
            float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float mref = m_run == -INFINITY ? 0.f : m_run;   // all masked: every p is 0
            {
                float w[32];   // columns 32 h + e hold the fp16 pair of keys 64 h + 2 e, + 1
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = ex2(s[2 * e] - mref), p1 = ex2(s[2 * e + 1] - mref);
                    ps8[(2 * e) & 7] += p0;
                    ps8[(2 * e + 1) & 7] += p1;
                    w[e] = __uint_as_float(pack_half2(p0, p1));
                }
                tc_st32(tmem + lane_base + kTmemP + 64u * b + 32u * h, w);
            }
            const float psum = ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
            l_run = l_run * alpha + psum;
            if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // the running output must hold every P V up to tile i - 1 before it is scaled;
                // this half scales output columns 64 h .. 64 h + 63
                if (!*abort_v && !tc_wait(bar(kBarPvFree + ((i - 1) & 1)), (uint32_t)(((i - 1) >> 1) & 1)))
                    *abort_v = 1;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float t[32];
                    tc_ld32(tmem + lane_base + kTmemO + 64u * h + 32u * c, t);
#pragma unroll
                    for (int e = 0; e < 32; ++e) t[e] *= alpha;
                    tc_st32(tmem + lane_base + kTmemO + 64u * h + 32u * c, t);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            tc_arrive(bar(kBarPFull + b));
        }
        // ---- epilogue: O / l, inverse rotation of the row, V signs, store
        const bool done = n_tiles > 0 && !*abort_v &&
                          tc_wait(bar(kBarPvFree + ((n_tiles - 1) & 1)), (uint32_t)(((n_tiles - 1) >> 1) & 1));
        tc_fence_after();
        sm.xch[n_tiles & 1][h][r] = l_run;   // slot of tile n_tiles - 2: the partner is past it
        float o[64];
        if (n_tiles > 0) {
            tc_ld64(tmem + lane_base + kTmemO + 64u * h, o);
        } else {   // a key range with no tiles (split, one-tile prompt): nothing was accumulated
#pragma unroll
            for (int e = 0; e < 64; ++e) o[e] = 0.f;
        }
        fwht64(o);   // strides 1 .. 32 of this half
        // the stride-64 butterfly pairs coord c with c + 64: the halves swap through the K
        // tile area, idle once every MMA has completed (float4 chunks XOR-swizzled by row)
        float *xo = reinterpret_cast<float *>(sm.k[0]);
        auto xo_at = [&](int row, int c4) { return xo + row * 128 + (((c4 ^ row) & 31) << 2); };
#pragma unroll
        for (int c = 0; c < 16; ++c)
            *reinterpret_cast<float4 *>(xo_at(r, 16 * h + c)) =
                make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        named_sync(pair_bar, 64);
        float l_row = l_run + sm.xch[n_tiles & 1][h ^ 1][r];
        // y: coords 64 h .. 64 h + 63 of the rotated-back row, before the division by l
        // (h = 0: coord c' = o + partner (coords c', c' + 64); h = 1: partner - o)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float4 u = *reinterpret_cast<const float4 *>(xo_at(r, 16 * (h ^ 1) + c));
            const float pv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) o[4 * c + e] = h ? pv[e] - o[4 * c + e] : o[4 * c + e] + pv[e];
        }
        bool write = valid && done;
        if (p.split == 2) {
            // The two CTAs of the query block merge by log-sum-exp: the CTA of rank h finishes
            // coords 64 h .. of every row; the thread of the other half publishes its coords and
            // the row's (max, sum) in the V tile area (idle after the last P V) for the partner.
            float *X = reinterpret_cast<float *>(sm.v[0]);                 // [row][64]
            float *Xml = reinterpret_cast<float *>(sm.v[1]);               // [row][2]
            const float m_row = n_tiles > 0 ? m_run : -INFINITY;
            if (h != rank) {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<float4 *>(X + r * 64 + 4 * c) =
                        make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                Xml[2 * r] = m_row;
                Xml[2 * r + 1] = l_row;
            }
            cluster_sync_all();
            if (h == rank) {
                const uint32_t peer = (uint32_t)(rank ^ 1);
                const float mp = ld_cluster_f32(smem_u32(Xml + 2 * r), peer);
                const float lp = ld_cluster_f32(smem_u32(Xml + 2 * r + 1), peer);
                const float M = fmaxf(m_row, mp);
                const float wa = m_row == -INFINITY ? 0.f : ex2(m_row - M);
                const float wb = mp == -INFINITY ? 0.f : ex2(mp - M);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 u = ld_cluster_f32x4(smem_u32(X + r * 64 + 4 * c), peer);
                    o[4 * c] = wa * o[4 * c] + wb * u.x;
                    o[4 * c + 1] = wa * o[4 * c + 1] + wb * u.y;
                    o[4 * c + 2] = wa * o[4 * c + 2] + wb * u.z;
                    o[4 * c + 3] = wa * o[4 * c + 3] + wb * u.w;
                }
                l_row = wa * l_row + wb * lp;
            }
            cluster_sync_all();   // the partner has read this CTA's exchange area
            write = valid && h == rank && !*abort_v;
        }
        if (write) {
            const float inv = l_row > 0.f ? p.out_scale / l_row : 0.f;
            float4 *dst = reinterpret_cast<float4 *>(p.out + ((j0 + jl) * Hq + g * G + hl) * (int64_t)kBlock + 64 * h);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v4[e] = __uint_as_float(__float_as_uint(o[4 * c + e] * inv) ^ sign_mask(p.vc, 64 * h + 4 * c + e));
                dst[c] = make_float4(v4[0], v4[1], v4[2], v4[3]);
            }
        }
    } else if (warp < kTcMmaWarp) {
        // ================= producers: warps 8-11 the K cache, 12-15 the V cache
        const int pt = (tid - kTcSoftmax) & (kTcGroup - 1);
        if (tid - kTcSoftmax < kTcGroup) tc_produce<TK, false>(p, sm, g, n_keys, tile0, n_tiles, pt, abort_v);
        else tc_produce<TV, true>(p, sm, g, n_keys, tile0, n_tiles, pt, abort_v);
    } else if (lane == 0) {
        // ================= MMA issue (one thread)
        constexpr uint32_t idesc_s = idesc_f16(false), idesc_pv = idesc_f16(true);
        const uint32_t q_base = smem_u32(sm.q), ql_base = smem_u32(sm.ql);
        bool ok = tc_wait(bar(kBarQ), 0);
        // issue S(ns) and P V(npv) in whichever order their inputs become ready: S(i + 1)
        // must not hold back P V(i) while tile i + 1 is still being decoded
        int ns = 0, npv = 0;
        uint32_t idle = 0;
        while (ok && npv < n_tiles) {
            bool progressed = false;
            if (ns < n_tiles) {
                const int b = ns & 1;
                if (tc_test(bar(kBarKFull + b), (uint32_t)((ns >> 1) & 1)) &&
                    (ns < 2 || tc_test(bar(kBarSFree + b), (uint32_t)(((ns - 2) >> 1) & 1)))) {
                    tc_fence_after();
                    const uint32_t k_base = smem_u32(sm.k[b]);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc_mma(tmem + 128u * b, sdesc(q_base + 256u * ks, 128, 2048),
                               sdesc(k_base + 256u * ks, 128, 2048), idesc_s, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // the low parts of the query
                        tc_mma(tmem + 128u * b, sdesc(ql_base + 256u * ks, 128, 2048),
                               sdesc(k_base + 256u * ks, 128, 2048), idesc_s, 1u);
                    tc_commit(bar(kBarSFull + b));
                    ++ns;
                    progressed = true;
                }
            }
            if (npv < ns && tc_test(bar(kBarPFull + (npv & 1)), (uint32_t)((npv >> 1) & 1)) &&
                tc_test(bar(kBarVFull + (npv & 1)), (uint32_t)((npv >> 1) & 1))) {
                tc_fence_after();
                const int b = npv & 1;
                const uint32_t v_base = smem_u32(sm.v[b]);
                // A = P from tensor memory (16 keys = 8 columns per MMA), B = the V tile
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(tmem + kTmemO, tmem + kTmemP + 64u * b + 8u * kk,
                              sdesc(v_base + 4096u * kk, 2048, 128), idesc_pv, (npv > 0 || kk > 0));
                tc_commit(bar(kBarPvFree + b));
                ++npv;
                progressed = true;
            }
            if (progressed) idle = 0;
            else if (++idle > kTcPollLimit || *abort_v) {
                if (!*abort_v) record_error(TQ_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
        }
        if (!ok) *abort_v = 1;
        tc_commit(bar(kBarDrain));   // arrives once everything issued above has completed
        tc_wait(bar(kBarDrain), 0);
    }
    // the other roles pass the two cluster barriers of the softmax warps' partial exchange
    if (p.split == 2 && warp >= kTcSoftmax / 32) {
        cluster_sync_all();
        cluster_sync_all();
    }
    // teardown: every MMA has completed (the softmax waited for the last P V, or all roles
    // gave up on a timeout); release the tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------------ head_dim 256
// Two 128-value blocks per head, each rotated and quantised on its own, each with its own
// norm.  One CTA per query block computes both output blocks:
//  - tensor memory holds the scores S [0,128) (block 0's 64 keys, then block 1's: S_b =
//    Q~_b C_b^T with N = 64, so each block is scaled by its own norm in fp32, as at head_dim
//    128), the output O [128,384) (256 coordinates) and the query's high fp16 parts
//    [384,512), the A operand of the high score MMAs;
//  - shared memory holds the query's low parts (64 KB, the A operand of the low score MMAs),
//    the K tile of 64 keys x 256 coordinates (double-buffered, one 16 KB tile per block), the
//    V tile of 64 keys x 256 coordinates (single) and P (double), the A operand of P V, which
//    is one N = 256 MMA per 16 keys.
// The key norms are kept for three tiles: the K producer may decode tile i + 2 once tile i's
// score MMAs are done, before the softmax has read tile i's norms.
constexpr int k2Keys = 64;   // keys per tile
constexpr uint32_t k2S = 0, k2O = 128, k2Qh = 384;

enum {
    k2BarQ = 0,        // queries written (256 arrivals)
    k2BarKFull = 1,    // [2] K tile (both blocks) and norms decoded (128 arrivals)
    k2BarKFree = 3,    // [2] the tile's score MMAs done: K buffer free (commit)
    k2BarSFull = 5,    // scores ready (commit)
    k2BarSFree = 6,    // scores and norms read (256 arrivals)
    k2BarVFull = 7,    // V tile decoded (128 arrivals)
    k2BarPFull = 8,    // [2] P written, O rescaled (256 arrivals)
    k2BarPvFree = 10,  // [2] the tile's P V done: V tile and P buffer free (commit)
    k2BarDrain = 12,   // every MMA of the CTA done (commit)
    k2BarCount = 13
};

struct TcSmem256 {
    alignas(1024) uint8_t ql[65536];       // Q~ low parts [row][coord 0..255], K-major
    alignas(1024) uint8_t k[2][2][16384];  // [buffer][block] K tile [key][coord], K-major
    alignas(1024) uint8_t v[32768];        // V tile [key][coord 0..255], MN-major
    alignas(1024) uint8_t p[2][16384];     // [buffer] P [row][key] fp16, K-major
    alignas(16) uint8_t raw_k[2][k2Keys * 64];   // staged K blocks (64-byte key windows)
    alignas(16) uint8_t raw_v[2][k2Keys * 64];   // staged V blocks
    // [tile mod 3][block][key] norms: the producer writes tile i + 2's norms once tile i's
    // score MMAs are done, possibly before the softmax has read tile i's
    float kn[3][2][k2Keys];
    float xch[2][2][kTcRows];
    uint8_t ok[4][k2Keys];                 // K block 0, K block 1, V block 0, V block 1
    alignas(8) uint64_t bar[k2BarCount];
    uint32_t tmem;
};

// Element (row, coord) of the 256-coordinate K-major query tile: 32 core matrices along K,
// so 8-row groups sit 4096 bytes apart.
__device__ __forceinline__ uint32_t canon256(int r, int c) {
    return (uint32_t)((r >> 3) * 4096 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}
// Element (row, key) of a 64-key K-major tile: 8 core matrices along K, so 8-row groups sit
// 1024 bytes apart.
__device__ __forceinline__ uint32_t canon64(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}
// Instruction descriptors, kind::f16 (fp32 accumulate, fp16 A and B, M = 128): the score MMA
// (both operands K-major, N = 64) and P V (B MN-major, N = 256).
constexpr uint32_t idesc_f16_n64() {
    return (1u << 4) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
}
constexpr uint32_t idesc_f16_pv256() {
    return (1u << 4) | (1u << 16) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
}

template <int TK, int TV>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc256_kernel(const TcParams p) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TcSmem256 &sm = *reinterpret_cast<TcSmem256 *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned qcta = blockIdx.x;   // longest first, as above
    const int g = (int)(qcta % (unsigned)p.n_kv_heads), G = p.group, Hq = p.n_q_heads;
    const int64_t j0 = (p.n_qblocks - 1 - (int64_t)(qcta / (unsigned)p.n_kv_heads)) * p.bq;
    const int64_t j_end = min64(p.n_q, j0 + p.bq);
    const int64_t n_keys = p.pos0 + j_end;
    const int64_t first_pos = p.pos0 + j0;
    const int n_tiles = (int)((n_keys + k2Keys - 1) / k2Keys);
    constexpr int D = 2 * kBlock;
    auto bar = [&](int i) { return smem_u32(&sm.bar[i]); };

    if (tid == 0) {
        abort_flag = 0;
        tc_bar_init(bar(k2BarQ), kTcSoftmax);
        tc_bar_init(bar(k2BarSFull), 1);
        tc_bar_init(bar(k2BarSFree), kTcSoftmax);
        tc_bar_init(bar(k2BarVFull), kTcGroup);
        for (int b = 0; b < 2; ++b) {
            tc_bar_init(bar(k2BarKFull + b), kTcGroup);
            tc_bar_init(bar(k2BarKFree + b), 1);
            tc_bar_init(bar(k2BarPFull + b), kTcSoftmax);
            tc_bar_init(bar(k2BarPvFree + b), 1);
        }
        tc_bar_init(bar(k2BarDrain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&sm.tmem)), "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;
    volatile int *abort_v = &abort_flag;

    if (warp < kTcSoftmax / 32) {
        // ================= softmax: thread (r, h) owns keys 32 h .. 32 h + 31 of every tile
        const int quad = warp & 3, h = warp >> 2;
        const int r = 32 * quad + lane, jl = r / G, hl = r - jl * G;
        const bool valid = jl < p.bq && j0 + jl < p.n_q;
        const int64_t qpos = valid ? p.pos0 + j0 + jl : INT64_MAX;
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint32_t pair_bar = 3u + (uint32_t)quad;
        // the query, block by block: coords 64 h .. 64 h + 63 of Q~_b = H (D q_b) * scale;
        // high fp16 parts into tensor memory (two K values per column), low parts into the
        // shared-memory tile
#pragma unroll 1
        for (int blk = 0; blk < 2; ++blk) {
            float x[64];
            if (valid) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.q + ((j0 + jl) * Hq + g * G + hl) * (int64_t)D + kBlock * blk);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 ua = src[c], ub = src[c + 8];
                    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = 8 * c + 2 * e;
                        const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&wa[e]));
                        const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&wb[e]));
                        float a0 = fa.x, a1 = fa.y, b0 = fb.x, b1 = fb.y;
                        if (p.kc.has_signs) {
                            a0 = __uint_as_float(__float_as_uint(a0) ^ sign_mask(p.kc, i0));
                            a1 = __uint_as_float(__float_as_uint(a1) ^ sign_mask(p.kc, i0 + 1));
                            b0 = __uint_as_float(__float_as_uint(b0) ^ sign_mask(p.kc, 64 + i0));
                            b1 = __uint_as_float(__float_as_uint(b1) ^ sign_mask(p.kc, 64 + i0 + 1));
                        }
                        x[i0] = h ? a0 - b0 : a0 + b0;
                        x[i0 + 1] = h ? a1 - b1 : a1 + b1;
                    }
                }
                fwht64(x);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) x[i] = 0.f;
            }
            // 16 columns (32 coords) at a time keeps the live registers down
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t w[16], wl[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    split_half2(x[32 * c + 2 * e] * p.score_scale, x[32 * c + 2 * e + 1] * p.score_scale,
                                w[e], wl[e]);
                tc_st16(tmem + lane_base + k2Qh + 64u * blk + 32u * h + 16u * c, w);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(sm.ql + canon256(r, kBlock * blk + 64 * h + 32 * c + 8 * q4)) =
                        make_uint4(wl[4 * q4], wl[4 * q4 + 1], wl[4 * q4 + 2], wl[4 * q4 + 3]);
            }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        tc_arrive(bar(k2BarQ));

        float m_run = -INFINITY, l_run = 0.f;
        for (int i = 0; i < n_tiles; ++i) {
            const int b = i & 1;
            if (!*abort_v && !tc_wait(bar(k2BarSFull), (uint32_t)(i & 1))) *abort_v = 1;
            tc_fence_after();
            float s[32], s1[32];
            tc_ld32(tmem + lane_base + k2S + 32u * h, s);
            tc_ld32(tmem + lane_base + k2S + 64u + 32u * h, s1);
            const float *n0 = sm.kn[i % 3][0] + 32 * h, *n1 = sm.kn[i % 3][1] + 32 * h;
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = m_run;
            if ((int64_t)i * k2Keys + (k2Keys - 1) <= first_pos) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = s[j] * n0[j] + s1[j] * n1[j];
                    mx8[j & 7] = fmaxf(mx8[j & 7], s[j]);
                }
            } else {
                const int64_t t0 = (int64_t)i * k2Keys + 32 * h;
                const int lim = (int)max64(-1, min64(qpos - t0, 32));   // keys j > lim are masked
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = j > lim ? -INFINITY : s[j] * n0[j] + s1[j] * n1[j];
                    mx8[j & 7] = fmaxf(mx8[j & 7], s[j]);
                }
            }
            // the score buffer and this tile's norms are free
            tc_fence_before();
            tc_arrive(bar(k2BarSFree));
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            sm.xch[b][h][r] = mx;
            named_sync(pair_bar, 64);
            mx = fmaxf(mx, sm.xch[b][h ^ 1][r]);
            float alpha = 1.f;
            if (m_run == -INFINITY || mx > m_run + 8.f) {
                alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
                m_run = mx;
            }
            // P buffer b is free once tile i - 2's P V is done
            if (i >= 2 && !*abort_v && !tc_wait(bar(k2BarPvFree + b), (uint32_t)(((i - 2) >> 1) & 1)))
                *abort_v = 1;
            tc_fence_after();
            float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float mref = m_run == -INFINITY ? 0.f : m_run;
#pragma unroll
            for (int c = 0; c < 4; ++c) {   // keys 32 h + 8 c .. + 7 of row r
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 8 * c + 2 * e;
                    const float p0 = ex2(s[j] - mref), p1 = ex2(s[j + 1] - mref);
                    ps8[j & 7] += p0;
                    ps8[(j + 1) & 7] += p1;
                    w[e] = pack_half2(p0, p1);
                }
                *reinterpret_cast<uint4 *>(sm.p[b] + canon64(r, 32 * h + 8 * c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            const float psum = ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
            l_run = l_run * alpha + psum;
            if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // the running output must hold every P V up to tile i - 1 before it is scaled;
                // this half scales output columns 128 h .. 128 h + 127
                if (!*abort_v && !tc_wait(bar(k2BarPvFree + ((i - 1) & 1)), (uint32_t)(((i - 1) >> 1) & 1)))
                    *abort_v = 1;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float t[32];
                    tc_ld32(tmem + lane_base + k2O + 128u * h + 32u * c, t);
#pragma unroll
                    for (int e = 0; e < 32; ++e) t[e] *= alpha;
                    tc_st32(tmem + lane_base + k2O + 128u * h + 32u * c, t);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // P for the MMA
            tc_fence_before();
            tc_arrive(bar(k2BarPFull + b));
        }
        // ---- epilogue: O / l, block by block: inverse rotation, V signs, store
        const bool done = n_tiles > 0 && !*abort_v &&
                          tc_wait(bar(k2BarPvFree + ((n_tiles - 1) & 1)), (uint32_t)(((n_tiles - 1) >> 1) & 1));
        tc_fence_after();
        sm.xch[n_tiles & 1][h][r] = l_run;
        named_sync(pair_bar, 64);
        const float l_row = l_run + sm.xch[n_tiles & 1][h ^ 1][r];
        const float inv = l_row > 0.f ? p.out_scale / l_row : 0.f;
        // the query's low-part tile is idle once every MMA has completed
        float *xo = reinterpret_cast<float *>(sm.ql);
        auto xo_at = [&](int row, int c4) { return xo + row * 128 + (((c4 ^ row) & 31) << 2); };
#pragma unroll 1
        for (int blk = 0; blk < 2; ++blk) {
            float o[64];
            if (n_tiles > 0) {
                tc_ld64(tmem + lane_base + k2O + 128u * blk + 64u * h, o);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) o[e] = 0.f;
            }
            fwht64(o);
            if (blk > 0) named_sync(pair_bar, 64);   // the partner has read the last block's halves
#pragma unroll
            for (int c = 0; c < 16; ++c)
                *reinterpret_cast<float4 *>(xo_at(r, 16 * h + c)) =
                    make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            named_sync(pair_bar, 64);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float4 u = *reinterpret_cast<const float4 *>(xo_at(r, 16 * (h ^ 1) + c));
                const float pv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) o[4 * c + e] = h ? pv[e] - o[4 * c + e] : o[4 * c + e] + pv[e];
            }
            if (valid && done) {
                float4 *dst = reinterpret_cast<float4 *>(p.out + ((j0 + jl) * Hq + g * G + hl) * (int64_t)D +
                                                         kBlock * blk + 64 * h);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float v4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v4[e] = __uint_as_float(__float_as_uint(o[4 * c + e] * inv) ^ sign_mask(p.vc, 64 * h + 4 * c + e));
                    dst[c] = make_float4(v4[0], v4[1], v4[2], v4[3]);
                }
            }
        }
    } else if (warp < kTcMmaWarp) {
        // ================= producers: thread (block, key) of the K group (warps 8-11) and of
        // the V group (warps 12-15)
        const int pt = (tid - kTcSoftmax) & (kTcGroup - 1);
        const int key = pt & (k2Keys - 1), blk = pt >> 6;
        if (tid - kTcSoftmax < kTcGroup) {
            // K: double-buffered tiles, one 16 KB tile per block
            const HalfTables tab = make_tables<TK>();
            if (n_tiles > 0)
                tc_stage<TK>(p.kc, p.seq, p.chunked_k, sm.raw_k[blk], sm.ok[blk], 2 * g + blk, 0, n_keys, key);
            cp_async_commit();
            for (int i = 0; i < n_tiles; ++i) {
                const int b = i & 1;
                cp_async_wait<0>();
                uint32_t nb[13];
                tc_window<TK>(sm.raw_k[blk], 2 * g + blk, key, nb);
                const bool present = sm.ok[blk][key] != 0;
                if (i + 1 < n_tiles)
                    tc_stage<TK>(p.kc, p.seq, p.chunked_k, sm.raw_k[blk], sm.ok[blk], 2 * g + blk,
                                 (int64_t)(i + 1) * k2Keys, n_keys, key);
                cp_async_commit();
                if (i >= 2 && !*abort_v && !tc_wait(bar(k2BarKFree + b), (uint32_t)(((i - 2) >> 1) & 1)))
                    *abort_v = 1;
                tc_decode<TK, false>(nb, present, tab, sm.k[b][blk], sm.kn[i % 3][blk], key);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_arrive(bar(k2BarKFull + b));
            }
            cp_async_wait<0>();
        } else {
            // V: one 256-coordinate tile, rewritten once the previous tile's P V is done
            const HalfTables tab = make_tables<TV>();
            if (n_tiles > 0)
                tc_stage<TV>(p.vc, p.seq, p.chunked_v, sm.raw_v[blk], sm.ok[2 + blk], 2 * g + blk, 0, n_keys, key);
            cp_async_commit();
            for (int i = 0; i < n_tiles; ++i) {
                cp_async_wait<0>();
                uint32_t nb[13];
                tc_window<TV>(sm.raw_v[blk], 2 * g + blk, key, nb);
                const bool present = sm.ok[2 + blk][key] != 0;
                if (i + 1 < n_tiles)
                    tc_stage<TV>(p.vc, p.seq, p.chunked_v, sm.raw_v[blk], sm.ok[2 + blk], 2 * g + blk,
                                 (int64_t)(i + 1) * k2Keys, n_keys, key);
                cp_async_commit();
                if (i >= 1 && !*abort_v &&
                    !tc_wait(bar(k2BarPvFree + ((i - 1) & 1)), (uint32_t)(((i - 1) >> 1) & 1)))
                    *abort_v = 1;
                tc_decode<TV, true, D>(nb, present, tab, sm.v, nullptr, key, kBlock * blk);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                tc_arrive(bar(k2BarVFull));
            }
            cp_async_wait<0>();
        }
    } else if (lane == 0) {
        // ================= MMA issue (one thread)
        constexpr uint32_t idesc_s = idesc_f16_n64(), idesc_pv = idesc_f16_pv256();
        const uint32_t ql_base = smem_u32(sm.ql), v_base = smem_u32(sm.v);
        bool ok = tc_wait(bar(k2BarQ), 0);
        int ns = 0, npv = 0;
        uint32_t idle = 0;
        while (ok && npv < n_tiles) {
            bool progressed = false;
            // S(ns) overwrites the single score buffer: the softmax has read S(ns - 1)
            if (ns < n_tiles && tc_test(bar(k2BarKFull + (ns & 1)), (uint32_t)((ns >> 1) & 1)) &&
                (ns == 0 || tc_test(bar(k2BarSFree), (uint32_t)((ns - 1) & 1)))) {
                tc_fence_after();
                // S_b = Q~_b C_b^T: the high parts from tensor memory (16 coords = 8 columns per
                // MMA), the low parts from shared memory; B = the block's K tile
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const uint32_t k_base = smem_u32(sm.k[ns & 1][blk]);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma_ts(tmem + k2S + 64u * blk, tmem + k2Qh + 64u * blk + 8u * kk,
                                  sdesc(k_base + 256u * kk, 128, 2048), idesc_s, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc_mma(tmem + k2S + 64u * blk, sdesc(ql_base + 2048u * blk + 256u * kk, 128, 4096),
                               sdesc(k_base + 256u * kk, 128, 2048), idesc_s, 1u);
                }
                tc_commit(bar(k2BarSFull));
                tc_commit(bar(k2BarKFree + (ns & 1)));
                ++ns;
                progressed = true;
            }
            if (npv < ns && tc_test(bar(k2BarPFull + (npv & 1)), (uint32_t)((npv >> 1) & 1)) &&
                tc_test(bar(k2BarVFull), (uint32_t)(npv & 1))) {
                tc_fence_after();
                const int b = npv & 1;
                const uint32_t p_base = smem_u32(sm.p[b]);
                // A = P from shared memory (16 keys per MMA), B = the V tile, N = 256
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem + k2O, sdesc(p_base + 256u * kk, 128, 1024),
                           sdesc(v_base + 8192u * kk, 4096, 128), idesc_pv, (npv > 0 || kk > 0));
                tc_commit(bar(k2BarPvFree + b));
                ++npv;
                progressed = true;
            }
            if (progressed) idle = 0;
            else if (++idle > kTcPollLimit || *abort_v) {
                if (!*abort_v) record_error(TQ_ERR_DEVICE_TIMEOUT);
                ok = false;
            }
        }
        if (!ok) *abort_v = 1;
        tc_commit(bar(k2BarDrain));
        tc_wait(bar(k2BarDrain), 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

template <int TK, int TV>
tq_status launch_tc256_t(const TcParams &p, unsigned n_ctas, cudaStream_t stream) {
    static_assert(sizeof(TcSmem256) + 1024 <= 227 * 1024, "one CTA per SM");
    const size_t smem = sizeof(TcSmem256) + 1024;
    const tq_status st = kernel_setup(reinterpret_cast<const void *>(prefill_tc256_kernel<TK, TV>),
                                      (int)smem, kTcThreads, nullptr);
    if (st != TQ_OK) return st;
    PdlConfig lc(dim3(n_ctas), dim3(kTcThreads), smem, stream);
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, prefill_tc256_kernel<TK, TV>, p));
}

template <int TK, int TV>
tq_status launch_tc_t(const TcParams &p, unsigned n_ctas, cudaStream_t stream) {
    const size_t smem = sizeof(TcSmem) + 1024;   // room to align the tiles to 1024 bytes
    const tq_status st = kernel_setup(reinterpret_cast<const void *>(prefill_tc_kernel<TK, TV>),
                                      (int)smem, kTcThreads, nullptr);
    if (st != TQ_OK) return st;
    PdlConfig lc(dim3(n_ctas * (unsigned)p.split), dim3(kTcThreads), smem, stream);
    if (p.split == 2) {   // the two CTAs of a query block form a cluster
        lc.attrs[1].id = cudaLaunchAttributeClusterDimension;
        lc.attrs[1].val.clusterDim.x = 2;
        lc.attrs[1].val.clusterDim.y = 1;
        lc.attrs[1].val.clusterDim.z = 1;
        lc.cfg.numAttrs = 2;
    }
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, prefill_tc_kernel<TK, TV>, p));
}

}  // namespace

bool prefill_supported(const tq_cache &k, const tq_cache &v, int n_q_heads) {
    if (k.head_dim != v.head_dim || (k.head_dim != kBlock && k.head_dim != 2 * kBlock)) return false;
    return n_q_heads % k.n_kv_heads == 0 && n_q_heads / k.n_kv_heads <= kTcRows;
}

tq_status launch_prefill(const tq_cache &k, const tq_cache &v, const void *q, int32_t seq_id,
                         int64_t pos0, int64_t n_q, int n_q_heads, float scale, float *out,
                         cudaStream_t stream) {
    if (!prefill_supported(k, v, n_q_heads)) return TQ_ERR_UNSUPPORTED;
    if (n_q == 0) return TQ_OK;
    TcParams p;
    p.kc = make_view(k);
    p.vc = make_view(v);
    p.q = static_cast<const __half *>(q);
    p.out = out;
    p.pos0 = pos0;
    p.n_q = n_q;
    p.seq = seq_id;
    p.n_q_heads = n_q_heads;
    p.group = n_q_heads / k.n_kv_heads;
    p.bq = kTcRows / p.group;
    p.chunked_k = p.kc.row_bytes % 16 == 0;
    p.chunked_v = p.vc.row_bytes % 16 == 0;
    // the fp16 centroid tables are scaled by h_scale (Codebook); the query scale divides the
    // K table's out, the output scale the V table's
    p.score_scale = scale * kTcLog2e * kInvSqrt128 / centroid_h_scale(k.type);
    p.out_scale = kInvSqrt128 / centroid_h_scale(v.type);
    p.n_kv_heads = k.n_kv_heads;
    p.n_qblocks = (n_q + p.bq - 1) / p.bq;
    const int64_t n_ctas = p.n_qblocks * k.n_kv_heads;
    if (n_ctas > 0x3fffffff) return TQ_ERR_UNSUPPORTED;
    const unsigned nc = (unsigned)n_ctas;
    if (k.head_dim == 2 * kBlock) {   // one CTA per query block, no key split
        p.split = 1;
        if (k.type == TQ_TURBO3 && v.type == TQ_TURBO3) return launch_tc256_t<3, 3>(p, nc, stream);
        if (k.type == TQ_TURBO2 && v.type == TQ_TURBO2) return launch_tc256_t<2, 2>(p, nc, stream);
        if (k.type == TQ_TURBO3 && v.type == TQ_TURBO2) return launch_tc256_t<3, 2>(p, nc, stream);
        return launch_tc256_t<2, 3>(p, nc, stream);
    }
    // Split each query block's key tiles over a cluster of two CTAs when that fills the last
    // wave of one-CTA-per-SM launches markedly better (the two CTAs both rotate the queries,
    // so a split costs a little): e.g. the 512 CTAs of a 2,048-token chunk of a Llama-shape
    // prompt run 3.37 waves on 152 SMs (84 % of the last wave's SMs busy over the launch), and
    // 1,024 half-length CTAs run 6.74 (96 %).
    {
        const double sms = (double)device_sm_count();
        const double w1 = (double)n_ctas / sms, w2 = 2.0 * w1;
        const double e1 = w1 / std::ceil(w1), e2 = w2 / std::ceil(w2);
        const int64_t max_tiles = (pos0 + n_q + kTcKeys - 1) / kTcKeys;
        p.split = (max_tiles >= 4 && e2 > 1.08 * e1) ? 2 : 1;
    }
    if (k.type == TQ_TURBO3 && v.type == TQ_TURBO3) return launch_tc_t<3, 3>(p, nc, stream);
    if (k.type == TQ_TURBO2 && v.type == TQ_TURBO2) return launch_tc_t<2, 2>(p, nc, stream);
    if (k.type == TQ_TURBO3 && v.type == TQ_TURBO2) return launch_tc_t<3, 2>(p, nc, stream);
    return launch_tc_t<2, 3>(p, nc, stream);
}

}  // namespace tq
