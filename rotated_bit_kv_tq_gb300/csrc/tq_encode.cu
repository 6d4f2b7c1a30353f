// tq_encode.cu -- fused encode: norm -> FWHT -> Lloyd-Max quantise -> bit-pack.
//
// "llama.cpp に TurboQuant を実装": the rotation is a fast Walsh-Hadamard transform, adds
// and subtracts only ("What TurboQuant does differently"), cheap enough to run inside
// the cache-write path; every 128 values become one fp16 norm plus 3- or 2-bit codes
// ("How small does it get").
//
// GB300 mapping.  One thread owns one 128-value block, so the whole FWHT, the norm tree
// and the quantiser run in registers with no cross-lane traffic; packed f32x2 adds and
// multiplies halve the issue slots of the FP32 work.  A persistent CTA of 128 threads
// walks over tiles of whole token rows (<= 128 blocks, 32 KB of fp16).  Each tile is
// prefetched with cp.async (16-byte, coalesced) into a double-buffered shared-memory
// tile whose 16-byte chunks are XOR-swizzled per block, so that the per-thread 16-byte
// reads of "its" block are bank-conflict free.  Packed blocks are staged in shared
// memory and written out as whole rows with 16-byte stores.
//
// Bit-exactness with the oracle: the same fixed operation order (pairwise norm tree
// i + len/2, butterfly stages h = 1..64, one IEEE sqrt and one IEEE divide, one multiply
// per value), every operation rounded separately (no FMA contraction: the f32x2
// instructions and __f*_rn intrinsics are never fused; the one explicit fused multiply-add,
// on the first level of the norm tree, squares an fp16 value, whose square is exact).
#include "tq_internal.cuh"
#include "tq_simd.cuh"
#include "tq_encode_warp.cuh"

namespace tq {
namespace {

constexpr int kThreads = 128;            // blocks per tile (one per thread)
constexpr int kInBytes = kThreads * 256;  // fp16 input tile

struct EncodeParams {
    CacheView dst;
    const __half *src;
    int64_t stride;            // elements between token rows of src
    const int32_t *seq_ids;    // or nullptr
    const int32_t *positions;  // or nullptr
    const int32_t *lens;       // decode-step append: token t -> sequence t, position lens[t] - 1
    int64_t pos0;
    int64_t n_tokens;
    int64_t n_tiles;
    int32_t seq_id;
    int32_t bpr;               // blocks per token row
    int32_t src_dense;         // stride == bpr * 128: the source rows form one byte run
    uint32_t bpr_magic;        // div_magic(bpr)
    int32_t rows_per_tile;
    int32_t row_bytes;
    uint32_t cpr_magic;        // div_magic(row_bytes / 16)  (16-byte path)
    uint32_t hpr_magic;        // div_magic(row_bytes / 2)   (2-byte path)
};

template <int TYPE>
struct EncodeSmem {
    alignas(128) uint8_t in[2][kInBytes];
    alignas(16) uint8_t out[kThreads * block_bytes(TYPE)];
    uint8_t *rowdst[kThreads];
};

// Issue the cp.async copies of one tile into `buf` (16-byte chunks, swizzled).
__device__ __forceinline__ void load_tile(const EncodeParams &p, int64_t tile, uint8_t *buf) {
    const int64_t row0 = tile * p.rows_per_tile;
    const int rows = (int)min64(p.rows_per_tile, p.n_tokens - row0);
    const uint32_t sbase = smem_u32(buf);
    if (p.src_dense) {
        // Token rows back to back: the tile is one byte run and chunk c = threadIdx.x + 128 i
        // of it belongs to block f = threadIdx.x / 16 + 8 i at the same 16-byte slot
        // j = threadIdx.x % 16, with the same swizzle f % 8, so every copy is a fixed offset.
        const int f0 = threadIdx.x >> 4, j = threadIdx.x & 15;
        const int nblk = rows * p.bpr;
        const uint8_t *g = reinterpret_cast<const uint8_t *>(p.src + row0 * p.stride) + threadIdx.x * 16;
        const uint32_t s = sbase + f0 * 256 + ((j ^ (f0 & 7)) << 4);
#pragma unroll
        for (int i = 0; i < kThreads / 8; ++i)
            if (f0 + 8 * i < nblk) cp_async16(s + i * 2048, g + i * 2048);
        return;
    }
    const int chunks = rows * p.bpr * 16;
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
        const int f = c >> 4, j = c & 15;
        const int r = (int)fast_div((uint32_t)f, p.bpr_magic);
        const int fb = f - r * p.bpr;
        const __half *g = p.src + (row0 + r) * p.stride + fb * kBlock + j * 8;
        cp_async16(sbase + f * 256 + ((j ^ (f & 7)) << 4), g);
    }
}

// Append the sign bit of `v` to a collection word, two positions per value:
// w = (w << 2) | (bits(v) >> 30).  Every float fed here has |v| < 2, so bit 30 (the top
// exponent bit) is 0 and each value lands as (sign, 0) at bits (2j+1, 2j).
__device__ __forceinline__ uint32_t collect2(uint32_t w, float v) {
    return __funnelshift_l(__float_as_uint(v), w, 2);
}

template <int TYPE>
__device__ __forceinline__ void encode_one(const uint8_t *blk_in, int f, uint8_t *out,
                                           const CacheView &cv) {
    const Codebook &cb = c_codebook[cb_index(TYPE)];
    // ---- 1. load and convert once
    float x[kBlock];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(blk_in + ((j ^ (f & 7)) << 4));
        const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 t = __half22float2(h2[e]);
            x[8 * j + 2 * e] = t.x;
            x[8 * j + 2 * e + 1] = t.y;
        }
    }
    // rotation-sign variant: the rotation is W D, so flagged coordinates are negated first
    if (cv.has_signs) {
#pragma unroll
        for (int i = 0; i < kBlock; ++i) x[i] = __uint_as_float(__float_as_uint(x[i]) ^ sign_mask(cv, i));
    }
    // ---- 2. norm: pairwise tree, element i pairs with i + len/2 at every level
    // (x comes from fp16: 11 significant bits, so x*x is exact in binary32 and the fused
    // x_i * x_i + fl(x_{i+64}^2) rounds once, like fl(fl(x_i^2) + fl(x_{i+64}^2)))
    float s1[64];
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
        const float2 b = mul2(make_float2(x[i + 64], x[i + 65]), make_float2(x[i + 64], x[i + 65]));
        const float2 r = fma2(make_float2(x[i], x[i + 1]), make_float2(x[i], x[i + 1]), b);
        s1[i] = r.x;
        s1[i + 1] = r.y;
    }
#pragma unroll
    for (int len = 64; len > 2; len >>= 1) {
#pragma unroll
        for (int i = 0; i < len / 2; i += 2) {
            const float2 r = add2(make_float2(s1[i], s1[i + 1]),
                                  make_float2(s1[i + len / 2], s1[i + len / 2 + 1]));
            s1[i] = r.x;
            s1[i + 1] = r.y;
        }
    }
    const float n = __fsqrt_rn(__fadd_rn(s1[0], s1[1]));
    const uint16_t norm16 = __half_as_ushort(__float2half_rn(fminf(n, 65504.0f)));
    const float k = n > 0.0f ? __fdiv_rn(kInvSqrt128, n) : 0.0f;

    // ---- 3. FWHT, stages h = 1, 2, ..., 64 in that order
#pragma unroll
    for (int i = 0; i < kBlock; i += 2) {
        const float a = x[i], b = x[i + 1];
        x[i] = __fadd_rn(a, b);
        x[i + 1] = __fsub_rn(a, b);
    }
#pragma unroll
    for (int h = 2; h < kBlock; h <<= 1) {
#pragma unroll
        for (int i = 0; i < kBlock; i += 2) {
            if (i & h) continue;
            const float2 a = make_float2(x[i], x[i + 1]);
            const float2 b = make_float2(x[i + h], x[i + h + 1]);
            const float2 s = add2(a, b), d = sub2(a, b);
            x[i] = s.x;
            x[i + 1] = s.y;
            x[i + h] = d.x;
            x[i + h + 1] = d.y;
        }
    }
    // ---- 4-5. scale to the unit sphere, y = fl(z k) in pairs, and take the
    // sign-magnitude Lloyd-Max index, bit-parallel.  "|y| > t" is the sign bit of
    // fl(t - |y|) (exact zero only when |y| == t, which is not "greater").  The subtraction
    // is a scalar IEEE operation on the stored y: fed straight from the paired product, it
    // was evaluated as one fused t - |z| k at full size, which counts a tie whose exact
    // product lies just above t as "greater".  Low-plane word w holds value
    // i = 16w + 8r + k at bits 4k+2r (code bit 0) and 4k+2r+1 (code bit 1): collecting
    // values in the order j = 2k + r, last first, puts value j's predicate at bit 2j+1.
    const float2 kk = make_float2(k, k);
#pragma unroll
    for (int i = 0; i < kBlock; i += 2) {
        const float2 y2 = mul2(make_float2(x[i], x[i + 1]), kk);
        x[i] = y2.x;
        x[i + 1] = y2.y;
    }
    uint32_t W[8], SP[8];
    const float t_lo = TYPE == TQ_TURBO3 ? cb.threshold[4] : cb.threshold[2];
    const float t_mid = TYPE == TQ_TURBO3 ? cb.threshold[5] : 0.0f;
    const float t_hi = TYPE == TQ_TURBO3 ? cb.threshold[6] : 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t ps = 0, p4 = 0, p5 = 0, p6 = 0;
#pragma unroll
        for (int j = 15; j >= 0; --j) {
            const float y = x[16 * w + 8 * (j & 1) + (j >> 1)];
            const float a = fabsf(y);
            ps = collect2(ps, y);
            p4 = collect2(p4, __fsub_rn(t_lo, a));
            if (TYPE == TQ_TURBO3) {
                p5 = collect2(p5, __fsub_rn(t_mid, a));
                p6 = collect2(p6, __fsub_rn(t_hi, a));
            }
        }
        if (TYPE == TQ_TURBO3) {
            // m = (|y|>t4) + (|y|>t5) + (|y|>t6): bit1 = |y|>t5, bit0 = |y|>(bit1 ? t6 : t4);
            // code & 3 = m ^ 3s  -> fields (bit1 ^ s, bit0 ^ s)
            const uint32_t b0 = (p5 & p6) | (~p5 & p4);
            W[w] = (p5 ^ ps) | ((b0 ^ ps) >> 1);
        } else {
            // code = s ? 1 - m : 2 + m  -> fields (!s, m ^ s)
            W[w] = (~ps & 0xAAAAAAAAu) | ((p4 ^ ps) >> 1);
        }
        SP[w] = ps;
    }
    // high plane (turbo3): code bit 2 = !s.  Word u gathers values 32u + 16w' + 8r + k at
    // bit 4k + 2w' + r; the sign of value (w = 2u + w', r, k) sits at bit 4k + 2r + 1.
    uint32_t V[4];
    if (TYPE == TQ_TURBO3) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint32_t a = SP[2 * u], b = SP[2 * u + 1];
            const uint32_t sv = ((a & 0x22222222u) >> 1) | ((a & 0x88888888u) >> 2) |
                                ((b & 0x22222222u) << 1) | (b & 0x88888888u);
            V[u] = ~sv;
        }
    }
    // norm-correction variant: store |x| / |c|, |c| over the same pairwise tree as the norm
    uint16_t norm_out = norm16;
    if (cv.norm_correction) {
        float c2[64];
#pragma unroll
        for (int i = 0; i < 64; ++i)
            c2[i] = __fadd_rn(code_sq<TYPE>(cb, x[i]), code_sq<TYPE>(cb, x[i + 64]));
#pragma unroll
        for (int len = 64; len > 1; len >>= 1)
#pragma unroll
            for (int i = 0; i < len / 2; ++i) c2[i] = __fadd_rn(c2[i], c2[i + len / 2]);
        const float r = __fdiv_rn(n, __fsqrt_rn(c2[0]));
        norm_out = __half_as_ushort(__float2half_rn(fminf(r, 65504.0f)));
    }
    // ---- 6. stage the packed block (2-byte aligned in shared memory)
    uint16_t *o = reinterpret_cast<uint16_t *>(out);
    o[0] = norm_out;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        o[1 + 2 * w] = (uint16_t)(W[w] & 0xffffu);
        o[2 + 2 * w] = (uint16_t)(W[w] >> 16);
    }
    if (TYPE == TQ_TURBO3) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            o[17 + 2 * u] = (uint16_t)(V[u] & 0xffffu);
            o[18 + 2 * u] = (uint16_t)(V[u] >> 16);
        }
    }
}

// blockIdx.y selects the cache: one launch can encode the K and the V rows of a step.
template <int TYPE>
__global__ void __launch_bounds__(kThreads, 3) encode_kernel(const EncodeParams p0,
                                                             const EncodeParams p1) {
    const EncodeParams &p = blockIdx.y ? p1 : p0;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EncodeSmem<TYPE> &sm = *reinterpret_cast<EncodeSmem<TYPE> *>(smem_raw);
    constexpr int B = block_bytes(TYPE);
    pdl_wait();
    pdl_launch_dependents();

    int64_t tile = blockIdx.x;
    if (tile < p.n_tiles) load_tile(p, tile, sm.in[0]);
    cp_async_commit();
    for (int it = 0; tile < p.n_tiles; ++it, tile += gridDim.x) {
        const int64_t next = tile + gridDim.x;
        if (next < p.n_tiles) load_tile(p, next, sm.in[(it + 1) & 1]);
        cp_async_commit();

        const int64_t row0 = tile * p.rows_per_tile;
        const int rows = (int)min64(p.rows_per_tile, p.n_tokens - row0);
        // The tile's destination rows form one byte run when every row is valid and lies R
        // bytes after the one before; each row thread checks its row against the first.
        bool in_run = true;
        if (threadIdx.x < rows) {
            const int64_t t = row0 + threadIdx.x;
            const int64_t seq = p.seq_ids ? (int64_t)p.seq_ids[t] : (int64_t)p.seq_id;
            const int64_t pos = p.positions ? (int64_t)p.positions[t] : p.pos0 + t;
            uint8_t *d = row_ptr(p.dst, seq, pos);
            sm.rowdst[threadIdx.x] = d;
            if (threadIdx.x > 0) {
                const int64_t seq0 = p.seq_ids ? (int64_t)p.seq_ids[row0] : (int64_t)p.seq_id;
                const int64_t pos0 = p.positions ? (int64_t)p.positions[row0] : p.pos0 + row0;
                const uint8_t *d0 = row_ptr(p.dst, seq0, pos0);
                in_run = d0 && d == d0 + (int64_t)threadIdx.x * p.row_bytes;
            } else {
                in_run = d != nullptr;
            }
        }
        cp_async_wait<1>();
        const bool run = __syncthreads_and(in_run) && (p.row_bytes & 15) == 0;

        const int nblk = rows * p.bpr;
        const int f = threadIdx.x;
        if (f < nblk) encode_one<TYPE>(sm.in[it & 1] + f * 256, f, sm.out + f * B, p.dst);
        __syncthreads();

        // ---- write whole rows out
        const int R = p.row_bytes;
        if (run) {
            uint4 *d = reinterpret_cast<uint4 *>(sm.rowdst[0]);
            const uint4 *o = reinterpret_cast<const uint4 *>(sm.out);
            for (int c = threadIdx.x; c < rows * (R >> 4); c += kThreads) d[c] = o[c];
        } else if ((R & 15) == 0) {
            const int cpr = R >> 4;
            for (int c = threadIdx.x; c < rows * cpr; c += kThreads) {
                const int r = (int)fast_div((uint32_t)c, p.cpr_magic);
                const int cc = c - r * cpr;
                uint8_t *d = sm.rowdst[r];
                if (d) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sm.out + r * R + cc * 16);
                    *reinterpret_cast<uint4 *>(d + cc * 16) = v;
                }
            }
        } else {
            const int hpr = R >> 1;
            for (int c = threadIdx.x; c < rows * hpr; c += kThreads) {
                const int r = (int)fast_div((uint32_t)c, p.hpr_magic);
                const int cc = c - r * hpr;
                uint8_t *d = sm.rowdst[r];
                if (d)
                    reinterpret_cast<uint16_t *>(d)[cc] =
                        reinterpret_cast<const uint16_t *>(sm.out + r * R)[cc];
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

template <int TYPE>
tq_status launch_encode_t(const EncodeParams &p0, const EncodeParams &p1, int n_caches,
                          cudaStream_t stream) {
    const size_t smem = sizeof(EncodeSmem<TYPE>);
    int per_sm = 0;
    const tq_status st = kernel_setup(reinterpret_cast<const void *>(encode_kernel<TYPE>),
                                      (int)smem, kThreads, &per_sm);
    if (st != TQ_OK) return st;
    const int64_t slots = max64(1, (int64_t)device_sm_count() * per_sm / n_caches);
    const int64_t grid = min64(max64(p0.n_tiles, p1.n_tiles), slots);
    PdlConfig lc(dim3((unsigned)grid, (unsigned)n_caches), dim3(kThreads), smem, stream);
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, encode_kernel<TYPE>, p0, p1));
}

// ------------------------------------------------------------------ small appends
// A decode step appends one token (or one per sequence): a few hundred blocks at most,
// too few to fill the GPU with one block per thread.  Here a warp encodes one block, four
// values per lane (tq_encode_warp.cuh, in the operation order of encode_one, so the codes
// and norms are the same bits), and the latency of a block is that of ~200 instructions.
constexpr int kWarpPathWarps = 8;               // warps (blocks) per CTA
constexpr int64_t kWarpPathMaxBlocks = 4096;    // larger calls use encode_kernel

template <int TYPE>
__global__ void __launch_bounds__(32 * kWarpPathWarps) encode_warp_kernel(const EncodeParams p0,
                                                                          const EncodeParams p1) {
    pdl_wait();
    pdl_launch_dependents();
    const EncodeParams &p = blockIdx.y ? p1 : p0;
    constexpr int B = block_bytes(TYPE);
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarpPathWarps + (threadIdx.x >> 5);
    if (gw >= p.n_tokens * p.bpr) return;   // whole warp
    const int64_t t = gw / p.bpr;
    const int jb = (int)(gw - t * p.bpr);
    const WarpBlock wb = warp_encode_block<TYPE>(p.src + t * p.stride + jb * kBlock, p.dst, lane);
    const int64_t seq = p.seq_ids ? (int64_t)p.seq_ids[t] : p.lens ? t : (int64_t)p.seq_id;
    const int64_t pos = p.lens ? (int64_t)p.lens[t] - 1 : p.positions ? (int64_t)p.positions[t] : p.pos0 + t;
    if (p.lens && pos < 0) return;   // an empty sequence appends nothing
    uint8_t *row = nullptr;
    if (lane == 0) row = row_ptr(p.dst, seq, pos);   // records an out-of-range row once
    row = reinterpret_cast<uint8_t *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row), 0));
    if (!row) return;
    warp_store_block<TYPE>(row + (int64_t)jb * B, wb, lane);
}

template <int TYPE>
tq_status launch_encode_warp_t(const EncodeParams &p0, const EncodeParams &p1, int n_caches,
                               cudaStream_t stream) {
    const int64_t blocks = max64(p0.n_tokens * p0.bpr, p1.n_tokens * p1.bpr);
    const int64_t grid = (blocks + kWarpPathWarps - 1) / kWarpPathWarps;
    PdlConfig lc(dim3((unsigned)grid, (unsigned)n_caches), dim3(32 * kWarpPathWarps), 0, stream);
    return check_cuda(cudaLaunchKernelEx(&lc.cfg, encode_warp_kernel<TYPE>, p0, p1));
}

// One launch for one or two caches of the same type: small calls take the warp path.
template <int TYPE>
tq_status launch_encode_any(const EncodeParams &p0, const EncodeParams &p1, int n_caches,
                            cudaStream_t stream) {
    const int64_t blocks = max64(p0.n_tokens * p0.bpr, p1.n_tokens * p1.bpr);
    return blocks <= kWarpPathMaxBlocks ? launch_encode_warp_t<TYPE>(p0, p1, n_caches, stream)
                                        : launch_encode_t<TYPE>(p0, p1, n_caches, stream);
}

EncodeParams make_params(const tq_cache &dst, const void *src, int64_t n_tokens, int64_t stride,
                         const int32_t *seq_ids, const int32_t *positions, int32_t seq_id,
                         int64_t pos0) {
    EncodeParams p;
    p.dst = make_view(dst);
    p.src = static_cast<const __half *>(src);
    p.stride = stride;
    p.seq_ids = seq_ids;
    p.positions = positions;
    p.lens = nullptr;
    p.pos0 = pos0;
    p.n_tokens = n_tokens;
    p.seq_id = seq_id;
    p.bpr = dst.n_kv_heads * (dst.head_dim / kBlock);
    p.bpr_magic = div_magic((uint32_t)p.bpr);
    p.src_dense = stride == (int64_t)p.bpr * kBlock;
    p.rows_per_tile = kThreads / p.bpr;
    p.n_tiles = (n_tokens + p.rows_per_tile - 1) / p.rows_per_tile;
    p.row_bytes = p.dst.row_bytes;
    p.cpr_magic = div_magic((uint32_t)(p.row_bytes / 16 > 0 ? p.row_bytes / 16 : 1));
    p.hpr_magic = div_magic((uint32_t)(p.row_bytes / 2));
    return p;
}

}  // namespace

tq_status launch_encode(const tq_cache &dst, const void *src, int64_t n_tokens, int64_t stride,
                        const int32_t *seq_ids, const int32_t *positions, int32_t seq_id,
                        int64_t pos0, cudaStream_t stream) {
    const EncodeParams p = make_params(dst, src, n_tokens, stride, seq_ids, positions, seq_id, pos0);
    return dst.type == TQ_TURBO3 ? launch_encode_any<TQ_TURBO3>(p, p, 1, stream)
                                 : launch_encode_any<TQ_TURBO2>(p, p, 1, stream);
}

tq_status launch_encode_kv(const tq_cache &k, const tq_cache &v, const void *k_src,
                           const void *v_src, int64_t n_tokens, int64_t k_stride,
                           int64_t v_stride, const int32_t *seq_ids, const int32_t *positions,
                           int32_t seq_id, int64_t pos0, cudaStream_t stream) {
    const EncodeParams pk = make_params(k, k_src, n_tokens, k_stride, seq_ids, positions, seq_id, pos0);
    const EncodeParams pv = make_params(v, v_src, n_tokens, v_stride, seq_ids, positions, seq_id, pos0);
    if (k.type != v.type) {   // one template per type: two launches
        tq_status st = launch_encode(k, k_src, n_tokens, k_stride, seq_ids, positions, seq_id,
                                     pos0, stream);
        if (st != TQ_OK) return st;
        return launch_encode(v, v_src, n_tokens, v_stride, seq_ids, positions, seq_id, pos0, stream);
    }
    return k.type == TQ_TURBO3 ? launch_encode_any<TQ_TURBO3>(pk, pv, 2, stream)
                               : launch_encode_any<TQ_TURBO2>(pk, pv, 2, stream);
}

// Decode-step append for shapes the fused attention kernel does not take: sequence s's new
// K and V rows ([n_seqs][Hkv][D] fp16) go to position seq_lens[s] - 1 (none if 0).
tq_status launch_append(const tq_cache &k, const tq_cache &v, const void *k_new, const void *v_new,
                        const int32_t *seq_lens, int n_seqs, cudaStream_t stream) {
    EncodeParams pk = make_params(k, k_new, n_seqs, (int64_t)k.n_kv_heads * k.head_dim, nullptr,
                                  nullptr, 0, 0);
    EncodeParams pv = make_params(v, v_new, n_seqs, (int64_t)v.n_kv_heads * v.head_dim, nullptr,
                                  nullptr, 0, 0);
    pk.lens = seq_lens;
    pv.lens = seq_lens;
    if (k.type != v.type) {
        tq_status st = k.type == TQ_TURBO3 ? launch_encode_warp_t<TQ_TURBO3>(pk, pk, 1, stream)
                                           : launch_encode_warp_t<TQ_TURBO2>(pk, pk, 1, stream);
        if (st != TQ_OK) return st;
        return v.type == TQ_TURBO3 ? launch_encode_warp_t<TQ_TURBO3>(pv, pv, 1, stream)
                                   : launch_encode_warp_t<TQ_TURBO2>(pv, pv, 1, stream);
    }
    return k.type == TQ_TURBO3 ? launch_encode_warp_t<TQ_TURBO3>(pk, pv, 2, stream)
                               : launch_encode_warp_t<TQ_TURBO2>(pk, pv, 2, stream);
}

}  // namespace tq
