// tq_decode.cu -- dequantise packed rows back to fp32 (tests, quality reports).
//
// "llama.cpp に TurboQuant を実装", "What TurboQuant does differently": the rotation is
// undone at read time and, being a Walsh-Hadamard transform, is its own inverse up to the
// 1/sqrt(128) scale.  x_hat = norm * (1/sqrt(128)) * W c(codes), in fp32.
//
// One warp per 128-value block, four values per lane: the codes are unpacked from the
// two bit planes, the two in-lane butterfly stages run in registers and the five
// cross-lane stages use warp shuffles; each lane writes one float4, so a warp writes its
// 512-byte output row segment fully coalesced.
#include "tq_internal.cuh"

namespace tq {
namespace {

struct DecodeParams {
    CacheView src;
    float *dst;
    int64_t pos0;
    int64_t n_blocks;   // n_tokens * bpr
    int32_t seq_id;
    int32_t bpr;
};

template <int TYPE>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeParams p) {
    constexpr int B = block_bytes(TYPE);
    const int lane = threadIdx.x & 31;
    const int64_t blk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= p.n_blocks) return;
    const int64_t t = blk / p.bpr;
    const int fb = (int)(blk - t * p.bpr);
    const uint8_t *row = row_ptr(p.src, p.seq_id, p.pos0 + t);
    float4 *out = reinterpret_cast<float4 *>(p.dst + blk * kBlock) + lane;
    if (!row) {
        *out = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const uint8_t *b = row + fb * B;
    const Codebook &cb = c_codebook[cb_index(TYPE)];
    // values 4*lane .. 4*lane+3
    const int i0 = 4 * lane;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int i = i0 + e;
        const int j = i & 15;
        const int lb = 32 * (i >> 4) + 4 * (j & 7) + 2 * (j >> 3);   // low-plane bit
        int code = (b[2 + (lb >> 3)] >> (lb & 7)) & 3;
        if (TYPE == TQ_TURBO3) {
            const int jv = i & 31;
            const int hb = 32 * (i >> 5) + 4 * (jv & 7) + (jv >> 3);  // high-plane bit
            code |= ((b[34 + (hb >> 3)] >> (hb & 7)) & 1) << 2;
        }
        v[e] = cb.centroid[code];
    }
    // butterflies h = 1, 2 inside the lane
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
    // h = 4 .. 64 across lanes (lane stride h/4)
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
            v[e] = upper ? o - v[e] : v[e] + o;
        }
    }
    const uint16_t nb = (uint16_t)(b[0] | (b[1] << 8));
    const float sc = __half2float(__ushort_as_half(nb)) * kInvSqrt128;
    // rotation-sign variant: D W c, coordinate i negated when its sign bit is set
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = __uint_as_float(__float_as_uint(v[e] * sc) ^ sign_mask(p.src, i0 + e));
    *out = make_float4(o[0], o[1], o[2], o[3]);
}

}  // namespace

tq_status launch_decode(const tq_cache &src, int32_t seq_id, int64_t pos0, int64_t n_tokens,
                        float *dst, cudaStream_t stream) {
    DecodeParams p;
    p.src = make_view(src);
    p.dst = dst;
    p.pos0 = pos0;
    p.seq_id = seq_id;
    p.bpr = src.n_kv_heads * (src.head_dim / kBlock);
    p.n_blocks = n_tokens * p.bpr;
    const int64_t grid = (p.n_blocks + 7) / 8;
    if (grid > 0x7fffffff) return TQ_ERR_UNSUPPORTED;
    if (src.type == TQ_TURBO3)
        decode_kernel<TQ_TURBO3><<<(unsigned)grid, 256, 0, stream>>>(p);
    else
        decode_kernel<TQ_TURBO2><<<(unsigned)grid, 256, 0, stream>>>(p);
    return check_cuda(cudaGetLastError());
}

}  // namespace tq
