// tq_encode_warp.cuh -- one 128-value block encoded by one warp, four values per lane.
// Used by the small-append encoder (tq_encode.cu) and by the decode-step attention kernel
// that appends the new token itself (tq_attn_mma.cu).
//
// "llama.cpp に TurboQuant を実装", "What TurboQuant does differently" / "How small does it
// get": norm, FWHT, Lloyd-Max index, bit-pack.  The operation order is the one of the
// one-thread-per-block encoder: the norm tree pairs element i with i + len/2 (lanes xor
// 16, 8, 4, 2, 1, then in-lane), butterflies run h = 1, 2 (in-lane) and 4 .. 64 (lanes xor
// 1 .. 16), every operation rounded separately, so codes and norms are the same bits.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.cuh"

namespace tq {
namespace {

// Squared centroid of a value's code: it depends only on the magnitude index
// m = #{positive thresholds below |y|} (the codebook is symmetric).
template <int TYPE>
__device__ __forceinline__ float code_sq(const Codebook &cb, float y) {
    constexpr int L = 1 << TYPE;
    const float a = fabsf(y);
    int m = a > cb.threshold[L / 2] ? 1 : 0;
    if (TYPE == TQ_TURBO3) m += (a > cb.threshold[5] ? 1 : 0) + (a > cb.threshold[6] ? 1 : 0);
    const float c = cb.centroid[L / 2 + m];
    return __fmul_rn(c, c);
}

// The packed form of one block, spread over the warp: the norm (every lane), this lane's
// 16-value low-plane word (complete in lanes 4j) and 32-value high-plane word (complete in
// lanes 8j, turbo3 only).
struct WarpBlock {
    uint16_t norm16;
    uint32_t wlo, whi;
};

// This lane's share of a block's fp16 source: values 4 lane .. 4 lane + 3 of the 128 at
// `src` (8-byte aligned).
__device__ __forceinline__ uint2 warp_block_load(const __half *src, int lane) {
    return *reinterpret_cast<const uint2 *>(src + 4 * lane);
}

// Encode a block from the lanes' shares `raw` (warp_block_load); `cv` supplies the variant
// flags (rotation signs, norm correction).
template <int TYPE>
__device__ __forceinline__ WarpBlock warp_encode_raw(uint2 raw, const CacheView &cv, int lane) {
    const Codebook &cb = c_codebook[cb_index(TYPE)];
    constexpr int L = 1 << TYPE;
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
    float x[4] = {f01.x, f01.y, f23.x, f23.y};
    if (cv.has_signs) {   // rotation-sign variant: W D
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __uint_as_float(__float_as_uint(x[e]) ^ sign_mask(cv, 4 * lane + e));
    }
    // norm
    float sq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sq[e] = __fmul_rn(x[e], x[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int e = 0; e < 4; ++e) sq[e] = __fadd_rn(sq[e], __shfl_xor_sync(0xffffffffu, sq[e], off));
    const float n = __fsqrt_rn(__fadd_rn(__fadd_rn(sq[0], sq[2]), __fadd_rn(sq[1], sq[3])));
    uint16_t norm16 = __half_as_ushort(__float2half_rn(fminf(n, 65504.0f)));
    const float k = n > 0.0f ? __fdiv_rn(kInvSqrt128, n) : 0.0f;
    // butterflies
    {
        const float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
        const float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
        x[0] = __fadd_rn(a0, a2);
        x[2] = __fsub_rn(a0, a2);
        x[1] = __fadd_rn(a1, a3);
        x[3] = __fsub_rn(a1, a3);
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = lane & m;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
            x[e] = upper ? __fsub_rn(o, x[e]) : __fadd_rn(x[e], o);
        }
    }
    // sign-magnitude quantiser: m = #{positive thresholds strictly below |y|},
    // code = signbit(y) ? L/2 - 1 - m : L/2 + m; pack into this lane's share of the words
    float ys[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) ys[e] = __fmul_rn(x[e], k);
    if (cv.norm_correction) {   // store |x| / |c|, |c| over the norm's pairwise tree
        float c2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) c2[e] = code_sq<TYPE>(cb, ys[e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int e = 0; e < 4; ++e) c2[e] = __fadd_rn(c2[e], __shfl_xor_sync(0xffffffffu, c2[e], off));
        const float cn = __fsqrt_rn(__fadd_rn(__fadd_rn(c2[0], c2[2]), __fadd_rn(c2[1], c2[3])));
        norm16 = __half_as_ushort(__float2half_rn(fminf(__fdiv_rn(n, cn), 65504.0f)));
    }
    uint32_t wlo = 0, whi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float y = ys[e];
        const float a = fabsf(y);
        uint32_t m = 0;
#pragma unroll
        for (int j = L / 2; j <= L - 2; ++j) m += a > cb.threshold[j] ? 1u : 0u;
        const uint32_t c = signbit(y) ? (uint32_t)(L / 2 - 1) - m : (uint32_t)(L / 2) + m;
        const int jl = 4 * (lane & 3) + e;          // value index within its 16-value word
        wlo |= (c & 3u) << (4 * (jl & 7) + 2 * (jl >> 3));
        if (TYPE == TQ_TURBO3) {
            const int jh = 4 * (lane & 7) + e;      // value index within its 32-value word
            whi |= (c >> 2) << (4 * (jh & 7) + (jh >> 3));
        }
    }
    wlo |= __shfl_xor_sync(0xffffffffu, wlo, 1);
    wlo |= __shfl_xor_sync(0xffffffffu, wlo, 2);
    if (TYPE == TQ_TURBO3) {
        whi |= __shfl_xor_sync(0xffffffffu, whi, 1);
        whi |= __shfl_xor_sync(0xffffffffu, whi, 2);
        whi |= __shfl_xor_sync(0xffffffffu, whi, 4);
    }
    return WarpBlock{norm16, wlo, whi};
}

// Encode the 128 fp16 values at `src` (8-byte aligned).
template <int TYPE>
__device__ __forceinline__ WarpBlock warp_encode_block(const __half *src, const CacheView &cv,
                                                       int lane) {
    return warp_encode_raw<TYPE>(warp_block_load(src, lane), cv, lane);
}

// Store a warp-encoded block at `o` (2-byte aligned; the block's byte layout of tq.h).
template <int TYPE>
__device__ __forceinline__ void warp_store_block(uint8_t *dst, const WarpBlock &wb, int lane) {
    uint16_t *o = reinterpret_cast<uint16_t *>(dst);
    if (lane == 0) o[0] = wb.norm16;
    if ((lane & 3) == 0) {
        o[1 + 2 * (lane >> 2)] = (uint16_t)(wb.wlo & 0xffffu);
        o[2 + 2 * (lane >> 2)] = (uint16_t)(wb.wlo >> 16);
    }
    if (TYPE == TQ_TURBO3 && (lane & 7) == 0) {
        o[17 + 2 * (lane >> 3)] = (uint16_t)(wb.whi & 0xffffu);
        o[18 + 2 * (lane >> 3)] = (uint16_t)(wb.whi >> 16);
    }
}

}  // namespace
}  // namespace tq
