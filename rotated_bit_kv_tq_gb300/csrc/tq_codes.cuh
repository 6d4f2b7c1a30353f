// tq_codes.cuh -- packed codes to fp16 tensor-core operands, shared by the decode-attention
// and prompt-attention kernels.
//
// A 3-bit (turbo3) or 2-bit (turbo2) code becomes the fp16 value of its Lloyd-Max centroid
// through byte-permute (prmt) lookups in registers: eight codes form the nibbles of a
// selector, one prmt per byte plane looks up four low bytes and one four high bytes, and
// two more prmt interleave them into fp16 pairs.  Layout of the codes: tq.h ("Packed block
// layout").  Also the mma.sync / movmatrix / shuffle-FWHT helpers both kernels use.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.cuh"

namespace tq {
namespace {

// Shift amounts as multipliers (2, 4, 2^16, 2^30, 2^31); run-time values keep the selector
// shifts on integer multiply-adds.
struct Shifts {
    uint32_t mul2, mul4, hi16, hi30, hi31;
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

// d = A B with a zero accumulator (the first k-step of a sum): no registers to clear.
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
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

// (a, b) as an fp16 pair hi = fp16(a, b) plus the fp16 rounding of the remainders, lo.
__device__ __forceinline__ void split_half2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 f = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_half2(a - f.x, b - f.y);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


__device__ __forceinline__ float ld_norm(const uint8_t *blk) {
    return __half2float(*reinterpret_cast<const __half *>(blk));
}

// ------------------------------------------------------------------ code -> fp16 lookup
// Byte tables of the fp16 codebook: L = low bytes, H = high bytes of entries 0..7.
struct HalfTables {
    uint32_t l0, l1, h0, h1;
};

// Selector of 8 codes: nibble k = code of value 8r + k (k = 0..7) of a 16-value group whose
// low-plane word is W, high-plane bit 4k+p of V (layout of tq.h).  Left shifts are
// integer multiplies so that they issue on the FMA pipe, not the half-rate ALU pipe.
template <int TYPE>
__device__ __forceinline__ uint32_t sel8(uint32_t W, uint32_t V, int r, int p, const Shifts &k) {
    uint32_t x = (r ? __umulhi(W, k.hi30) : W) & 0x33333333u;      // W >> 2 for r = 1
    if (TYPE == TQ_TURBO3) {
        // bit 4k+p of V moves to 4k+2: V << 2, V << 1, V, V >> 1
        const uint32_t hv = p == 0 ? V * k.mul4 : p == 1 ? V * k.mul2 : p == 2 ? V : __umulhi(V, k.hi31);
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

// The 4 fp16x2 pairs (values 8r+2i, 8r+2i+1 for i = 0..3) of one selector.
__device__ __forceinline__ void pairs8(const HalfTables &t, uint32_t sel, uint32_t hi16,
                                       uint32_t (&o)[4]) {
    uint32_t L, H, Lh, Hh;
    lookup4(t, sel, L, H);
    lookup4(t, __umulhi(sel, hi16), Lh, Hh);   // sel >> 16 on the FMA pipe
    o[0] = prmt(L, H, 0x5140);
    o[1] = prmt(L, H, 0x7362);
    o[2] = prmt(Lh, Hh, 0x5140);
    o[3] = prmt(Lh, Hh, 0x7362);
}

// Code words of values 32 q4 .. 32 q4 + 31 of one packed block (2-byte aligned in shared
// memory; `sh` = 16 when the low-plane words sit at an address = 2 mod 4, else 0; the
// high-plane words then share that alignment because they start 32 bytes later).
template <int TYPE>
struct Quarter {
    uint32_t W0, W1, V;
};
// `row` is a 16-byte aligned packed row in shared memory; ow / ov are the word-aligned
// byte offsets (within the row) of the quarter's low-plane and high-plane words.
template <int TYPE>
__device__ __forceinline__ Quarter<TYPE> load_quarter(const uint8_t *row, int ow, int ov,
                                                      uint32_t sh) {
    Quarter<TYPE> r;
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row + ow);
    const uint32_t a = w[0], b = w[1], c = w[2];
    r.W0 = __funnelshift_r(a, b, sh);
    r.W1 = __funnelshift_r(b, c, sh);
    if (TYPE == TQ_TURBO3) {
        const uint32_t *v = reinterpret_cast<const uint32_t *>(row + ov);
        r.V = __funnelshift_r(v[0], v[1], sh);
    } else {
        r.V = 0u;
    }
    return r;
}

// Group (ww, r) of a quarter: the 4 pairs 8ww + 4r + {0..3}.
template <int TYPE>
__device__ __forceinline__ void group_pairs(const Quarter<TYPE> &qw, int ww, int r,
                                            const HalfTables &t, const Shifts &k,
                                            uint32_t (&o)[4]) {
    pairs8(t, sel8<TYPE>(ww ? qw.W1 : qw.W0, qw.V, r, 2 * ww + r, k), k.hi16, o);
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

// Byte tables of a type's fp16 codebook (entries past 2^type are zero).
template <int TYPE>
__device__ __forceinline__ HalfTables make_tables() {
    const __half *c = c_codebook[cb_index(TYPE)].centroid_h;
    uint32_t l[2] = {0, 0}, h[2] = {0, 0};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint16_t a = e < (1 << TYPE) ? __half_as_ushort(c[e]) : 0;
        l[e >> 2] |= (uint32_t)(a & 0xff) << (8 * (e & 3));
        h[e >> 2] |= (uint32_t)(a >> 8) << (8 * (e & 3));
    }
    return HalfTables{l[0], l[1], h[0], h[1]};
}

}  // namespace
}  // namespace tq
