// gq_mma_sync.cuh -- operand conversion and the m16n8k16 MMA shared by the
// warp-level tensor-core kernels (gq_skinny.cu, gq_skinny_q0.cu).  Codes
// become exact fp16 integers with the 0x6400 trick; within each group of
// eight elements both operands take the order (e0, e4, e1, e5, e2, e6, e3,
// e7), the order in which a nibble word unpacks, so lane (g, t) of a
// fragment holds elements 8 t .. 8 t + 7 of a 32-element K block.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace gq {
namespace ms {

__device__ __forceinline__ __half2 h2_bits(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ uint32_t bits_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Eight int8 codes e0..e3 (bytes of u0), e4..e7 (bytes of u1) as fp16 pairs
// (e0, e4), (e1, e5), (e2, e6), (e3, e7): a byte b ^ 0x80 in the mantissa of
// 0x6400 is the exact fp16 1024 + (b + 128), less 1152 is b.
__device__ __forceinline__ uint4 i8x8_to_f16(uint32_t u0, uint32_t u1) {
    const uint32_t x0 = __byte_perm(u0, u1, 0x5140) ^ 0x80808080u;
    const uint32_t x1 = __byte_perm(u0, u1, 0x7362) ^ 0x80808080u;
    const __half2 bias = __float2half2_rn(-1152.0f);
    return make_uint4(bits_h2(__hadd2(h2_bits(__byte_perm(x0, 0x64646464u, 0x4140)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x0, 0x64646464u, 0x4342)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x1, 0x64646464u, 0x4140)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x1, 0x64646464u, 0x4342)), bias)));
}

// One nibble word (byte i: element 2i low, 2i + 1 high) to the fp16 pairs
// (v e0, v e4), (v e1, v e5), (v e2, v e6), (v e3, v e7), v e an affine map of
// the nibble fixed by the fma constants k.  A nibble in mantissa bits 0-3
// (4-7) of 0x6400 is the exact fp16 1024 + e (1024 + 16 e); one fma with
// (k.x, k.y) for the low nibbles and (k.z, k.w) for the high ones maps it.
// Q4_K (v e = sc e - 512): k = (sc, -512 (2 sc + 1), sc / 16, -64 (sc + 8));
// Q4_0 (v e = e - 8): k = (1, -1032, 1 / 16, -72).  Both are exact: the
// product is exact inside the fma and the result is a representable integer.
__device__ __forceinline__ uint4 nib8_to_f16(uint32_t w, uint4 k) {
    const uint32_t w8 = w >> 8;
    const __half2 s1 = h2_bits(k.x), c1 = h2_bits(k.y), s16 = h2_bits(k.z), c16 = h2_bits(k.w);
    return make_uint4(bits_h2(__hfma2(h2_bits((w & 0x000F000Fu) | 0x64006400u), s1, c1)),
                      bits_h2(__hfma2(h2_bits((w & 0x00F000F0u) | 0x64006400u), s16, c16)),
                      bits_h2(__hfma2(h2_bits((w8 & 0x000F000Fu) | 0x64006400u), s1, c1)),
                      bits_h2(__hfma2(h2_bits((w8 & 0x00F000F0u) | 0x64006400u), s16, c16)));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// d += A * B on one m16n8k16 tile (fp16 operands, fp32 accumulate).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace ms
}  // namespace gq
