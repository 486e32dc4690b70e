// gq_quant8.cuh -- per-element Q8 code helpers shared by the GEMV kernels
// that quantize fp32 activations in the CTA (gq_gemv.cu, gq_q5k.cu,
// gq_q6k.cu).  Same operations, in the same order, as the standalone Q8_K /
// Q8_0 quantizers of gq_codec.cu (round-to-nearest division, roundf), with
// every rounding explicit, so the codes equal theirs bit for bit whatever the
// including file's contraction flags.
#pragma once

#include "gq_common.cuh"

namespace gq {
namespace q8 {

__device__ __forceinline__ float clamp127(float v) {
    return v < -127.0f ? -127.0f : (v > 127.0f ? 127.0f : v);
}

// Code of x in a block with scale d != 0 and r = RN(1/d): roundf of the
// IEEE quotient x / d, clamped to [-127, 127].  For |x / d| <= 128 the
// product p = RN(x * r) lies within 2^-16 of x / d and RN(x / d) within
// 2^-17, so the two round alike under roundf unless p is within 2^-15 of a
// half-integer; p's distance is tested against 2^-14 and the near cases
// (and a non-finite r, which makes the test fail through a NaN) take the
// IEEE division.  Away from a half-integer, roundf(|p|) = floor(|p|) + (frac
// > 1/2) exactly.
__device__ __forceinline__ float q8_code(float x, float d, float r) {
    const float p = __fmul_rn(x, r);
    const float a = fabsf(p);
    const float fl = floorf(a);
    const float f = a - fl;
    float q;
    if (fabsf(f - 0.5f) > 0x1p-14f)
        q = copysignf(fl + (f > 0.5f ? 1.0f : 0.0f), p);
    else
        q = roundf(__fdiv_rn(x, d));
    return clamp127(q);
}

// Codes of eight elements of a block with scale d and r = RN(1/d), packed as
// signed bytes (lowest element in the lowest byte), each equal to
// q8_code(e[i], d, r), and zero when d == 0.  Away from a half-integer the
// product p = RN(e * r) rounds the same to nearest-even (rintf) as half away
// from zero, and |p - rintf(p)| is exact, so the fast path tests the same
// 2^-14 window as q8_code and falls back to it for the whole group when any
// element lies in the window (or r is not finite, which makes the test fail).
// Every |e| <= 127 d up to the rounding of d (at most 2^-11 relative, for an
// fp16 scale), so |p| < 127.5 and the fast codes need no clamp.
__device__ __forceinline__ void q8_codes8(const float (&e)[8], float d, float r, uint32_t &w0,
                                          uint32_t &w1) {
    int q[8];
    bool slow = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float p = __fmul_rn(e[i], r);
        const float t = rintf(p);
        slow |= !(fabsf(fabsf(p - t) - 0.5f) > 0x1p-14f);
        q[i] = (int)t;
    }
    if (d == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = 0;
    } else if (slow) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = (int)q8_code(e[i], d, r);
    }
    w0 = __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
    w1 = __byte_perm(__byte_perm(q[4], q[5], 0x0040), __byte_perm(q[6], q[7], 0x0040), 0x5410);
}

__device__ __forceinline__ void unpack8(const float4 (&v)[2], float (&e)[8]) {
    e[0] = v[0].x; e[1] = v[0].y; e[2] = v[0].z; e[3] = v[0].w;
    e[4] = v[1].x; e[5] = v[1].y; e[6] = v[1].z; e[7] = v[1].w;
}

__device__ __forceinline__ float absmax8(const float (&e)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(e[i]));
    return m;
}

// Split-order words of 8 codes: (a0 a2 a4 a6) and (a1 a3 a5 a7).
__device__ __forceinline__ uint2 split8_codes(uint32_t w0, uint32_t w1) {
    return make_uint2(__byte_perm(w0, w1, 0x6420), __byte_perm(w0, w1, 0x7531));
}

// One fp32 activation vector of nblk 256-element blocks quantized to Q8_K
// straight into the staged layout of the Q5_K / Q6_K GEMVs: codes at `act`
// (unit u of half-block hb -- codes 16 u .. 16 u + 15 of the half -- at
// hb * 128 + (u ^ (hb & 7)) * 16, each group of eight as its split-order
// pair), then SPB int32 code sums per block (SPB = 8: the sub-block sums
// t_j; SPB = 2: the half-block sums), then one fp32 scale per block.  A warp
// takes a block, lane l its elements 8 l .. 8 l + 7; each warp loads four of
// its blocks before quantizing any, so their loads are in flight together.
template <int SPB>
__device__ void stage_q8_k_from_f32(uint8_t *act, const float *__restrict__ x, int nblk) {
    static_assert(SPB == 8 || SPB == 2, "sums per block");
    constexpr int LPS = 32 / SPB;  // lanes per summed group
    constexpr int NB = 4;
    int32_t *sums = reinterpret_cast<int32_t *>(act + (size_t)nblk * 256);
    float *dx = reinterpret_cast<float *>(sums + SPB * nblk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int b0 = warp; b0 < nblk; b0 += NB * nw) {
        float4 v[NB][2];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int blk = b0 + u * nw;
            if (blk < nblk) {
                const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)blk * 256 + 8 * lane);
                v[u][0] = __ldg(p);
                v[u][1] = __ldg(p + 1);
            } else {
                v[u][0] = v[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int blk = b0 + u * nw;
            if (blk >= nblk) break;  // warp-uniform
            float e[8];
            unpack8(v[u], e);
            float am = absmax8(e);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            const float d = __fdiv_rn(am, 127.0f), r = __frcp_rn(d);
            uint32_t w0, w1;
            q8_codes8(e, d, r, w0, w1);
            int s = __dp4a((int)w0, 0x01010101, __dp4a((int)w1, 0x01010101, 0));
#pragma unroll
            for (int o = 1; o < LPS; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const int hb = 2 * blk + (lane >> 4), unit = (lane & 15) >> 1;
            *reinterpret_cast<uint2 *>(act + (size_t)hb * 128 + ((unit ^ (hb & 7)) << 4) + 8 * (lane & 1)) =
                split8_codes(w0, w1);
            if ((lane & (LPS - 1)) == 0) sums[blk * SPB + lane / LPS] = s;
            if (lane == 0) dx[blk] = d;
        }
    }
}

}  // namespace q8
}  // namespace gq
