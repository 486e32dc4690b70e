// gq_codec.cu -- block codecs: quantize (fp32 -> blocks) and dequantize
// (blocks -> fp32) for Q4_0, Q8_0, Q4_K, Q5_K and Q8_K.
//
// Every step is the IEEE fp32 operation the format definition names, written
// with explicit round-to-nearest intrinsics (and this file is compiled with
// -fmad=false), so the bytes produced are identical to the reference
// definition:
//   "llama.cpp 推理引擎" (runguoli.com), §5.1 symmetric quantization
//   (scale = max|x| / (2^(b-1) - 1), Q = round(x / scale)) for Q8_0 (b = 8),
//   Q4_0 (b = 4, the §5.1 worked example) and the activation block Q8_K;
//   §5.2 asymmetric quantization (scale and zero point from the min/max) and
//   §5.5 (super-block scale d and min dmin over 6-bit per-sub-block factors)
//   for Q4_K and Q5_K (the 5-bit K-quant, one bit more than Q4_K: the
//   discosf.com page "为什么说 llama.cpp 是'裸引擎'…", §4; the same fit with
//   codes in [0, 31], their fifth bits in a bit plane of their own); §6.4
//   for the nibble order (element 2j in the low nibble of byte j).  Codes
//   round half away from zero (roundf).
//
// Work split: one warp per block.  Q8_0 / Q4_0: lane i owns element i.
// Q4_K / Q8_K: lane l owns elements 8l..8l+7, so the four lanes 4j..4j+3 own
// sub-block j and sub-block statistics are 2-step shuffle reductions.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

__device__ __forceinline__ float clampf(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// Symmetric block of 32 (Q8_0 when QMAX = 127, Q4_0 when QMAX = 7).  Source
// block b is element row b / row_blocks, block b % row_blocks of that row;
// destination rows are dst_row_stride blocks apart (row_blocks = nblocks for
// one contiguous run).
template <int QMAX>
__global__ void __launch_bounds__(256) quantize32_kernel(const float *__restrict__ x,
                                                         uint8_t *__restrict__ dst,
                                                         int64_t nblocks, int64_t row_blocks,
                                                         int64_t dst_row_stride) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    pdl_launch_dependents();  // dependents still wait for this grid's completion
    pdl_wait();
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += warps) {
        const float v = x[b * 32 + lane];
        const int64_t ob = (b / row_blocks) * dst_row_stride + b % row_blocks;  // destination block
        // max|x| (fabsf never yields -0, so the max of the block is well defined)
        const float amax = warp_max(fabsf(v));
        const __half dh = __float2half_rn(__fdiv_rn(amax, (float)QMAX));
        const float d = __half2float(dh);
        if (QMAX == 127) {
            const float q = (d == 0.0f) ? 0.0f : clampf(roundf(__fdiv_rn(v, d)), -127.0f, 127.0f);
            const int qi = (int)q & 0xff;
            const int nxt = __shfl_down_sync(FULL, qi, 1);
            uint8_t *blk = dst + ob * Q8_0_BYTES;
            if ((lane & 1) == 0)
                *reinterpret_cast<uint16_t *>(blk + 2 + lane) = (uint16_t)(qi | (nxt << 8));
            if (lane == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(dh);
        } else {
            const float q = (d == 0.0f) ? 0.0f : clampf(roundf(__fdiv_rn(v, d)), -8.0f, 7.0f);
            const int c = (int)q + 8;  // stored code 0..15
            const int hi = __shfl_down_sync(FULL, c, 1);
            const int byte = c | (hi << 4);  // valid on even lanes: element 2j low, 2j+1 high
            const int byte2 = __shfl_down_sync(FULL, byte, 2);
            uint8_t *blk = dst + ob * Q4_0_BYTES;
            if ((lane & 3) == 0)
                *reinterpret_cast<uint16_t *>(blk + 2 + (lane >> 1)) =
                    (uint16_t)((byte & 0xff) | ((byte2 & 0xff) << 8));
            if (lane == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(dh);
        }
    }
}

// Q8_K: 256 elements, fp32 scale d = max|x| / 127, eight int16 sub-block sums.
__global__ void __launch_bounds__(256) quantize_q8_k_kernel(const float *__restrict__ x,
                                                            uint8_t *__restrict__ dst,
                                                            int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    pdl_launch_dependents();  // dependents still wait for this grid's completion
    pdl_wait();
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += warps) {
        const float *xb = x + b * QK_K + 8 * lane;
        float v[8];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = xb[i];
            amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = warp_max(amax);
        const float d = __fdiv_rn(amax, 127.0f);
        uint32_t w0 = 0, w1 = 0;
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q =
                (d == 0.0f) ? 0.0f : clampf(roundf(__fdiv_rn(v[i], d)), -127.0f, 127.0f);
            const int qi = (int)q;
            sum += qi;
            if (i < 4)
                w0 |= (uint32_t)(qi & 0xff) << (8 * i);
            else
                w1 |= (uint32_t)(qi & 0xff) << (8 * (i - 4));
        }
        sum += __shfl_xor_sync(FULL, sum, 1);
        sum += __shfl_xor_sync(FULL, sum, 2);
        uint8_t *blk = dst + b * Q8_K_BYTES;
        reinterpret_cast<uint32_t *>(blk + 4 + 8 * lane)[0] = w0;
        reinterpret_cast<uint32_t *>(blk + 4 + 8 * lane)[1] = w1;
        if ((lane & 3) == 0)
            *reinterpret_cast<int16_t *>(blk + 260 + 2 * (lane >> 2)) = (int16_t)sum;
        if (lane == 0) *reinterpret_cast<float *>(blk) = d;
    }
}

// Q4_K (QMAX = 15) and Q5_K (QMAX = 31): per 32-element sub-block j (lanes
// 4j..4j+3):
//   lo_j = min(0, min x), hi_j = max x
//   dmin = fp16_up(max_j(-lo_j) / 63), m_j = min(63, ceil(-lo_j / dmin))
//   base_j = -(dmin * m_j), r_j = hi_j - base_j
//   d = fp16_up(max_j r_j / (63 QMAX)), sc_j = min(63, ceil(r_j / (QMAX d)))
//   q = clamp(round((x - base_j) / (d * sc_j)), 0, QMAX)
// The low four bits of the codes fill bytes 16..143 (element 2l in the low
// nibble of byte 16 + l); Q5_K puts the fifth bit of element
// 32j + 8t + 2i + p into bit 2t + p of byte 144 + 4j + i.
//
// ERRMIN: the error-minimizing refinement ("llama.cpp 推理引擎" §5.5 with
// §7.1: sub-block scales chosen for the least reconstruction error, uniform
// importance).  d and dmin stay the fit's; per sub-block every (sc, m) within
// EM_WINDOW of the fit's pair (clipped to 0..63) is scored by the squared
// error of its 32 reconstructed values (codes the nearest in [0, QMAX]),
// computed in fp32 in a fixed order -- each lane's eight elements in turn,
// then (g0 + g1) + (g2 + g3) over the sub-block's four lanes -- and the first
// candidate in (sc, m) ascending order strictly below the best so far wins,
// starting from the fit's pair.
constexpr int EM_WINDOW = 4;

// Squared reconstruction error of this lane's sub-block (all four lanes get
// the same value) for the pair (sc, m).
template <int QMAX>
__device__ __forceinline__ float em_sub_error(const float (&v)[8], float d, float dmin, float sc, float m) {
    const float step = __fmul_rn(d, sc);
    const float base = -__fmul_rn(dmin, m);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float q =
            (step == 0.0f) ? 0.0f : clampf(roundf(__fdiv_rn(__fsub_rn(v[i], base), step)), 0.0f, (float)QMAX);
        const float e = __fsub_rn(v[i], __fadd_rn(__fmul_rn(step, q), base));
        acc = __fadd_rn(acc, __fmul_rn(e, e));
    }
    acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, 1));
    return __fadd_rn(acc, __shfl_xor_sync(FULL, acc, 2));
}

template <int QMAX, bool ERRMIN>
__global__ void __launch_bounds__(256) quantize_k_kernel(const float *__restrict__ x,
                                                         uint8_t *__restrict__ dst,
                                                         int64_t nblocks) {
    constexpr int BYTES = QMAX == 15 ? Q4_K_BYTES : Q5_K_BYTES;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    pdl_launch_dependents();  // dependents still wait for this grid's completion
    pdl_wait();
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks;
         b += warps) {
        const float *xb = x + b * QK_K + 8 * lane;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = xb[i];
        float mn = v[0], mx = v[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) {
            mn = fminf(mn, v[i]);
            mx = fmaxf(mx, v[i]);
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(FULL, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
        }
        const float lo = mn < 0.0f ? mn : 0.0f;
        const float hi = mx;
        // max over sub-blocks of -lo_j, as a +0-initialised maximum
        float nlo = mn < 0.0f ? -mn : 0.0f;
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) nlo = fmaxf(nlo, __shfl_xor_sync(FULL, nlo, o));
        if (!(nlo > 0.0f)) nlo = 0.0f;
        const __half dminh = __float2half_ru(__fdiv_rn(nlo, 63.0f));
        const float dmin = __half2float(dminh);
        float m = (dmin == 0.0f) ? 0.0f : ceilf(__fdiv_rn(-lo, dmin));
        if (m > 63.0f) m = 63.0f;
        float base = -__fmul_rn(dmin, m);
        const float r = __fsub_rn(hi, base);
        float rmax = r;
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) rmax = fmaxf(rmax, __shfl_xor_sync(FULL, rmax, o));
        if (!(rmax > 0.0f)) rmax = 0.0f;
        const __half dh = __float2half_ru(__fdiv_rn(rmax, (float)(63 * QMAX)));
        const float d = __half2float(dh);
        float sc = (d == 0.0f) ? 0.0f : ceilf(__fdiv_rn(r, __fmul_rn((float)QMAX, d)));
        if (sc > 63.0f) sc = 63.0f;
        if (ERRMIN) {
            const float sc0 = sc, m0 = m;
            float best = em_sub_error<QMAX>(v, d, dmin, sc0, m0);
            for (int a = -EM_WINDOW; a <= EM_WINDOW; ++a) {
                for (int c = -EM_WINDOW; c <= EM_WINDOW; ++c) {
                    const float cs = sc0 + (float)a, cm = m0 + (float)c;
                    const bool ok = cs >= 0.0f && cs <= 63.0f && cm >= 0.0f && cm <= 63.0f;
                    const float e = em_sub_error<QMAX>(v, d, dmin, ok ? cs : sc0, ok ? cm : m0);  // uniform shuffles
                    if (ok && e < best) {
                        best = e;
                        sc = cs;
                        m = cm;
                    }
                }
            }
            base = -__fmul_rn(dmin, m);
        }
        const float step = __fmul_rn(d, sc);
        uint32_t packed = 0, fifth = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q = (step == 0.0f)
                                ? 0.0f
                                : clampf(roundf(__fdiv_rn(__fsub_rn(v[i], base), step)), 0.0f,
                                         (float)QMAX);
            const uint32_t qi = (uint32_t)q;
            packed |= (qi & 15u) << (4 * i);  // element 8l+i -> nibble i of the word
            // element 8l + i = 32j + 8t + 2(i/2) + (i&1), t = l % 4: fifth bit
            // to bit 8(i/2) + 2t + (i&1) of the sub-block's fifth-bit word
            fifth |= (qi >> 4) << (8 * (i >> 1) + 2 * (lane & 3) + (i & 1));
        }
        uint8_t *blk = dst + b * BYTES;
        reinterpret_cast<uint32_t *>(blk + 16)[lane] = packed;
        if (QMAX == 31) {
            fifth |= __shfl_xor_sync(FULL, fifth, 1);
            fifth |= __shfl_xor_sync(FULL, fifth, 2);
            if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(blk + 144)[lane >> 2] = fifth;
        }
        // gather the eight (sc_j, m_j) pairs and pack sixteen 6-bit fields
        uint32_t w[3] = {0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t scj = (uint32_t)__shfl_sync(FULL, (int)sc, 4 * j);
            const uint32_t mj = (uint32_t)__shfl_sync(FULL, (int)m, 4 * j);
#pragma unroll
            for (int f = 0; f < 2; ++f) {
                const uint32_t val = f ? mj : scj;
                const int bit = 6 * (j + 8 * f);
                const int wi = bit >> 5, sh = bit & 31;
                w[wi] |= val << sh;
                if (sh > 26) w[wi + 1] |= val >> (32 - sh);
            }
        }
        if (lane == 0) {
            uint32_t *hdr = reinterpret_cast<uint32_t *>(blk);
            hdr[0] = (uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(dminh) << 16);
            hdr[1] = w[0];
            hdr[2] = w[1];
            hdr[3] = w[2];
        }
    }
}

// ------------------------------------------------------------------ decoders
// One thread per element; each output is the exact reconstruction rounded
// once to fp32 (products of the scales with the small integer codes are
// exact in fp32, only the Q4_K difference and the fp32 Q8_K product round).

__global__ void dequantize_kernel(int type, const uint8_t *__restrict__ src,
                                  float *__restrict__ dst, int64_t n) {
    pdl_launch_dependents();  // dependents still wait for this grid's completion
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
        float out;
        if (type == GQ_Q4_0) {
            const uint8_t *blk = src + (e >> 5) * Q4_0_BYTES;
            const int i = (int)(e & 31);
            const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
            const int byte = blk[2 + (i >> 1)];
            const int c = (i & 1) ? (byte >> 4) : (byte & 15);
            out = __fmul_rn(d, (float)(c - 8));
        } else if (type == GQ_Q8_0) {
            const uint8_t *blk = src + (e >> 5) * Q8_0_BYTES;
            const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
            out = __fmul_rn(d, (float)(int8_t)blk[2 + (e & 31)]);
        } else if (type == GQ_Q4_K || type == GQ_Q5_K) {
            const uint8_t *blk = src + (e >> 8) * (type == GQ_Q4_K ? Q4_K_BYTES : Q5_K_BYTES);
            const int i = (int)(e & 255), j = i >> 5;
            const uint32_t *hdr = reinterpret_cast<const uint32_t *>(blk);
            const float d = half_bits_to_float(hdr[0]);
            const float dmin = half_bits_to_float(hdr[0] >> 16);
            const uint64_t lo64 = (uint64_t)hdr[1] | ((uint64_t)hdr[2] << 32);
            const uint64_t hi64 = (uint64_t)hdr[2] | ((uint64_t)hdr[3] << 32);
            const float sc = (float)((lo64 >> (6 * j)) & 63);
            const float m = (float)((hi64 >> (6 * j + 16)) & 63);
            const int byte = blk[16 + (i >> 1)];
            int qi = (i & 1) ? (byte >> 4) : (byte & 15);
            if (type == GQ_Q5_K) {
                const int r = i & 31;  // element 8t + 2i' + p of sub-block j
                qi |= ((blk[144 + 4 * j + ((r & 7) >> 1)] >> (2 * (r >> 3) + (r & 1))) & 1) << 4;
            }
            const float q = (float)qi;
            out = __fsub_rn(__fmul_rn(__fmul_rn(d, sc), q), __fmul_rn(dmin, m));
        } else {
            const uint8_t *blk = src + (e >> 8) * Q8_K_BYTES;
            const float d = *reinterpret_cast<const float *>(blk);
            out = __fmul_rn(d, (float)(int8_t)blk[4 + (e & 255)]);
        }
        dst[e] = out;
    }
}

int grid_for(int64_t work_items, int per_cta, int num_sms) {
    int64_t g = (work_items + per_cta - 1) / per_cta;
    const int64_t cap = (int64_t)num_sms * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

}  // namespace

cudaError_t launch_quantize(gq_type t, const float *src, void *dst, int64_t n,
                            const LaunchCtx &ctx) {
    const int64_t nb = n / (t == GQ_Q4_K || t == GQ_Q5_K || t == GQ_Q8_K ? QK_K : 32);
    const int grid = grid_for(nb, 8, ctx.num_sms);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    switch (t) {
    case GQ_Q8_0:
        return launch_pdl(quantize32_kernel<127>, grid, 256, 0, ctx.stream, src, d8, nb, std::max<int64_t>(nb, 1),
                          (int64_t)0);
    case GQ_Q4_0:
        return launch_pdl(quantize32_kernel<7>, grid, 256, 0, ctx.stream, src, d8, nb, std::max<int64_t>(nb, 1),
                          (int64_t)0);
    case GQ_Q4_K:
        return launch_pdl(quantize_k_kernel<15, false>, grid, 256, 0, ctx.stream, src, d8, nb);
    case GQ_Q5_K:
        return launch_pdl(quantize_k_kernel<31, false>, grid, 256, 0, ctx.stream, src, d8, nb);
    case GQ_Q8_K:
        return launch_pdl(quantize_q8_k_kernel, grid, 256, 0, ctx.stream, src, d8, nb);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_k_errmin(gq_type t, const float *src, void *dst, int64_t n, const LaunchCtx &ctx) {
    const int64_t nb = n / QK_K;
    const int grid = grid_for(nb, 8, ctx.num_sms);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    if (t == GQ_Q4_K) return launch_pdl(quantize_k_kernel<15, true>, grid, 256, 0, ctx.stream, src, d8, nb);
    if (t == GQ_Q5_K) return launch_pdl(quantize_k_kernel<31, true>, grid, 256, 0, ctx.stream, src, d8, nb);
    return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_rows_strided(gq_type t, const float *src, void *dst, int64_t rows,
                                         int64_t row_blocks, int64_t dst_row_stride, const LaunchCtx &ctx) {
    const int64_t nb = rows * row_blocks;
    const int grid = grid_for(nb, 8, ctx.num_sms);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    switch (t) {
    case GQ_Q8_0:
        return launch_pdl(quantize32_kernel<127>, grid, 256, 0, ctx.stream, src, d8, nb, row_blocks, dst_row_stride);
    case GQ_Q4_0:
        return launch_pdl(quantize32_kernel<7>, grid, 256, 0, ctx.stream, src, d8, nb, row_blocks, dst_row_stride);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dequantize(gq_type t, const void *src, float *dst, int64_t n,
                              const LaunchCtx &ctx) {
    const int grid = grid_for(n, 256, ctx.num_sms);
    return launch_pdl(dequantize_kernel, grid, 256, 0, ctx.stream, (int)t,
                      static_cast<const uint8_t *>(src), dst, n);
}

}  // namespace gq
