// gq_gemv.cu -- memory-bound GEMV kernels (and their small-batch form) for
// Q4_K x Q8_K, Q4_0 x Q8_0 and Q8_0 x Q8_0.
//
// The per-block integer dot of "llama.cpp 推理引擎" (runguoli.com) §6.4 --
// low nibble of byte j pairs with activation 2j, high nibble with 2j+1, the
// block offset of 8 is applied to the integer sum, and the block scales
// multiply the integer result -- done with __dp4a on int8 activations; the
// two-level Q4_K scales of §5.5 are applied per 32-element sub-block in
// integers (sc_j * s_j, m_j * t_j) before one float scaling per super-block.
// Token generation is bound by memory bandwidth ("llama.cpp 推理引擎" §7.3),
// so the kernels are built to stream the weights once at HBM speed:
//   - every warp owns whole rows (grid-stride over rows, a persistent grid
//     of a few CTAs per SM for tall matrices) and streams each row through
//     its own two-stage shared-memory ring, filled by the TMA engine
//     (cp.async.bulk, ~2.3 KB chunks, completion on an mbarrier; every wait
//     is bounded);
//   - the CTA's activation vectors are staged once in shared memory, each
//     group of 8 int8 codes stored as (a0,a2,a4,a6 | a1,a3,a5,a7) so a
//     packed nibble word w feeds dp4a as (w & 0x0F0F0F0F) and
//     ((w >> 4) & 0x0F0F0F0F); the fused variants quantize fp32
//     activations straight into that layout (same arithmetic as the
//     standalone quantizer, so the codes are identical);
//   - Q4_0 / Q8_0 blocks (18 / 34 bytes, 2-byte aligned) are read from the
//     ring with aligned 32-bit loads and funnel shifts;
//   - per-lane fp32 partial sums, one warp-shuffle reduction per row.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr unsigned FULL = 0xffffffffu;
// Launch-shape parameters (compile-time; the defaults are the measured best).
#ifndef GQ_GEMV_NSTAGE
#define GQ_GEMV_NSTAGE 2
#endif
#ifndef GQ_GEMV_ROWS_PER_WARP
#define GQ_GEMV_ROWS_PER_WARP 2
#endif
#ifndef GQ_GEMV_CTAS_PER_SM
#define GQ_GEMV_CTAS_PER_SM 4
#endif
#ifndef GQ_GEMV_Q4K_CHUNK
#define GQ_GEMV_Q4K_CHUNK 16
#endif
#ifndef GQ_GEMV_EARLY_TRIGGER
#define GQ_GEMV_EARLY_TRIGGER 0
#endif

constexpr int WARPS = 8;                  // warps per CTA
constexpr int NSTAGE = GQ_GEMV_NSTAGE;    // ring stages per warp

// Weight formats as seen by the streaming kernel: block bytes, elements per
// block, and blocks per ring chunk (chunks are 16-byte multiples).
template <int WT>
struct Fmt;
template <>
struct Fmt<GQ_Q4_0> {
    static constexpr int BB = Q4_0_BYTES, BE = 32, CH = 128;  // 2304-byte chunks
};
template <>
struct Fmt<GQ_Q8_0> {
    static constexpr int BB = Q8_0_BYTES, BE = 32, CH = 64;  // 2176-byte chunks
};
template <>
struct Fmt<GQ_Q4_K> {
    static constexpr int BB = Q4_K_BYTES, BE = 256, CH = GQ_GEMV_Q4K_CHUNK;  // 2304-byte chunks
};

template <int WT, int NW>
struct Ring {
    static constexpr int CHUNK = Fmt<WT>::CH * Fmt<WT>::BB;
    static constexpr int BUF = ((CHUNK + 16 + 15) / 16) * 16;  // +16: over-read slack
    // WARPS * NSTAGE mbarriers of 8 bytes come first, then the ring buffers
    static constexpr int BARS_BYTES = NW * NSTAGE * 8;
    static constexpr int BUFS_OFF = ((BARS_BYTES + 127) / 128) * 128;
    static_assert(BUFS_OFF >= BARS_BYTES, "mbarriers must not overlap the ring");
    static_assert(BUFS_OFF % 16 == 0 && BUF % 16 == 0, "bulk-copy destinations are 16-byte aligned");
    static constexpr int ACT_OFF = BUFS_OFF + NW * NSTAGE * BUF;
};

// Staged activations.  Q8_K (for Q4_K weights): per vector and super-block
// 256 code bytes, the fp32 scale and the eight sub-block sums.  Q8_0 (for
// Q4_0 / Q8_0 weights): per vector and block 32 code bytes, the scale as
// fp32 and the sum of the 32 codes (for the Q4_0 offset of 8).
struct Act {
    uint8_t *codes;
    float *dx;
    int32_t *isum;
};

template <int WT>
__host__ __device__ constexpr int act_block_bytes() {
    return WT == GQ_Q4_K ? 256 + 4 + 32 : 32 + 4 + 4;
}

template <int WT>
__device__ __forceinline__ Act act_layout(uint8_t *base, int nb, int nblk) {
    constexpr int CB = WT == GQ_Q4_K ? 256 : 32;
    Act a;
    a.codes = base;
    a.dx = reinterpret_cast<float *>(base + (size_t)nb * nblk * CB);
    a.isum = reinterpret_cast<int32_t *>(a.dx + (size_t)nb * nblk);
    return a;
}

__device__ __forceinline__ uint2 split8(uint32_t a0, uint32_t a1) {
    return make_uint2(__byte_perm(a0, a1, 0x6420), __byte_perm(a0, a1, 0x7531));
}

// ---- unfused staging: copy quantized activation blocks into the layout.
// All loads of a pass are issued before any store, so a pass costs one
// L2 round trip.

__device__ void stage_q8_k(const Act &a, const uint8_t *__restrict__ xq, int nblocks) {
    const int groups = nblocks * 32;
    // pass p copies groups [4p*T, 4(p+1)*T) and block headers [p*T, (p+1)*T)
    // (T = blockDim.x); there are at least as many group passes as header
    // passes since every block has 32 groups.
    int pass = 0;
    for (int base = 0; base < groups; base += 4 * blockDim.x, ++pass) {
        uint32_t w0[4], w1[4], hd[5];
        const int hb = pass * blockDim.x + threadIdx.x;
        const bool has_h = hb < nblocks;
        if (has_h) {
            const uint8_t *src = xq + (size_t)hb * Q8_K_BYTES;
            hd[0] = __ldg(reinterpret_cast<const uint32_t *>(src));
#pragma unroll
            for (int i = 0; i < 4; ++i) hd[1 + i] = __ldg(reinterpret_cast<const uint32_t *>(src + 260) + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * blockDim.x + threadIdx.x;
            if (g < groups) {
                const uint32_t *src = reinterpret_cast<const uint32_t *>(
                    xq + (size_t)(g >> 5) * Q8_K_BYTES + 4 + 8 * (g & 31));
                w0[u] = __ldg(src);
                w1[u] = __ldg(src + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * blockDim.x + threadIdx.x;
            if (g < groups) reinterpret_cast<uint2 *>(a.codes)[g] = split8(w0[u], w1[u]);
        }
        if (has_h) {
            a.dx[hb] = __uint_as_float(hd[0]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a.isum[hb * 8 + 2 * i] = (int32_t)(int16_t)(hd[1 + i] & 0xffffu);
                a.isum[hb * 8 + 2 * i + 1] = (int32_t)(int16_t)(hd[1 + i] >> 16);
            }
        }
    }
}

template <bool SPLIT>
__device__ void stage_q8_0(const Act &a, const uint8_t *__restrict__ xq, int nblocks) {
    for (int base = 0; base < nblocks; base += blockDim.x) {
        const int blk = base + threadIdx.x;
        if (blk >= nblocks) continue;
        const uint16_t *src = reinterpret_cast<const uint16_t *>(xq + (size_t)blk * Q8_0_BYTES);
        uint32_t h[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) h[i] = __ldg(src + i);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = h[1 + 2 * i] | (h[2 + 2 * i] << 16);
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = dp4a((int)w[i], 0x01010101, s);
        a.isum[blk] = s;
        a.dx[blk] = half_bits_to_float(h[0]);
        uint4 *dst = reinterpret_cast<uint4 *>(a.codes + (size_t)blk * 32);
        if (SPLIT) {
            const uint2 p0 = split8(w[0], w[1]), p1 = split8(w[2], w[3]);
            const uint2 p2 = split8(w[4], w[5]), p3 = split8(w[6], w[7]);
            dst[0] = make_uint4(p0.x, p0.y, p1.x, p1.y);
            dst[1] = make_uint4(p2.x, p2.y, p3.x, p3.y);
        } else {
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

// ---- fused staging: quantize fp32 activations straight into the layout.
// Same operations, in the same order, as the standalone Q8_K / Q8_0
// quantizers (round-to-nearest division, roundf, fp16 round-to-nearest for
// the Q8_0 scale), so the codes equal theirs bit for bit.

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

__device__ __forceinline__ float clamp127(float v) {
    return v < -127.0f ? -127.0f : (v > 127.0f ? 127.0f : v);
}

// Q8_K: one warp per 256-element block, lane l owns elements 8l..8l+7
// (= code group l of the layout).
__device__ void quant_stage_q8_k(const Act &a, const float *__restrict__ x, int nblocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int b0 = warp; b0 < nblocks; b0 += 2 * nw) {
        float4 v[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int blk = b0 + u * nw;
            if (blk < nblocks) {
                const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)blk * QK_K + 8 * lane);
                v[u][0] = __ldg(p);
                v[u][1] = __ldg(p + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int blk = b0 + u * nw;
            if (blk >= nblocks) break;  // warp-uniform
            const float e[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(e[i]));
            amax = warp_max(amax);
            const float d = __fdiv_rn(amax, 127.0f);
            uint32_t w0 = 0, w1 = 0;
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float q = (d == 0.0f) ? 0.0f : clamp127(roundf(__fdiv_rn(e[i], d)));
                const int qi = (int)q;
                sum += qi;
                if (i < 4)
                    w0 |= (uint32_t)(qi & 0xff) << (8 * i);
                else
                    w1 |= (uint32_t)(qi & 0xff) << (8 * (i - 4));
            }
            reinterpret_cast<uint2 *>(a.codes)[(size_t)blk * 32 + lane] = split8(w0, w1);
            sum += __shfl_xor_sync(FULL, sum, 1);
            sum += __shfl_xor_sync(FULL, sum, 2);
            if ((lane & 3) == 0) a.isum[blk * 8 + (lane >> 2)] = sum;
            if (lane == 0) a.dx[blk] = d;
        }
    }
}

// Q8_0: one warp per 32-element block, lane = element.
template <bool SPLIT>
__device__ void quant_stage_q8_0(const Act &a, const float *__restrict__ x, int nblocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // position of this lane's code in the staged block
    const int e = lane & 7;
    const int pos = SPLIT ? ((lane & ~7) | ((e & 1) ? 4 + (e >> 1) : (e >> 1))) : lane;
    const int nw = blockDim.x >> 5;
    for (int b0 = warp; b0 < nblocks; b0 += 8 * nw) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int blk = b0 + u * nw;
            v[u] = blk < nblocks ? __ldg(x + (size_t)blk * 32 + lane) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int blk = b0 + u * nw;
            if (blk >= nblocks) break;  // warp-uniform
            const float amax = warp_max(fabsf(v[u]));
            const float d = __half2float(__float2half_rn(__fdiv_rn(amax, 127.0f)));
            const float q = (d == 0.0f) ? 0.0f : clamp127(roundf(__fdiv_rn(v[u], d)));
            int qi = (int)q;
            a.codes[(size_t)blk * 32 + pos] = (uint8_t)(qi & 0xff);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) qi += __shfl_xor_sync(FULL, qi, o);
            if (lane == 0) {
                a.isum[blk] = qi;
                a.dx[blk] = d;
            }
        }
    }
}

// ------------------------------------------------------------ chunk compute

// Q4_K chunk of nb_c super-blocks starting at super-block sb0 of the row.
// Lane = sub-block j = lane & 7 of super-block 4t + (lane >> 3).
// The high nibbles are used in place (bytes 16 q, unsigned) and the second
// dp4a chain's sum divided by 16 -- exact, every term is a multiple of 16.
// sums (diagnostic) points at [b = 0][row][sb = 0][0] with stride bstride
// between vectors.
template <int NB, bool SUMS>
__device__ __forceinline__ void chunk_q4_k(const uint8_t *ch, int nb_c, int sb0, int nsb,
                                           const Act &a, int nvec, float (&acc)[NB],
                                           int32_t *sums, size_t bstride, int lane) {
    const int j = lane & 7, sbl = lane >> 3;
    // bit offsets of this lane's 6-bit scale / min inside header words 1..3
    const int sh_sc = (6 * j) & 31, sh_m = (48 + 6 * j) & 31;
    const bool sc_hi = j >= 6, m_hi = j >= 3;
#pragma unroll
    for (int t = 0; t < Fmt<GQ_Q4_K>::CH / 4; ++t) {
        if (4 * t >= nb_c) break;  // warp-uniform
        const int sl = 4 * t + sbl;
        if (sl < nb_c) {
            const uint4 h = *reinterpret_cast<const uint4 *>(ch + sl * Q4_K_BYTES);
            const uint4 q = *reinterpret_cast<const uint4 *>(ch + sl * Q4_K_BYTES + 16 + 16 * j);
            const uint32_t lo0 = q.x & NIB, hi0 = q.x & ~NIB, lo1 = q.y & NIB, hi1 = q.y & ~NIB;
            const uint32_t lo2 = q.z & NIB, hi2 = q.z & ~NIB, lo3 = q.w & NIB, hi3 = q.w & ~NIB;
            const int sc = (int)(__funnelshift_r(sc_hi ? h.z : h.y, sc_hi ? h.w : h.z, sh_sc) & 63u);
            const int m = (int)(__funnelshift_r(m_hi ? h.w : h.z, m_hi ? 0u : h.w, sh_m) & 63u);
            const float d = half_bits_to_float(h.x), dmin = half_bits_to_float(h.x >> 16);
            const int sb = sb0 + sl;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= nvec) break;
                const int blk = b * nsb + sb;
                const int4 *ap = reinterpret_cast<const int4 *>(a.codes + (size_t)blk * 256 + 32 * j);
                const int4 a0 = ap[0], a1 = ap[1];
                int sl_ = dp4a_us(lo0, a0.x, 0), sh_ = dp4a_us(hi0, a0.y, 0);
                sl_ = dp4a_us(lo1, a0.z, sl_);
                sh_ = dp4a_us(hi1, a0.w, sh_);
                sl_ = dp4a_us(lo2, a1.x, sl_);
                sh_ = dp4a_us(hi2, a1.y, sh_);
                sl_ = dp4a_us(lo3, a1.z, sl_);
                sh_ = dp4a_us(hi3, a1.w, sh_);
                const int s = sl_ + (sh_ >> 4);
                int is1 = sc * s, is2 = m * a.isum[blk * 8 + j];
                if (SUMS) {
                    const int cnt = min(4, nb_c - 4 * t);  // super-blocks present in this step
                    const unsigned gmask = FULL >> (32 - 8 * cnt);
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) {
                        is1 += __shfl_xor_sync(gmask, is1, o);
                        is2 += __shfl_xor_sync(gmask, is2, o);
                    }
                    if (j == 0) {
                        int32_t *o = sums + b * bstride + (size_t)sb * 2;
                        o[0] = is1;
                        o[1] = is2;
                    }
                } else {
                    acc[b] += a.dx[blk] * (d * (float)is1 - dmin * (float)is2);
                }
            }
        }
    }
}

// Q4_0 / Q8_0 chunk of nb_c blocks starting at block blk0 of the row; lane k
// takes blocks k, k + 32, ...  A block starting `off` bytes into the chunk is
// read as aligned words from off & ~3; its code bytes begin 2 or 4 bytes into
// the first word, so funnel shifts by 16 or 32 (clamped) realign them.
template <int WT, int NB, bool SUMS>
__device__ __forceinline__ void chunk_q_0(const uint8_t *ch, int nb_c, int blk0, int nblk,
                                          const Act &a, int nvec, float (&acc)[NB],
                                          int32_t *sums, size_t bstride, int lane) {
    constexpr bool Q4 = WT == GQ_Q4_0;
    constexpr int BB = Fmt<WT>::BB;
    constexpr int PER = Fmt<WT>::CH / 32;
#pragma unroll
    for (int hh = 0; hh < PER; ++hh) {
        const int k = lane + 32 * hh;
        if (k >= nb_c) break;
        const int off = k * BB;
        const uint32_t *w = reinterpret_cast<const uint32_t *>(ch + (off & ~3));
        const uint32_t sh = (off & 2) ? 32u : 16u;
        constexpr int NW = Q4 ? 5 : 9;
        uint32_t v[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) v[i] = w[i];
        const float dw = half_bits_to_float((off & 2) ? (v[0] >> 16) : v[0]);
        int wl[8];  // dp4a operands in activation-layout order
        if (Q4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t c = __funnelshift_rc(v[i], v[i + 1], sh);
                wl[2 * i] = (int)(c & NIB);
                wl[2 * i + 1] = (int)((c >> 4) & NIB);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) wl[i] = (int)__funnelshift_rc(v[i], v[i + 1], sh);
        }
        const int blk = blk0 + k;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= nvec) break;
            const int ab = b * nblk + blk;
            const int4 *ap = reinterpret_cast<const int4 *>(a.codes + (size_t)ab * 32);
            const int4 a0 = ap[0], a1 = ap[1];
            int s = dp4a(wl[0], a0.x, 0);
            s = dp4a(wl[1], a0.y, s);
            s = dp4a(wl[2], a0.z, s);
            s = dp4a(wl[3], a0.w, s);
            s = dp4a(wl[4], a1.x, s);
            s = dp4a(wl[5], a1.y, s);
            s = dp4a(wl[6], a1.z, s);
            s = dp4a(wl[7], a1.w, s);
            if (Q4) s -= 8 * a.isum[ab];
            if (SUMS)
                sums[b * bstride + blk] = s;
            else
                acc[b] += dw * a.dx[ab] * (float)s;
        }
    }
}

// ------------------------------------------------------------- the kernel

// One launch covers NB activation vectors (blockIdx.y selects the chunk of
// vectors) and all rows.  FUSED: `act` is fp32 [batch][cols] and is
// quantized in the CTA; otherwise `act` holds the quantized blocks.
// w_static != 0 lets the first weight chunks be requested before the
// dependency wait on the preceding kernel (the caller guarantees no kernel
// still in flight writes W).
template <int WT, int NB, bool SUMS, bool FUSED, int NW>
__global__ void __launch_bounds__(NW * 32) gemv_kernel(const uint8_t *__restrict__ W,
                                                   const void *__restrict__ act_in,
                                                   float *__restrict__ y,
                                                   int32_t *__restrict__ sums, int rows,
                                                   int nblk, int batch, int w_static,
                                                   uint32_t *__restrict__ status) {
    using F = Fmt<WT>;
    using R = Ring<WT, NW>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b0 = blockIdx.y * NB;
    const int nvec = min(NB, batch - b0);
    const int warps_total = gridDim.x * NW;
    const int wg = blockIdx.x * NW + warp;
    const int nrows_w = wg < rows ? (rows - 1 - wg) / warps_total + 1 : 0;
    const int nchunk = (nblk + F::CH - 1) / F::CH;
    const int total = nrows_w * nchunk;
    const size_t row_bytes = (size_t)nblk * F::BB;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem) + warp * NSTAGE;
    uint8_t *ring = smem + R::BUFS_OFF + warp * NSTAGE * R::BUF;

    // item i of this warp = chunk (i % nchunk) of its (i / nchunk)-th row
    auto issue = [&](int i) {
        const int row = wg + (i / nchunk) * warps_total;
        const int c = i % nchunk;
        const int nb_c = min(F::CH, nblk - c * F::CH);
        const uint32_t bytes = (uint32_t)(nb_c * F::BB);
        const int st = i % NSTAGE;
        mbar_arrive_expect_tx(bar + st, bytes);
        bulk_g2s(ring + st * R::BUF, W + row * row_bytes + (size_t)c * F::CH * F::BB, bytes, bar + st);
    };

    // With the early trigger the next kernel in the stream may launch right
    // away (its CTAs wait on griddepcontrol.wait before touching anything this
    // kernel produces); otherwise it launches once this kernel's activations
    // are staged.
    if (GQ_GEMV_EARLY_TRIGGER) pdl_launch_dependents();
    if (lane == 0 && total > 0) {
#pragma unroll
        for (int s = 0; s < NSTAGE; ++s) mbar_init(bar + s, 1);
        fence_mbar_init();
        if (w_static)
            for (int i = 0; i < NSTAGE && i < total; ++i) issue(i);
    }
    pdl_wait();  // activations (and, unless static, W) may come from the preceding kernel
    if (lane == 0 && !w_static)
        for (int i = 0; i < NSTAGE && i < total; ++i) issue(i);

    const Act a = act_layout<WT>(smem + R::ACT_OFF, NB, nblk);
    const int nact = nvec * nblk;
    if (FUSED) {
        const float *x = static_cast<const float *>(act_in) + (size_t)b0 * nblk * F::BE;
        if (WT == GQ_Q4_K)
            quant_stage_q8_k(a, x, nact);
        else
            quant_stage_q8_0<WT == GQ_Q4_0>(a, x, nact);
    } else {
        const uint8_t *xq = static_cast<const uint8_t *>(act_in);
        if (WT == GQ_Q4_K)
            stage_q8_k(a, xq + (size_t)b0 * nblk * Q8_K_BYTES, nact);
        else
            stage_q8_0<WT == GQ_Q4_0>(a, xq + (size_t)b0 * nblk * Q8_0_BYTES, nact);
    }
    __syncthreads();
    if (!GQ_GEMV_EARLY_TRIGGER) pdl_launch_dependents();

    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    const size_t bstride = (size_t)rows * nblk * (WT == GQ_Q4_K ? 2 : 1);

    for (int i = 0; i < total; ++i) {
        const int st = i % NSTAGE;
        if (!mbar_wait_bounded(bar + st, (uint32_t)(i / NSTAGE) & 1u)) {
            // A transfer never completed: flag it, let the other issued
            // stages drain (bounded), and leave the remaining rows unwritten.
            if (lane == 0) atomicOr(status, STATUS_GEMV_TMA_TIMEOUT);
            for (int k = i + 1; k < total && k < i + NSTAGE; ++k)
                mbar_wait_bounded(bar + k % NSTAGE, (uint32_t)(k / NSTAGE) & 1u);
            return;
        }
        const int row = wg + (i / nchunk) * warps_total;
        const int c = i % nchunk;
        const int nb_c = min(F::CH, nblk - c * F::CH);
        const uint8_t *ch = ring + st * R::BUF;
        int32_t *srow = SUMS ? sums + ((size_t)b0 * rows + row) * nblk * (WT == GQ_Q4_K ? 2 : 1) : nullptr;
        if (WT == GQ_Q4_K)
            chunk_q4_k<NB, SUMS>(ch, nb_c, c * F::CH, nblk, a, nvec, acc, srow, bstride, lane);
        else
            chunk_q_0<WT, NB, SUMS>(ch, nb_c, c * F::CH, nblk, a, nvec, acc, srow, bstride, lane);
        __syncwarp();
        if (lane == 0 && i + NSTAGE < total) issue(i + NSTAGE);
        if (!SUMS && c == nchunk - 1) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < nvec) {
                    const float v = warp_sum(acc[b]);
                    if (lane == 0) y[(size_t)(b0 + b) * rows + row] = v;
                }
                acc[b] = 0.0f;
            }
        }
    }
}

// Plain per-block kernel for Q4_0 / Q8_0 rows whose byte length is not a
// multiple of 16 (cols % 256 != 0): warp per row, lane per block, 16-bit
// global loads, activations read from global memory.
template <bool Q4, bool SUMS>
__global__ void __launch_bounds__(256) gemv_plain_kernel(const uint8_t *__restrict__ W,
                                                         const uint8_t *__restrict__ xq,
                                                         float *__restrict__ y,
                                                         int32_t *__restrict__ sums, int rows,
                                                         int nblk, int batch) {
    constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * WARPS + warp;
    const int b = blockIdx.y;
    pdl_launch_dependents();
    pdl_wait();
    if (row >= rows || b >= batch) return;
    float acc = 0.0f;
    for (int blk = lane; blk < nblk; blk += 32) {
        const uint16_t *wb = reinterpret_cast<const uint16_t *>(W + ((size_t)row * nblk + blk) * BB);
        const uint16_t *ab = reinterpret_cast<const uint16_t *>(xq + ((size_t)b * nblk + blk) * Q8_0_BYTES);
        int s = 0;
        if (Q4) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w2 = __ldg(wb + 1 + i);       // code bytes 2i, 2i+1
                const uint32_t a01 = __ldg(ab + 1 + 2 * i);  // activations 4i, 4i+1
                const uint32_t a23 = __ldg(ab + 2 + 2 * i);  // activations 4i+2, 4i+3
                const int c0 = (int)(w2 & 15) - 8, c1 = (int)((w2 >> 4) & 15) - 8;
                const int c2 = (int)((w2 >> 8) & 15) - 8, c3 = (int)((w2 >> 12) & 15) - 8;
                s += c0 * (int)(int8_t)(a01 & 0xff) + c1 * (int)(int8_t)(a01 >> 8) +
                     c2 * (int)(int8_t)(a23 & 0xff) + c3 * (int)(int8_t)(a23 >> 8);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t w2 = __ldg(wb + 1 + i), a2 = __ldg(ab + 1 + i);
                s += (int)(int8_t)(w2 & 0xff) * (int)(int8_t)(a2 & 0xff) +
                     (int)(int8_t)(w2 >> 8) * (int)(int8_t)(a2 >> 8);
            }
        }
        if (SUMS) {
            sums[((size_t)b * rows + row) * nblk + blk] = s;
        } else {
            const float dw = half_bits_to_float(__ldg(wb)), dx = half_bits_to_float(__ldg(ab));
            acc += dw * dx * (float)s;
        }
    }
    if (!SUMS) {
        acc = warp_sum(acc);
        if (lane == 0) y[(size_t)b * rows + row] = acc;
    }
}

// ------------------------------------------------------------------ launch

constexpr int SMEM_MAX = 232448;  // opt-in shared memory per CTA on sm_103
constexpr int ROWS_PER_WARP = GQ_GEMV_ROWS_PER_WARP;  // target rows per warp before the grid caps
constexpr int CTAS_PER_SM = GQ_GEMV_CTAS_PER_SM;

template <int WT, int NW = WARPS>
size_t smem_bytes(int nb, int nblk) {
    return (size_t)Ring<WT, NW>::ACT_OFF + (size_t)nb * nblk * act_block_bytes<WT>();
}

template <int WT, int NB, bool SUMS, bool FUSED, int NW>
cudaError_t launch_one(const void *W, const void *act, float *y, int32_t *sums, int rows,
                       int nblk, int batch, int w_static, int rows_per_warp, const LaunchCtx &ctx) {
    auto k = gemv_kernel<WT, NB, SUMS, FUSED, NW>;
    const size_t smem = smem_bytes<WT, NW>(NB, nblk);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        if (e != cudaSuccess) return e;
    }
    const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(CTAS_PER_SM, SMEM_MAX / (smem + 1024)));
    int grid = (rows + NW * rows_per_warp - 1) / (NW * rows_per_warp);
    grid = std::max(1, std::min(grid, ctx.num_sms * per_sm));
    dim3 g(grid, (batch + NB - 1) / NB);
    return launch_pdl(k, g, dim3(NW * 32), smem, ctx.stream, static_cast<const uint8_t *>(W), act,
                      y, sums, rows, nblk, batch, w_static, ctx.status);
}

// Largest batch chunk in {8, 4, 2, 1} not above `batch` whose staged
// activations fit in shared memory; 0 if none fits.
template <int WT>
int pick_nb(int batch, int nblk) {
    for (int nb = 8; nb >= 1; nb >>= 1)
        if (nb <= std::max(batch, 1) && smem_bytes<WT>(nb, nblk) <= (size_t)SMEM_MAX) return nb;
    return 0;
}

template <int WT, bool SUMS, bool FUSED>
cudaError_t dispatch_wt(const void *W, const void *act, float *y, int32_t *sums, int rows,
                        int nblk, int batch, int w_static, const LaunchCtx &ctx) {
    const int nb = pick_nb<WT>(batch, nblk);
    const int rpw = ROWS_PER_WARP;
    switch (nb) {
    case 8: return launch_one<WT, 8, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, rpw, ctx);
    case 4: return launch_one<WT, 4, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, rpw, ctx);
    case 2: return launch_one<WT, 2, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, rpw, ctx);
    case 1: return launch_one<WT, 1, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, rpw, ctx);
    }
    return cudaErrorInvalidValue;
}

template <bool SUMS, bool FUSED>
cudaError_t dispatch(gq_type wtype, const void *W, const void *act, float *y, int32_t *sums,
                     int rows, int cols, int batch, int w_static, const LaunchCtx &ctx) {
    if (wtype == GQ_Q4_K)
        return dispatch_wt<GQ_Q4_K, SUMS, FUSED>(W, act, y, sums, rows, cols / QK_K, batch, w_static, ctx);
    const int nblk = cols / 32;
    if (cols % 256 != 0) {
        if (FUSED) return cudaErrorInvalidValue;
        dim3 grid((rows + WARPS - 1) / WARPS, batch);
        const uint8_t *w8 = static_cast<const uint8_t *>(W);
        const uint8_t *a8 = static_cast<const uint8_t *>(act);
        if (wtype == GQ_Q4_0)
            return launch_pdl(gemv_plain_kernel<true, SUMS>, grid, dim3(256), 0, ctx.stream, w8, a8,
                              y, sums, rows, nblk, batch);
        return launch_pdl(gemv_plain_kernel<false, SUMS>, grid, dim3(256), 0, ctx.stream, w8, a8, y,
                          sums, rows, nblk, batch);
    }
    if (wtype == GQ_Q4_0)
        return dispatch_wt<GQ_Q4_0, SUMS, FUSED>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
    return dispatch_wt<GQ_Q8_0, SUMS, FUSED>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
}

}  // namespace

bool gemv_fits(gq_type wtype, int64_t cols) {
    if (wtype == GQ_Q4_K) return pick_nb<GQ_Q4_K>(1, (int)(cols / QK_K)) > 0;
    if (cols % 256 != 0) return true;
    if (wtype == GQ_Q4_0) return pick_nb<GQ_Q4_0>(1, (int)(cols / 32)) > 0;
    return pick_nb<GQ_Q8_0>(1, (int)(cols / 32)) > 0;
}

cudaError_t launch_gemv(gq_type wtype, const void *W, const void *act, float *y, int32_t *sums,
                        int64_t rows, int64_t cols, int64_t batch, bool fused_f32, bool w_static,
                        const LaunchCtx &ctx) {
    const int ws = w_static ? 1 : 0;
    if (fused_f32)
        return sums ? dispatch<true, true>(wtype, W, act, y, sums, (int)rows, (int)cols, (int)batch, ws, ctx)
                    : dispatch<false, true>(wtype, W, act, y, sums, (int)rows, (int)cols, (int)batch, ws, ctx);
    return sums ? dispatch<true, false>(wtype, W, act, y, sums, (int)rows, (int)cols, (int)batch, ws, ctx)
                : dispatch<false, false>(wtype, W, act, y, sums, (int)rows, (int)cols, (int)batch, ws, ctx);
}

}  // namespace gq
