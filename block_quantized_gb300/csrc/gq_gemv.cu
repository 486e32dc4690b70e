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
//   - a persistent grid of at most one CTA per SM; every warp owns whole row
//     groups (grid-stride) and streams them through its own shared-memory
//     ring, filled by the TMA engine (cp.async.bulk with an evict-first L2
//     policy, completion on an mbarrier, every wait bounded).  A ring item
//     is R whole rows in one bulk copy (R <= 4; 9.2 KB for four 4096-column
//     rows) when two such items per warp fit the ring budget, else one
//     16-super-block chunk of one row.  The ring depth is chosen per launch
//     (a tall matrix keeps ~150 KB per SM in flight); the first stage is
//     requested before the dependency wait, the rest once the activations
//     are staged;
//   - the CTA's activation vectors are staged once in shared memory, each
//     group of 8 int8 codes stored as (a0,a2,a4,a6 | a1,a3,a5,a7) so a
//     packed nibble word w feeds dp4a as (w & 0x0F0F0F0F) and
//     (w & 0xF0F0F0F0) (high nibbles in place, sum divided by 16); the
//     fused variants quantize fp32 activations straight into that layout
//     (same arithmetic as the standalone quantizer, so the codes are
//     identical);
//   - Q4_K: a lane takes half a super-block (four sub-blocks), so one warp
//     instruction covers a 16-super-block row chunk; at batch 1 the lane's
//     activation slice stays in registers and the rows of an item are
//     interleaved, with one transposed butterfly reducing all of them;
//   - Q4_0 / Q8_0 blocks (18 / 34 bytes, 2-byte aligned) are read from the
//     ring with aligned 32-bit loads and funnel shifts;
//   - per-lane fp32 partial sums, warp-shuffle reductions per row.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_quant8.cuh"

namespace gq {
namespace {

using namespace q8;

constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr unsigned FULL = 0xffffffffu;
// Launch-shape parameters (compile-time; the defaults are the measured best).
#ifndef GQ_GEMV_CTAS_PER_SM
#define GQ_GEMV_CTAS_PER_SM 1
#endif
#ifndef GQ_GEMV_RING_BUDGET
#define GQ_GEMV_RING_BUDGET (150 * 1024)
#endif
#ifndef GQ_GEMV_EARLY_TRIGGER
#define GQ_GEMV_EARLY_TRIGGER 1
#endif
#ifndef GQ_GEMV_WARPS
#define GQ_GEMV_WARPS 8
#endif
#ifndef GQ_GEMV_MAX_R
#define GQ_GEMV_MAX_R 4
#endif
#ifndef GQ_GEMV_MIN_BLOCKS
#define GQ_GEMV_MIN_BLOCKS 1
#endif
// Weight copies carry an evict-first L2 policy (the weights are streamed
// once per pass; activations and outputs are what later launches reuse).
#ifndef GQ_GEMV_W_EVICT_FIRST
#define GQ_GEMV_W_EVICT_FIRST 1
#endif
// R rows per item need at least warps / GQ_GEMV_R_SPREAD items: on a
// 4096-row matrix, four-row items (one 9.2 KB copy per warp, some warps idle)
// beat two-row items (two copies on most warps), since a warp completes only
// about one bulk copy per 0.6 us.
#ifndef GQ_GEMV_R_SPREAD
#define GQ_GEMV_R_SPREAD 2
#endif
#ifndef GQ_GEMV_PREFETCH
#define GQ_GEMV_PREFETCH 1
#endif

constexpr int WARPS = GQ_GEMV_WARPS;      // warps per CTA

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
    // 2304-byte chunks: one super-block per lane pair
    static constexpr int BB = Q4_K_BYTES, BE = 256, CH = 16;
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

// Q8_K: codes, then the sub-block sums (16-byte aligned for vector loads),
// then the scales.  Q8_0: codes, scales, sums.
template <int WT>
__device__ __forceinline__ Act act_layout(uint8_t *base, int nb, int nblk) {
    Act a;
    a.codes = base;
    if (WT == GQ_Q4_K) {
        a.isum = reinterpret_cast<int32_t *>(base + (size_t)nb * nblk * 256);
        a.dx = reinterpret_cast<float *>(a.isum + (size_t)nb * nblk * 8);
    } else {
        a.dx = reinterpret_cast<float *>(base + (size_t)nb * nblk * 32);
        a.isum = reinterpret_cast<int32_t *>(a.dx + (size_t)nb * nblk);
    }
    return a;
}

// Q8_K codes of one super-block are kept as 16 units of 16 bytes.  Half h
// (sub-blocks 4h..4h+3) owns units 8h..8h+7; its logical unit k' holds code
// groups 2k' and 2k'+1 of that half (each group = 8 codes in the split order
// of split8), and is stored at unit 8h + (k' ^ ((2 sb + h) & 7)) so that the
// eight lanes of a quarter-warp, which read the same k' of consecutive
// half-super-blocks, hit eight different bank quads.  sb is the super-block's
// index within its vector; g is the code group (0..31) within the super-block.
__device__ __forceinline__ int q8k_group_off(int sb, int g) {
    const int j = g >> 2, i = g & 3, h = j >> 2;
    const int kp = 2 * (j & 3) + (i >> 1);
    return 128 * h + 16 * (kp ^ ((2 * sb + h) & 7)) + 8 * (i & 1);
}

__device__ __forceinline__ uint2 split8(uint32_t a0, uint32_t a1) {
    return make_uint2(__byte_perm(a0, a1, 0x6420), __byte_perm(a0, a1, 0x7531));
}

// ---- unfused staging: copy quantized activation blocks into the layout.
// All loads of a pass are issued before any store, so a pass costs one
// L2 round trip.

constexpr int SG_BATCH = 6;  // code groups per thread per pass

__device__ void stage_q8_k(const Act &a, const uint8_t *__restrict__ xq, int nblocks, int nsb) {
    const int groups = nblocks * 32;
    // pass p copies groups [SG_BATCH*p*T, SG_BATCH*(p+1)*T) and block headers
    // [p*T, (p+1)*T) (T = blockDim.x); there are at least as many group
    // passes as header passes since every block has 32 groups.
    int pass = 0;
    for (int base = 0; base < groups; base += SG_BATCH * blockDim.x, ++pass) {
        uint32_t w0[SG_BATCH], w1[SG_BATCH], hd[5];
        const int hb = pass * blockDim.x + threadIdx.x;
        const bool has_h = hb < nblocks;
        if (has_h) {
            const uint8_t *src = xq + (size_t)hb * Q8_K_BYTES;
            hd[0] = __ldg(reinterpret_cast<const uint32_t *>(src));
#pragma unroll
            for (int i = 0; i < 4; ++i) hd[1 + i] = __ldg(reinterpret_cast<const uint32_t *>(src + 260) + i);
        }
#pragma unroll
        for (int u = 0; u < SG_BATCH; ++u) {
            const int g = base + u * blockDim.x + threadIdx.x;
            if (g < groups) {
                const uint32_t *src = reinterpret_cast<const uint32_t *>(
                    xq + (size_t)(g >> 5) * Q8_K_BYTES + 4 + 8 * (g & 31));
                w0[u] = __ldg(src);
                w1[u] = __ldg(src + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < SG_BATCH; ++u) {
            const int g = base + u * blockDim.x + threadIdx.x;
            if (g < groups) {
                const int blk = g >> 5;
                *reinterpret_cast<uint2 *>(a.codes + (size_t)blk * 256 + q8k_group_off(blk % nsb, g & 31)) =
                    split8(w0[u], w1[u]);
            }
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



// Q8_K: one warp per 256-element block, lane l owns elements 8l..8l+7
// (= code group l of the layout).
// Each warp loads up to QS_BATCH of its blocks before quantizing any, so a
// row of up to QS_BATCH * warps blocks costs one L2 round trip, and then
// quantizes them two at a time with the two dependency chains interleaved.
constexpr int QS_BATCH = 6;
static_assert(QS_BATCH % 2 == 0, "blocks are quantized in pairs");

__device__ void quant_stage_q8_k(const Act &a, const float *__restrict__ x, int nblocks, int nsb) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int b0 = warp; b0 < nblocks; b0 += QS_BATCH * nw) {
        float4 v[QS_BATCH][2];
#pragma unroll
        for (int u = 0; u < QS_BATCH; ++u) {
            const int blk = b0 + u * nw;
            if (blk < nblocks) {
                const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)blk * QK_K + 8 * lane);
                v[u][0] = __ldg(p);
                v[u][1] = __ldg(p + 1);
            } else {
                v[u][0] = v[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int u = 0; u < QS_BATCH; u += 2) {
            if (b0 + u * nw >= nblocks) break;  // warp-uniform
            float e[2][8], am[2], d[2], r[2];
            uint32_t w0[2], w1[2];
            int sum[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                unpack8(v[u + k], e[k]);
                am[k] = absmax8(e[k]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int k = 0; k < 2; ++k) am[k] = fmaxf(am[k], __shfl_xor_sync(FULL, am[k], o));
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                d[k] = __fdiv_rn(am[k], 127.0f);
                r[k] = __frcp_rn(d[k]);
                q8_codes8(e[k], d[k], r[k], w0[k], w1[k]);
                sum[k] = dp4a((int)w0[k], 0x01010101, dp4a((int)w1[k], 0x01010101, 0));
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
                for (int k = 0; k < 2; ++k) sum[k] += __shfl_xor_sync(FULL, sum[k], o);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int blk = b0 + (u + k) * nw;
                if (blk < nblocks) {
                    *reinterpret_cast<uint2 *>(a.codes + (size_t)blk * 256 + q8k_group_off(blk % nsb, lane)) =
                        split8(w0[k], w1[k]);
                    if ((lane & 3) == 0) a.isum[blk * 8 + (lane >> 2)] = sum[k];
                    if (lane == 0) a.dx[blk] = d[k];
                }
            }
        }
    }
}

// Q8_0: a warp pass covers eight consecutive 32-element blocks, four lanes
// per block and eight elements per lane (two 16-byte loads, 1 KB per warp,
// coalesced).  Passes are batched and quantized in interleaved pairs as for
// Q8_K.
template <bool SPLIT>
__device__ void quant_stage_q8_0(const Act &a, const float *__restrict__ x, int nblocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int sub = lane & 3;  // eight-element group within the block
    const int npass = (nblocks + 7) / 8;
    for (int p0 = warp; p0 < npass; p0 += QS_BATCH * nw) {
        float4 v[QS_BATCH][2];
#pragma unroll
        for (int u = 0; u < QS_BATCH; ++u) {
            const int blk = (p0 + u * nw) * 8 + (lane >> 2);
            if (blk < nblocks) {
                const float4 *p = reinterpret_cast<const float4 *>(x + (size_t)blk * 32 + 8 * sub);
                v[u][0] = __ldg(p);
                v[u][1] = __ldg(p + 1);
            } else {
                v[u][0] = v[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
#pragma unroll
        for (int u = 0; u < QS_BATCH; u += 2) {
            if (p0 + u * nw >= npass) break;  // warp-uniform
            float e[2][8], am[2], d[2], r[2];
            uint32_t w0[2], w1[2];
            int sum[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                unpack8(v[u + k], e[k]);
                am[k] = absmax8(e[k]);
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
                for (int k = 0; k < 2; ++k) am[k] = fmaxf(am[k], __shfl_xor_sync(FULL, am[k], o));
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                d[k] = __half2float(__float2half_rn(__fdiv_rn(am[k], 127.0f)));
                r[k] = __frcp_rn(d[k]);
                q8_codes8(e[k], d[k], r[k], w0[k], w1[k]);
                sum[k] = dp4a((int)w0[k], 0x01010101, dp4a((int)w1[k], 0x01010101, 0));
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1)
#pragma unroll
                for (int k = 0; k < 2; ++k) sum[k] += __shfl_xor_sync(FULL, sum[k], o);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int blk = (p0 + (u + k) * nw) * 8 + (lane >> 2);
                if (blk < nblocks) {
                    *reinterpret_cast<uint2 *>(a.codes + (size_t)blk * 32 + 8 * sub) =
                        SPLIT ? split8(w0[k], w1[k]) : make_uint2(w0[k], w1[k]);
                    if (sub == 0) {
                        a.isum[blk] = sum[k];
                        a.dx[blk] = d[k];
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------ chunk compute

// Q4_K chunk: nb_c (<= 16) super-blocks of one row, starting at super-block
// sb0.  Lane l takes half h = l & 1 (sub-blocks 4h..4h+3) of super-block
// l >> 1, so one warp instruction covers the whole chunk: per lane four
// 16-byte nibble loads, one (pair-shared) header load, 32 dp4a, and one
// float update for the pair of integer sums
//   S1 = sum_j sc_j * s_j,   S2 = sum_j m_j * t_j   (j over the half)
// with s_j the sub-block integer dot and t_j the Q8_K sub-block sum.  The
// high nibbles are used in place (values 16 q, unsigned) and that dp4a
// chain's sum is divided by 16 -- exact, every term is a multiple of 16.
// The lane's activation slice (8 units of 16 codes, the four t_j and the
// vector scale) lives in registers: loaded once per kernel when the row has
// a single chunk and NB == 1, else reloaded per chunk and vector.
struct Q4KAct {
    uint4 u[8];
    int4 t;
    float dx;
};

__device__ __forceinline__ void load_q4k_act(Q4KAct &r, const Act &a, int blk, int h, int sw) {
    const uint4 *u = reinterpret_cast<const uint4 *>(a.codes + (size_t)blk * 256 + 128 * h);
#pragma unroll
    for (int k = 0; k < 8; ++k) r.u[k] = u[k ^ sw];
    r.t = reinterpret_cast<const int4 *>(a.isum + (size_t)blk * 8)[h];
    r.dx = a.dx[blk];
}

__device__ __forceinline__ void dot_q4k_half(const uint4 (&q)[4], const Q4KAct &r, uint32_t sc24,
                                             uint32_t m24, int &S1, int &S2) {
    const int t[4] = {r.t.x, r.t.y, r.t.z, r.t.w};
    S1 = 0;
    S2 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 w = q[k], a0 = r.u[2 * k], a1 = r.u[2 * k + 1];
        int sl = dp4a_us(w.x & NIB, (int)a0.x, 0), sh = dp4a_us(w.x & ~NIB, (int)a0.y, 0);
        sl = dp4a_us(w.y & NIB, (int)a0.z, sl);
        sh = dp4a_us(w.y & ~NIB, (int)a0.w, sh);
        sl = dp4a_us(w.z & NIB, (int)a1.x, sl);
        sh = dp4a_us(w.z & ~NIB, (int)a1.y, sh);
        sl = dp4a_us(w.w & NIB, (int)a1.z, sl);
        sh = dp4a_us(w.w & ~NIB, (int)a1.w, sh);
        const int s = sl + (sh >> 4);
        S1 += (int)((sc24 >> (6 * k)) & 63u) * s;
        S2 += (int)((m24 >> (6 * k)) & 63u) * t[k];
    }
}

// sums (diagnostic) points at [b = 0][row][sb = 0][0] with stride bstride
// between vectors.  act_resident: `reg` already holds this lane's slice.
template <int NB, bool SUMS>
__device__ __forceinline__ void chunk_q4_k(const uint8_t *ch, int nb_c, int sb0, int nsb,
                                           const Act &a, int nvec, float (&acc)[NB], Q4KAct &reg,
                                           bool act_resident, int32_t *sums, size_t bstride,
                                           int lane) {
    const int h = lane & 1, sbl = lane >> 1;
    const bool active = sbl < nb_c;
    const uint8_t *p = ch + sbl * Q4_K_BYTES;
    uint4 hd = make_uint4(0, 0, 0, 0), q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) q[k] = make_uint4(0, 0, 0, 0);
    if (active) {
        hd = *reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = *reinterpret_cast<const uint4 *>(p + 16 + 64 * h + 16 * k);
    }
    // header bytes 4..15 = words y, z, w: the 6-bit fields sc_0..sc_7 then
    // m_0..m_7, LSB first.  This half's four sc (bits 24h..24h+23) and four m
    // (bits 48+24h..71+24h) are three whole bytes each.
    const uint32_t sc24 = __byte_perm(hd.y, hd.z, h ? 0x0543u : 0x0210u);
    const uint32_t m24 = __byte_perm(hd.z, hd.w, h ? 0x0765u : 0x0432u);
    const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
    const int sb = sb0 + sbl;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b >= nvec) break;  // warp-uniform
        const int blk = b * nsb + sb;
        if (!act_resident && active) load_q4k_act(reg, a, blk, h, lane & 7);
        int S1 = 0, S2 = 0;
        if (active) dot_q4k_half(q, reg, sc24, m24, S1, S2);
        if (SUMS) {
            S1 += __shfl_xor_sync(FULL, S1, 1);
            S2 += __shfl_xor_sync(FULL, S2, 1);
            if (active && h == 0) {
                int32_t *o = sums + b * bstride + (size_t)sb * 2;
                o[0] = S1;
                o[1] = S2;
            }
        } else if (active) {
            acc[b] += reg.dx * (d * (float)S1 - dmin * (float)S2);
        }
    }
}

// Batch-1 Q4_K fast path for an item of nr <= RR whole rows (row = one
// chunk): the rows' loads and dp4a chains are interleaved, and the RR row
// sums are reduced across the warp in a transposed butterfly -- each level
// halves the rows a lane keeps -- so four rows cost six shuffles instead of
// twenty.  Afterwards lane l holds the sum of row 2 * bit4(l) + bit3(l) (for
// RR == 4; row bit4(l) for RR == 2; row 0 for RR == 1).
template <int RR>
__device__ __forceinline__ float rows_q4_k_nb1(const uint8_t *ch, size_t row_bytes, int nr, int nblk,
                                               const Q4KAct &reg, int lane) {
    const int h = lane & 1, sbl = lane >> 1;
    const bool active = sbl < nblk;
    const uint32_t sel_sc = h ? 0x0543u : 0x0210u, sel_m = h ? 0x0765u : 0x0432u;
    uint4 hd[RR], q[RR][4];
#pragma unroll
    for (int r = 0; r < RR; ++r) {
        hd[r] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < 4; ++k) q[r][k] = make_uint4(0, 0, 0, 0);
        if (active && r < nr) {
            const uint8_t *p = ch + r * row_bytes + sbl * Q4_K_BYTES;
            hd[r] = *reinterpret_cast<const uint4 *>(p);
#pragma unroll
            for (int k = 0; k < 4; ++k) q[r][k] = *reinterpret_cast<const uint4 *>(p + 16 + 64 * h + 16 * k);
        }
    }
    float v[RR];
#pragma unroll
    for (int r = 0; r < RR; ++r) {
        int S1, S2;
        dot_q4k_half(q[r], reg, __byte_perm(hd[r].y, hd[r].z, sel_sc), __byte_perm(hd[r].z, hd[r].w, sel_m), S1,
                     S2);
        const float d = half_bits_to_float(hd[r].x), dmin = half_bits_to_float(hd[r].x >> 16);
        v[r] = active ? reg.dx * (d * (float)S1 - dmin * (float)S2) : 0.0f;
    }
    float s;
    if (RR == 4) {
        const bool up = lane & 16;
        const float x0 = __shfl_xor_sync(FULL, up ? v[0] : v[2], 16);
        const float x1 = __shfl_xor_sync(FULL, up ? v[1] : v[3], 16);
        const float k0 = (up ? v[2] : v[0]) + x0, k1 = (up ? v[3] : v[1]) + x1;
        const bool up8 = lane & 8;
        s = (up8 ? k1 : k0) + __shfl_xor_sync(FULL, up8 ? k0 : k1, 8);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    } else if (RR == 2) {
        const bool up = lane & 16;
        s = (up ? v[1] : v[0]) + __shfl_xor_sync(FULL, up ? v[0] : v[1], 16);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    } else {
        s = warp_sum(v[0]);
    }
    return s;
}

// Transposed butterfly over V = 2^k values per lane (V <= 32): each level
// halves the values a lane keeps, so the V warp sums cost V - 1 shuffles plus
// 5 - k for the rest of the butterfly.  Afterwards lane l holds the sum of
// value index sum_j bit(4 - j, l) << (k - 1 - j), j < k.
template <int V>
__device__ __forceinline__ float transpose_reduce(float (&v)[V], int lane) {
#pragma unroll
    for (int lvl = 0; (1 << lvl) < V; ++lvl) {
        const int n = V >> lvl, o = 16 >> lvl;
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float recv = __shfl_xor_sync(FULL, up ? v[i] : v[i + n / 2], o);
            v[i] = (up ? v[i + n / 2] : v[i]) + recv;
        }
    }
    constexpr int K = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
    float s = v[0];
#pragma unroll
    for (int o = 16 >> K; o > 0; o >>= 1) s += __shfl_xor_sync(FULL, s, o);
    return s;
}

__device__ __forceinline__ int transpose_index(int lane, int k) {
    int idx = 0;
    for (int j = 0; j < k; ++j) idx |= ((lane >> (4 - j)) & 1) << (k - 1 - j);
    return idx;
}

// Q4_K product of NB > 1 vectors with an item of nr <= MR whole rows: per
// chunk, the rows' nibbles and scales are loaded into registers once and each
// vector's activation slice once, so the shared-memory traffic per row and
// vector is the dot product's alone.  The MR x NB sums are reduced together
// and written by the lanes that hold them.
template <int NB, int MR>
__device__ __forceinline__ void item_q4k_multi(const uint8_t *ch, size_t row_bytes, int nr, int nblk, int nvec,
                                               const Act &a, float *__restrict__ y, int rows, int row0, int b0,
                                               int lane) {
    const int h = lane & 1, sbl = lane >> 1;
    const uint32_t sel_sc = h ? 0x0543u : 0x0210u, sel_m = h ? 0x0765u : 0x0432u;
    float v[MR * NB];
#pragma unroll
    for (int i = 0; i < MR * NB; ++i) v[i] = 0.0f;
    const int nchunk = (nblk + 15) / 16;
    for (int c = 0; c < nchunk; ++c) {
        const int sb = 16 * c + sbl;
        const bool active = sb < nblk;
        uint4 hd[MR], q[MR][4];
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            hd[r] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) q[r][k] = make_uint4(0, 0, 0, 0);
            if (active && r < nr) {
                const uint8_t *p = ch + r * row_bytes + (size_t)sb * Q4_K_BYTES;
                hd[r] = *reinterpret_cast<const uint4 *>(p);
#pragma unroll
                for (int k = 0; k < 4; ++k) q[r][k] = *reinterpret_cast<const uint4 *>(p + 16 + 64 * h + 16 * k);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b >= nvec) break;  // warp-uniform
            Q4KAct act;
            if (active) load_q4k_act(act, a, b * nblk + sb, h, lane & 7);
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                if (r >= nr) break;  // warp-uniform
                int S1 = 0, S2 = 0;
                if (active) {
                    dot_q4k_half(q[r], act, __byte_perm(hd[r].y, hd[r].z, sel_sc), __byte_perm(hd[r].z, hd[r].w, sel_m),
                                 S1, S2);
                    const float d = half_bits_to_float(hd[r].x), dmin = half_bits_to_float(hd[r].x >> 16);
                    v[r * NB + b] += act.dx * (d * (float)S1 - dmin * (float)S2);
                }
            }
        }
    }
    constexpr int V = MR * NB;
    constexpr int K = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : 1;
    const float s = transpose_reduce<V>(v, lane);
    const int idx = transpose_index(lane, K);
    const int r = idx / NB, b = idx % NB;
    if ((lane & ((1 << (5 - K)) - 1)) == 0 && r < nr && b < nvec) y[(size_t)(b0 + b) * rows + row0 + r] = s;
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

// Ring geometry, chosen per launch.  A ring item is R whole rows (one bulk
// copy of R * row_bytes contiguous bytes) when two stages of a row fit the
// ring budget, else one chunk of one row (R = 1).  A bulk copy costs about
// the same issue time whatever its size, so whole rows stream better than
// chunks.  Each warp owns `ns` stages of `stage_bytes`.
struct Geo {
    int R;            // rows per item (1, 2 or 4)
    int ns;           // stages per warp, 1..MAX_STAGE
    int stage_bytes;  // bytes per stage: a 16-byte multiple with 16 bytes of over-read slack
    int whole;        // 1: items are whole rows; 0: items are single chunks of one row
};
constexpr int MAX_STAGE = 8;
constexpr int MAX_R = GQ_GEMV_MAX_R;

template <int NW>
__host__ __device__ constexpr int bufs_off() {
    return ((NW * MAX_STAGE * 8 + 127) / 128) * 128;  // the mbarriers come first
}

// One launch covers NB activation vectors (blockIdx.y selects the chunk of
// vectors) and all rows.  FUSED: `act` is fp32 [batch][cols] and is
// quantized in the CTA; otherwise `act` holds the quantized blocks.
// w_static != 0 lets the first ring items be requested before the
// dependency wait on the preceding kernel (the caller guarantees no kernel
// still in flight writes W).
template <int WT, int NB, bool SUMS, bool FUSED, int NW>
__global__ void __launch_bounds__(NW * 32, GQ_GEMV_MIN_BLOCKS) gemv_kernel(const uint8_t *__restrict__ W,
                                                   const void *__restrict__ act_in,
                                                   float *__restrict__ y,
                                                   int32_t *__restrict__ sums, int rows,
                                                   int nblk, int batch, int w_static, Geo geo,
                                                   uint32_t *__restrict__ status) {
    using F = Fmt<WT>;
    constexpr int SPB = WT == GQ_Q4_K ? 2 : 1;  // int32 sums per block (diagnostic output)
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b0 = blockIdx.y * NB;
    const int nvec = min(NB, batch - b0);
    const int warps_total = gridDim.x * NW;
    const int wg = blockIdx.x * NW + warp;
    const int nchunk = (nblk + F::CH - 1) / F::CH;
    const int R = geo.R, ns = geo.ns;
    const int ipg = geo.whole ? 1 : nchunk;  // ring items per row group
    const int ngroups = (rows + R - 1) / R;
    const int mine = wg < ngroups ? (ngroups - 1 - wg) / warps_total + 1 : 0;
    const int total = mine * ipg;
    const size_t row_bytes = (size_t)nblk * F::BB;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem) + warp * MAX_STAGE;
    uint8_t *ring = smem + bufs_off<NW>() + (size_t)warp * ns * geo.stage_bytes;

    const uint64_t wpol = GQ_GEMV_W_EVICT_FIRST ? l2_evict_first_policy() : 0ull;
    // item i of this warp = row group wg + (i / ipg) * warps_total, whole or
    // its chunk i % ipg
    auto issue = [&](int i, int st) {
        const int g = wg + (i / ipg) * warps_total;
        const uint8_t *src;
        uint32_t bytes;
        if (geo.whole) {
            const int nr = min(R, rows - g * R);
            src = W + (size_t)g * R * row_bytes;
            bytes = (uint32_t)(nr * row_bytes);
        } else {
            const int c = i % ipg;
            src = W + (size_t)g * row_bytes + (size_t)c * F::CH * F::BB;
            bytes = (uint32_t)(min(F::CH, nblk - c * F::CH) * F::BB);
        }
        mbar_arrive_expect_tx(bar + st, bytes);
        if (GQ_GEMV_W_EVICT_FIRST)
            bulk_g2s_hint(ring + (size_t)st * geo.stage_bytes, src, bytes, bar + st, wpol);
        else
            bulk_g2s(ring + (size_t)st * geo.stage_bytes, src, bytes, bar + st);
    };

    // With the early trigger the next kernel in the stream may launch right
    // away (its CTAs wait on griddepcontrol.wait before touching anything this
    // kernel produces); otherwise it launches once this kernel's activations
    // are staged.
    if (GQ_GEMV_EARLY_TRIGGER) pdl_launch_dependents();
    // Items requested before the activations are staged; the rest of the
    // first ring fill follows the staging, so the activation loads do not
    // queue behind a full ring of weight copies.
    const int pre = min(ns, GQ_GEMV_PREFETCH);
    if (lane == 0 && total > 0) {
        for (int s = 0; s < ns; ++s) mbar_init(bar + s, 1);
        fence_mbar_init();
        if (w_static)
            for (int i = 0; i < pre && i < total; ++i) issue(i, i);
    }
    pdl_wait();  // activations (and, unless static, W) may come from the preceding kernel
    if (lane == 0 && !w_static)
        for (int i = 0; i < pre && i < total; ++i) issue(i, i);

    const Act a = act_layout<WT>(smem + bufs_off<NW>() + (size_t)NW * ns * geo.stage_bytes, NB, nblk);
    const int nact = nvec * nblk;
    if (FUSED) {
        const float *x = static_cast<const float *>(act_in) + (size_t)b0 * nblk * F::BE;
        if (WT == GQ_Q4_K)
            quant_stage_q8_k(a, x, nact, nblk);
        else
            quant_stage_q8_0<WT == GQ_Q4_0>(a, x, nact);
    } else {
        const uint8_t *xq = static_cast<const uint8_t *>(act_in);
        if (WT == GQ_Q4_K)
            stage_q8_k(a, xq + (size_t)b0 * nblk * Q8_K_BYTES, nact, nblk);
        else
            stage_q8_0<WT == GQ_Q4_0>(a, xq + (size_t)b0 * nblk * Q8_0_BYTES, nact);
    }
    __syncthreads();
    if (!GQ_GEMV_EARLY_TRIGGER) pdl_launch_dependents();
    if (lane == 0)
        for (int i = pre; i < ns && i < total; ++i) issue(i, i);

    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;
    const size_t bstride = (size_t)rows * nblk * SPB;
    // Q4_K, one vector, rows of one chunk: every item this warp sees pairs
    // with the same activation slice, so it stays in registers.
    Q4KAct reg;
    const bool act_resident = WT == GQ_Q4_K && NB == 1 && nchunk == 1;
    if (act_resident && (lane >> 1) < nblk) load_q4k_act(reg, a, lane >> 1, lane & 1, lane & 7);

    // one row segment: accumulate into acc (or write the diagnostic sums)
    auto segment = [&](const uint8_t *ch, int row, int c) {
        const int nb_c = min(F::CH, nblk - c * F::CH);
        int32_t *srow = SUMS ? sums + ((size_t)b0 * rows + row) * nblk * SPB : nullptr;
        if (WT == GQ_Q4_K)
            chunk_q4_k<NB, SUMS>(ch, nb_c, c * F::CH, nblk, a, nvec, acc, reg, act_resident, srow,
                                 bstride, lane);
        else
            chunk_q_0<WT, NB, SUMS>(ch, nb_c, c * F::CH, nblk, a, nvec, acc, srow, bstride, lane);
    };
    auto finish_row = [&](int row) {
        if (!SUMS) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < nvec) {
                    const float v = warp_sum(acc[b]);
                    if (lane == 0) y[(size_t)(b0 + b) * rows + row] = v;
                }
                acc[b] = 0.0f;
            }
        }
    };

    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < total; ++i) {
        if (!mbar_wait_bounded(bar + st, ph)) {
            // A transfer never completed: flag it, let the other issued
            // stages drain (bounded), and leave the remaining rows unwritten.
            if (lane == 0) atomicOr(status, STATUS_GEMV_TMA_TIMEOUT);
            int s2 = st;
            uint32_t p2 = ph;
            for (int k = i + 1; k < total && k < i + ns; ++k) {
                if (++s2 == ns) {
                    s2 = 0;
                    p2 ^= 1u;
                }
                mbar_wait_bounded(bar + s2, p2);
            }
            return;
        }
        const int g = wg + (i / ipg) * warps_total;
        const uint8_t *ch = ring + (size_t)st * geo.stage_bytes;
        if (WT == GQ_Q4_K && NB == 1 && !SUMS && nchunk == 1) {
            // batch-1 hot path: the item's rows interleaved (act_resident holds)
            const int nr = min(R, rows - g * R), r0 = g * R;
            float v;
            int rr;
            if (MAX_R >= 4 && R == 4) {
                v = rows_q4_k_nb1<4>(ch, row_bytes, nr, nblk, reg, lane);
                rr = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            } else if (MAX_R >= 2 && R == 2) {
                v = rows_q4_k_nb1<2>(ch, row_bytes, nr, nblk, reg, lane);
                rr = (lane >> 4) & 1;
            } else {
                v = rows_q4_k_nb1<1>(ch, row_bytes, nr, nblk, reg, lane);
                rr = 0;
            }
            if ((lane & 7) == 0 && rr < nr && (R == 4 || (lane & 8) == 0) && (R >= 2 || lane == 0))
                y[(size_t)b0 * rows + r0 + rr] = v;
        } else if (WT == GQ_Q4_K && NB > 1 && !SUMS && geo.whole) {
            // batch 2..8: rows in registers, each vector's slice loaded once per chunk
            item_q4k_multi<NB, (NB * MAX_R <= 32 ? MAX_R : 32 / NB)>(ch, row_bytes, min(R, rows - g * R), nblk,
                                                                     nvec, a, y, rows, g * R, b0, lane);
        } else if (geo.whole) {
            const int nr = min(R, rows - g * R);
            for (int r = 0; r < nr; ++r) {
                for (int c = 0; c < nchunk; ++c)
                    segment(ch + r * row_bytes + (size_t)c * F::CH * F::BB, g * R + r, c);
                finish_row(g * R + r);
            }
        } else {
            const int c = i % ipg;
            segment(ch, g, c);
            if (c == nchunk - 1) finish_row(g);
        }
        __syncwarp();
        if (lane == 0 && i + ns < total) issue(i + ns, st);
        if (++st == ns) {
            st = 0;
            ph ^= 1u;
        }
    }
}

// Plain per-block kernel for Q4_0 / Q8_0 rows whose byte length is not a
// multiple of 16 (cols % 256 != 0): warp per row, lane per block, 16-bit
// global loads, activations read from global memory.
constexpr int PLAIN_WARPS = 8;

template <bool Q4, bool SUMS>
__global__ void __launch_bounds__(PLAIN_WARPS * 32) gemv_plain_kernel(const uint8_t *__restrict__ W,
                                                         const uint8_t *__restrict__ xq,
                                                         float *__restrict__ y,
                                                         int32_t *__restrict__ sums, int rows,
                                                         int nblk, int batch) {
    constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * PLAIN_WARPS + warp;
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
constexpr int CTAS_PER_SM = GQ_GEMV_CTAS_PER_SM;
constexpr int RING_BUDGET = GQ_GEMV_RING_BUDGET;

inline int round16(size_t v) { return (int)((v + 15) / 16 * 16); }

template <int WT>
size_t act_bytes(int nb, int nblk) {
    return (size_t)nb * nblk * act_block_bytes<WT>();
}

template <int WT, int NW>
size_t smem_bytes(const Geo &g, int nb, int nblk) {
    return (size_t)bufs_off<NW>() + (size_t)NW * g.ns * g.stage_bytes + act_bytes<WT>(nb, nblk);
}

// Ring geometry for `rows` rows of `nblk` blocks streamed by `warps` warps.
// Items are whole rows when two stages of one row per warp fit the ring
// budget.  Then R is the most rows per bulk copy (up to 4) that still gives
// at least half the warps an item and keeps two stages per warp within the
// budget (bigger copies stream better, and fewer copies per warp finish a
// short matrix sooner).  Finally there are as many stages as the warp has items, within the
// budget.
template <int WT, int NW>
Geo pick_geo(int rows, int nblk, int warps) {
    using F = Fmt<WT>;
    const int nchunk = (nblk + F::CH - 1) / F::CH;
    const size_t row_bytes = (size_t)nblk * F::BB;
    Geo g;
    g.R = 1;
    g.whole = (size_t)NW * 2 * (size_t)round16(row_bytes + 16) <= (size_t)RING_BUDGET ? 1 : 0;
    if (g.whole)
        for (int r = MAX_R; r > 1; r >>= 1)
            if ((rows + r - 1) / r * GQ_GEMV_R_SPREAD >= warps &&
                (size_t)NW * 2 * (size_t)round16(r * row_bytes + 16) <= (size_t)RING_BUDGET) {
                g.R = r;
                break;
            }
    g.stage_bytes = round16((g.whole ? g.R * row_bytes : (size_t)F::CH * F::BB) + 16);
    const int items = (rows + g.R - 1) / g.R * (g.whole ? 1 : nchunk);
    const int per_warp = (items + warps - 1) / warps;
    const int ns_budget = std::max(1, RING_BUDGET / (NW * g.stage_bytes));
    g.ns = std::max(1, std::min(std::min(per_warp, ns_budget), MAX_STAGE));
    return g;
}

template <int WT, int NB, bool SUMS, bool FUSED, int NW>
cudaError_t launch_one(const void *W, const void *act, float *y, int32_t *sums, int rows,
                       int nblk, int batch, int w_static, const LaunchCtx &ctx) {
    auto k = gemv_kernel<WT, NB, SUMS, FUSED, NW>;
    Geo geo = pick_geo<WT, NW>(rows, nblk, ctx.num_sms * CTAS_PER_SM * NW);
    while (geo.ns > 1 && smem_bytes<WT, NW>(geo, NB, nblk) > (size_t)SMEM_MAX) --geo.ns;
    if (geo.whole && smem_bytes<WT, NW>(geo, NB, nblk) > (size_t)SMEM_MAX) {
        // many staged vectors leave no room for whole rows: stream chunks
        geo.whole = 0;
        geo.R = 1;
        geo.ns = 1;
        geo.stage_bytes = round16((size_t)Fmt<WT>::CH * Fmt<WT>::BB + 16);
    }
    const size_t smem = smem_bytes<WT, NW>(geo, NB, nblk);
    if (smem > (size_t)SMEM_MAX) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
        if (e != cudaSuccess) return e;
    }
    // resident CTAs per SM: the occupancy calculator covers registers and
    // shared memory; the persistent grid never exceeds one wave.
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, NW * 32, smem);
    if (e != cudaSuccess) return e;
    const int per_sm = std::max(1, std::min(CTAS_PER_SM, occ));
    const int groups = (rows + geo.R - 1) / geo.R;
    int grid = (groups + NW - 1) / NW;
    grid = std::max(1, std::min(grid, ctx.num_sms * per_sm));
    dim3 g(grid, (batch + NB - 1) / NB);
    return launch_pdl(k, g, dim3(NW * 32), smem, ctx.stream, static_cast<const uint8_t *>(W), act,
                      y, sums, rows, nblk, batch, w_static, geo, ctx.status);
}

// Vectors per launch chunk: the smallest of {1, 2, 4, 8} that covers the
// batch, so a batch of up to 8 streams the weights once (a batch of 3 runs as
// one chunk of 4 with the last slot unused, not as 2 + 1 with two passes);
// larger batches take chunks of 8.  A smaller chunk is taken when the staged
// activations would not fit in shared memory next to a one-stage ring; 0 if
// none fits.
template <int WT>
int pick_nb(int batch, int nblk) {
    using F = Fmt<WT>;
    Geo g1;
    g1.R = 1;
    g1.ns = 1;
    g1.whole = 0;
    g1.stage_bytes = round16((size_t)F::CH * F::BB + 16);
    int want = 8;
    for (int nb = 1; nb <= 8; nb <<= 1)
        if (nb >= batch) {
            want = nb;
            break;
        }
    for (int nb = want; nb >= 1; nb >>= 1)
        if (smem_bytes<WT, WARPS>(g1, nb, nblk) <= (size_t)SMEM_MAX) return nb;
    return 0;
}

template <int WT, bool SUMS, bool FUSED>
cudaError_t dispatch_wt(const void *W, const void *act, float *y, int32_t *sums, int rows,
                        int nblk, int batch, int w_static, const LaunchCtx &ctx) {
    const int nb = pick_nb<WT>(batch, nblk);
    switch (nb) {
    case 8: return launch_one<WT, 8, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
    case 4: return launch_one<WT, 4, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
    case 2: return launch_one<WT, 2, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
    case 1: return launch_one<WT, 1, SUMS, FUSED, WARPS>(W, act, y, sums, rows, nblk, batch, w_static, ctx);
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
        dim3 grid((rows + PLAIN_WARPS - 1) / PLAIN_WARPS, batch);
        const uint8_t *w8 = static_cast<const uint8_t *>(W);
        const uint8_t *a8 = static_cast<const uint8_t *>(act);
        if (wtype == GQ_Q4_0)
            return launch_pdl(gemv_plain_kernel<true, SUMS>, grid, dim3(PLAIN_WARPS * 32), 0, ctx.stream, w8, a8,
                              y, sums, rows, nblk, batch);
        return launch_pdl(gemv_plain_kernel<false, SUMS>, grid, dim3(PLAIN_WARPS * 32), 0, ctx.stream, w8, a8, y,
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
