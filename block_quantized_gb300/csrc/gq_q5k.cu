// gq_q5k.cu -- the Q5_K x Q8_K GEMV.
//
// Q5_K is the 5-bit K-quant, one bit more than Q4_K (the discosf.com page
// "为什么说 llama.cpp 是'裸引擎'——从模型加载的每一行代码说起", §4 量化不是"压缩"，
// 而是"精度重分配"): the Q4_K super-block of "llama.cpp 推理引擎" §5.5 (fp16 d
// and dmin, 6-bit scale sc_j and min m_j per 32-element sub-block) with codes
// q in [0, 31], w = d * sc_j * q - dmin * m_j.  Block (176 B): bytes 0..143 as
// Q4_K (d, dmin, the sixteen 6-bit fields, the low four bits of the codes in
// the Q4_0 nibble order), then 32 bytes @144 with the fifth bits: bit 2t + p
// of byte 144 + 4j + i is the fifth bit of element 32j + 8t + 2i + p.  That
// places, for the nibble word t of sub-block j (elements 8t..8t+7), the fifth
// bits of its even elements at bits 2t, 2t + 8, 2t + 16, 2t + 24 of the
// sub-block's fifth-bit word -- one shift and one mask line them up with the
// bytes of the word's low-nibble operand (likewise bit 2t + 1 for the odd
// elements).  The codecs live with the other K-quant codecs (gq_codec.cu).
//
// The product, per super-block and activation vector ("llama.cpp 推理引擎"
// §5.5 two-level scales, §6.4 block dot): s_j = sum_{i in j} q_i * a_i,
// S1 = sum_j sc_j * s_j, S2 = sum_j m_j * t_j (t_j the Q8_K sub-block sums),
// y += d_x * (d * S1 - dmin * S2).
//
// GEMV.  Decode is bound by the bytes of W streamed ("llama.cpp 推理引擎"
// §7.3), so the kernel streams each row once:
//   - a persistent grid of at most one CTA per SM, 16 warps (8 when sixteen
//     two-stage rings do not fit); warp w of the grid owns rows w, w + warps,
//     ...; each warp streams its rows through a private shared-memory ring of
//     2-4 whole-row stages, one bulk copy (cp.async.bulk, evict-first L2
//     policy) per row completing on an mbarrier; every wait is bounded.
//     Blocks are 176 = 11 x 16 bytes, so every row and every block field is
//     16-byte aligned and all shared loads are 128-bit;
//   - the CTA stages up to eight Q8_K vectors (the smallest group of 1, 2, 4
//     or 8 that covers the batch, fewer when wide vectors leave no room for
//     the rings), so W streams once per group; each vector: codes in 128-byte
//     half-super-block units, each 8-code group stored as (a0 a2 a4 a6 |
//     a1 a3 a5 a7) so the even and odd elements of a nibble word meet their
//     activations in one dp4a each, 16-byte pieces XOR-swizzled by the unit
//     index (distinct banks for a quarter-warp); then the eight sub-block
//     sums and the scale;
//   - a lane takes half a super-block (four sub-blocks, 128 elements): one
//     header load, four 16-byte nibble loads and one 16-byte fifth-bit load;
//     per 8 elements two 5-bit code words built with shifts and masks, once,
//     and two dp4a per staged vector; S1 and S2 of the half in int32; fp32
//     partials per lane and vector, one warp-shuffle reduction per row and
//     vector.  14336 x 4096 at batch 1 / 2 / 4 / 8: 9.4 / 11.5 / 16.2 / 25.6
//     us (one vector per pass: 9.3 / 16.4 / 30.2 / 56.4).
// Rows too long for a two-stage ring take a plain warp-per-row kernel that
// reads W and the activations from global memory.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_quant8.cuh"

namespace gq {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr uint32_t BIT4 = 0x10101010u;
constexpr int MAX_NS = 4;  // ring stages per warp
// the mbarriers, at the start of shared memory
__host__ __device__ constexpr int bars_bytes(int nw) { return nw * MAX_NS * 8; }

// Shared-memory footprint of one staged Q8_K vector of nblk blocks: codes,
// then the eight int32 sub-block sums per block, then one fp32 scale per
// block.
__host__ __device__ constexpr size_t act_smem_bytes(int nblk) {
    return (size_t)nblk * 256 + (size_t)nblk * 8 * 4 + (size_t)nblk * 4;
}
// Staged vectors follow one another at this stride (16-byte aligned).
__host__ __device__ constexpr size_t act_stride(int nblk) { return (act_smem_bytes(nblk) + 15) / 16 * 16; }

// Split-order words of 8 codes: (a0 a2 a4 a6) and (a1 a3 a5 a7).
__device__ __forceinline__ uint2 split8(uint32_t w0, uint32_t w1) {
    return make_uint2(__byte_perm(w0, w1, 0x6420), __byte_perm(w0, w1, 0x7531));
}

// Stage one Q8_K vector (nblk blocks at xq) into shared memory at `act`.
// Unit u (16 codes: elements 128h + 16u .. +15) of half-block hb = 2k + h is
// stored at hb * 128 + (u ^ (hb & 7)) * 16 as {split(g0).x, .y, split(g1).x, .y}.
__device__ void stage_q8_k_vec(uint8_t *act, const uint8_t *__restrict__ xq, int nblk) {
    int32_t *tsum = reinterpret_cast<int32_t *>(act + (size_t)nblk * 256);
    float *dx = reinterpret_cast<float *>(tsum + 8 * nblk);
    for (int idx = threadIdx.x; idx < nblk * 16; idx += blockDim.x) {
        const int hb = idx >> 3, u = idx & 7;
        const uint8_t *blk = xq + (size_t)(hb >> 1) * Q8_K_BYTES;  // 4-byte aligned
        const uint32_t *c = reinterpret_cast<const uint32_t *>(blk + 4 + (hb & 1) * 128 + u * 16);
        const uint2 g0 = split8(c[0], c[1]), g1 = split8(c[2], c[3]);
        *reinterpret_cast<uint4 *>(act + (size_t)hb * 128 + ((u ^ (hb & 7)) << 4)) =
            make_uint4(g0.x, g0.y, g1.x, g1.y);
    }
    for (int i = threadIdx.x; i < 8 * nblk; i += blockDim.x) {
        const uint8_t *blk = xq + (size_t)(i >> 3) * Q8_K_BYTES;
        tsum[i] = (int32_t) reinterpret_cast<const int16_t *>(blk + 260)[i & 7];
        if ((i & 7) == 0) dx[i >> 3] = *reinterpret_cast<const float *>(blk);
    }
}

// Integer sums of half h of the block at `blk` (shared memory, 16-byte
// aligned) against the staged codes of half-block hb of NV vectors (vector v
// at act + v * astride): S1[v] = sum_j sc_j s_j and S2[v] = sum_j m_j t_j over
// the half's four sub-blocks j = 4h + k.  The 5-bit code words are built once
// and serve every vector.
template <int NV>
__device__ __forceinline__ void half_sums(const uint8_t *blk, int h, const uint8_t *act, size_t astride, int nblk,
                                          int hb, int (&S1)[NV], int (&S2)[NV]) {
    const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
    // header bytes 4..15 = words y, z, w: this half's four sc (bits 24h..24h+23)
    // and four m (bits 48+24h..71+24h) are three whole bytes each
    const uint32_t sc24 = __byte_perm(hd.y, hd.z, h ? 0x0543u : 0x0210u);
    const uint32_t m24 = __byte_perm(hd.z, hd.w, h ? 0x0765u : 0x0432u);
    uint32_t ce[4][4], co[4][4];  // [sub-block k][nibble word tt]: even / odd element codes
    {
        const uint4 fb = *reinterpret_cast<const uint4 *>(blk + 144 + 16 * h);  // fifth bits of the half
        const uint32_t F[4] = {fb.x, fb.y, fb.z, fb.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 q = *reinterpret_cast<const uint4 *>(blk + 16 + 64 * h + 16 * k);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {  // nibble word tt: elements 8tt..8tt+7
                // fifth bits of the even (odd) elements at bits 2tt (2tt + 1)
                // of each byte of F[k], moved to bit 4 of each byte
                const uint32_t fe = (2 * tt <= 4 ? F[k] << (4 - 2 * tt) : F[k] >> (2 * tt - 4)) & BIT4;
                const uint32_t fo = (2 * tt + 1 <= 4 ? F[k] << (3 - 2 * tt) : F[k] >> (2 * tt - 3)) & BIT4;
                ce[k][tt] = (w[tt] & NIB) | fe;
                co[k][tt] = ((w[tt] >> 4) & NIB) | fo;
            }
        }
    }
    const int sw = hb & 7;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const uint8_t *av = act + (size_t)v * astride;
        const uint8_t *ah = av + (size_t)hb * 128;
        const int4 t = reinterpret_cast<const int4 *>(av + (size_t)nblk * 256)[hb];  // t_j of the half
        const int tj[4] = {t.x, t.y, t.z, t.w};
        int s1 = 0, s2 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // sub-block 4h + k: units 2k, 2k + 1 of the half
            const uint4 a0 = *reinterpret_cast<const uint4 *>(ah + (((2 * k) ^ sw) << 4));
            const uint4 a1 = *reinterpret_cast<const uint4 *>(ah + (((2 * k + 1) ^ sw) << 4));
            const uint32_t ae[4] = {a0.x, a0.z, a1.x, a1.z}, ao[4] = {a0.y, a0.w, a1.y, a1.w};
            int sk = 0;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                sk = dp4a_us(ce[k][tt], (int)ae[tt], sk);
                sk = dp4a_us(co[k][tt], (int)ao[tt], sk);
            }
            s1 += (int)((sc24 >> (6 * k)) & 63u) * sk;
            s2 += (int)((m24 >> (6 * k)) & 63u) * tj[k];
        }
        S1[v] = s1;
        S2[v] = s2;
    }
}

// Streaming kernel: NV activation vectors per blockIdx.y (vectors NV y ..
// NV y + NV - 1 of the nvec in this launch), so W streams once per NV
// vectors.  SUMS: write the int32 sums S1, S2 of every block instead of y.
template <bool SUMS, int GW, bool FUSED, int NV>
__global__ void __launch_bounds__(GW * 32, 1) gemv_q5k_kernel(const uint8_t *__restrict__ W,
                                                             const void *__restrict__ act_in,
                                                             float *__restrict__ y, int32_t *__restrict__ sums,
                                                             int rows, int nblk, int ns, int stage_bytes, int nvec,
                                                             int w_static, uint32_t *__restrict__ status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b0 = blockIdx.y * NV, nv = min(NV, nvec - b0);
    const size_t astride = act_stride(nblk);
    const int warps_total = gridDim.x * GW;
    const int wg = blockIdx.x * GW + warp;
    const int total = wg < rows ? (rows - 1 - wg) / warps_total + 1 : 0;
    const uint32_t row_bytes = (uint32_t)nblk * Q5_K_BYTES;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem) + warp * MAX_NS;
    uint8_t *ring = smem + bars_bytes(GW) + (size_t)warp * ns * stage_bytes;
    uint8_t *act = smem + bars_bytes(GW) + (size_t)GW * ns * stage_bytes;
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int i, int st) {
        const size_t row = (size_t)wg + (size_t)i * warps_total;
        mbar_arrive_expect_tx(bar + st, row_bytes);
        bulk_g2s_hint(ring + (size_t)st * stage_bytes, W + row * row_bytes, row_bytes, bar + st, pol);
    };

    pdl_launch_dependents();
    if (lane == 0 && total > 0) {
        for (int s = 0; s < ns; ++s) mbar_init(bar + s, 1);
        fence_mbar_init();
        // weights no kernel in flight writes (GQ_FLAG_W_STATIC): the first
        // ring stages are requested before the dependency wait
        if (w_static)
            for (int i = 0; i < ns && i < total; ++i) issue(i, i);
    }
    __syncwarp();
    pdl_wait();  // xq (and, unless static, W) may come from the preceding kernel in the stream
    if (lane == 0 && !w_static)
        for (int i = 0; i < ns && i < total; ++i) issue(i, i);
    for (int v = 0; v < nv; ++v) {
        const size_t b = (size_t)(b0 + v);
        if (FUSED)  // fp32 activations, quantized to Q8_K here exactly as by the codec
            q8::stage_q8_k_from_f32<8>(act + v * astride, static_cast<const float *>(act_in) + b * nblk * QK_K,
                                       nblk);
        else
            stage_q8_k_vec(act + v * astride, static_cast<const uint8_t *>(act_in) + b * nblk * Q8_K_BYTES, nblk);
    }
    __syncthreads();

    const size_t dx_off = (size_t)nblk * 256 + (size_t)nblk * 8 * 4;  // the scales, within a staged vector
    const int iters = (2 * nblk + 31) / 32;
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < total; ++i) {
        if (!mbar_wait_bounded(bar + st, ph)) {
            // A transfer never completed: flag it, let the other issued
            // stages drain (bounded) and leave this warp's remaining rows.
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
        const int row = wg + i * warps_total;
        const uint8_t *stage = ring + (size_t)st * stage_bytes;
        float acc[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[v] = 0.0f;
        for (int t = 0; t < iters; ++t) {
            const int hb = lane + 32 * t;
            int S1[NV], S2[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) S1[v] = S2[v] = 0;
            if (hb < 2 * nblk) {
                const int k = hb >> 1;
                const uint8_t *blk = stage + (size_t)k * Q5_K_BYTES;
                half_sums<NV>(blk, hb & 1, act, astride, nblk, hb, S1, S2);
                if (!SUMS) {
                    const uint32_t dd = *reinterpret_cast<const uint32_t *>(blk);
                    const float d = half_bits_to_float(dd), dmin = half_bits_to_float(dd >> 16);
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const float dxv = reinterpret_cast<const float *>(act + v * astride + dx_off)[k];
                        acc[v] += dxv * (d * (float)S1[v] - dmin * (float)S2[v]);
                    }
                }
            }
            if (SUMS) {
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int s1 = S1[v] + __shfl_xor_sync(FULL, S1[v], 1);  // the two halves of block hb / 2
                    const int s2 = S2[v] + __shfl_xor_sync(FULL, S2[v], 1);
                    if (v < nv && hb < 2 * nblk && (hb & 1) == 0) {
                        int32_t *o = sums + (((size_t)(b0 + v) * rows + row) * nblk + (hb >> 1)) * 2;
                        o[0] = s1;
                        o[1] = s2;
                    }
                }
            }
        }
        if (!SUMS) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const float a = warp_sum(acc[v]);
                if (lane == 0 && v < nv) y[(size_t)(b0 + v) * rows + row] = a;
            }
        }
        __syncwarp();
        if (lane == 0 && i + ns < total) issue(i + ns, st);
        if (++st == ns) {
            st = 0;
            ph ^= 1u;
        }
    }
}

// Plain kernel for any cols (a multiple of 256): warp per (row, vector), lane
// per half block, byte loads from global memory.
constexpr int PW = 8;

template <bool SUMS>
__global__ void __launch_bounds__(PW * 32) gemv_q5k_plain_kernel(const uint8_t *__restrict__ W,
                                                                 const uint8_t *__restrict__ xq,
                                                                 float *__restrict__ y,
                                                                 int32_t *__restrict__ sums, int rows, int nblk) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * PW + warp;
    const int b = blockIdx.y;
    pdl_launch_dependents();
    pdl_wait();
    if (row >= rows) return;
    const int iters = (2 * nblk + 31) / 32;
    float acc = 0.0f;
    for (int t = 0; t < iters; ++t) {
        const int hb = lane + 32 * t;
        int S1 = 0, S2 = 0;
        float d = 0.0f, dmin = 0.0f, dxv = 0.0f;
        if (hb < 2 * nblk) {
            const int k = hb >> 1, h = hb & 1;
            const uint8_t *wb = W + ((size_t)row * nblk + k) * Q5_K_BYTES;
            const uint8_t *ab = xq + ((size_t)b * nblk + k) * Q8_K_BYTES;
            uint32_t f[16];  // the sixteen 6-bit fields, LSB-first in bytes 4..15
            uint64_t lo = 0, hi = 0;
            for (int i = 0; i < 8; ++i) lo |= (uint64_t)__ldg(wb + 4 + i) << (8 * i);
            for (int i = 0; i < 4; ++i) hi |= (uint64_t)__ldg(wb + 12 + i) << (8 * i);
            for (int i = 0; i < 10; ++i) f[i] = (uint32_t)((lo >> (6 * i)) & 63);
            f[10] = (uint32_t)(((lo >> 60) | (hi << 4)) & 63);
            for (int i = 11; i < 16; ++i) f[i] = (uint32_t)((hi >> (6 * i - 64)) & 63);
            for (int j = 4 * h; j < 4 * h + 4; ++j) {
                int s = 0;
                for (int r = 0; r < 32; ++r) {
                    const int e = 32 * j + r;
                    const int nib = (__ldg(wb + 16 + (e >> 1)) >> (4 * (e & 1))) & 15;
                    const int fifth = (__ldg(wb + 144 + 4 * j + ((r & 7) >> 1)) >> (2 * (r >> 3) + (r & 1))) & 1;
                    s += (nib | (fifth << 4)) * (int)(int8_t)__ldg(ab + 4 + e);
                }
                S1 += (int)f[j] * s;
                S2 += (int)f[8 + j] * (int)__ldg(reinterpret_cast<const int16_t *>(ab + 260) + j);
            }
            d = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(wb)));
            dmin = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(wb) + 1));
            dxv = __ldg(reinterpret_cast<const float *>(ab));
        }
        if (SUMS) {
            const int s1 = S1 + __shfl_xor_sync(FULL, S1, 1);
            const int s2 = S2 + __shfl_xor_sync(FULL, S2, 1);
            if (hb < 2 * nblk && (hb & 1) == 0) {
                int32_t *o = sums + (((size_t)b * rows + row) * nblk + (hb >> 1)) * 2;
                o[0] = s1;
                o[1] = s2;
            }
        } else {
            acc += dxv * (d * (float)S1 - dmin * (float)S2);
        }
    }
    if (!SUMS) {
        acc = warp_sum(acc);
        if (lane == 0) y[(size_t)b * rows + row] = acc;
    }
}

// ------------------------------------------------------------------ launch

constexpr int SMEM_LIMIT = 232448;  // opt-in shared memory per CTA on sm_103
constexpr int64_t Y_MAX = 65535;    // vectors per launch (grid.y)

size_t stream_smem(int nw, int ns, int nblk, int nv) {
    return bars_bytes(nw) + (size_t)nw * ns * ((size_t)nblk * Q5_K_BYTES) + (size_t)nv * act_stride(nblk);
}

// Ring stages per warp for the streaming kernel with nw warps: as many as fit
// (2..4) next to nv staged vectors; 0 when two stages do not fit.
int pick_ns(int nw, int nblk, int nv) {
    for (int ns = MAX_NS; ns >= 2; --ns)
        if (stream_smem(nw, ns, nblk, nv) <= (size_t)SMEM_LIMIT) return ns;
    return 0;
}

// Launch shape of the streaming kernel for a batch: nv vectors per CTA (the
// smallest of 1, 2, 4, 8 that covers the batch, fewer when their staged
// copies leave no room for a two-stage ring), 16 warps when sixteen rings fit
// (eight vectors always take 8 warps: at 16 the kernel is capped at 128
// registers and spills; 25.6 vs 29.8 us at 14336 x 4096), else 8, and the
// ring depth.  ns == 0: not even one vector fits.
struct Shape {
    int nv, nw, ns;
};
Shape pick_shape(int nblk, int64_t batch) {
    int nv = batch >= 8 ? 8 : batch >= 4 ? (batch > 4 ? 8 : 4) : batch >= 2 ? (batch > 2 ? 4 : 2) : 1;
    for (; nv >= 1; nv >>= 1) {
        if (nv < 8)
            if (int ns = pick_ns(16, nblk, nv)) return {nv, 16, ns};
        if (int ns = pick_ns(8, nblk, nv)) return {nv, 8, ns};
    }
    return {1, 8, 0};
}

template <bool SUMS, int NW, bool FUSED, int NV>
cudaError_t launch_stream(const uint8_t *W, const void *xb, float *yb, int32_t *sb, int64_t rows, int nblk,
                          int nb, int ns, int w_static, const LaunchCtx &ctx) {
    auto k = gemv_q5k_kernel<SUMS, NW, FUSED, NV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    const int64_t gx = std::min<int64_t>(ctx.num_sms, (rows + NW - 1) / NW);
    return launch_pdl(k, dim3((unsigned)gx, (nb + NV - 1) / NV), dim3(NW * 32), stream_smem(NW, ns, nblk, NV),
                      ctx.stream, W, xb, yb, sb, (int)rows, nblk, ns, nblk * Q5_K_BYTES, nb, w_static, ctx.status);
}

template <bool SUMS, bool FUSED, int NW>
cudaError_t launch_nv(const Shape &sh, const uint8_t *W, const void *xb, float *yb, int32_t *sb, int64_t rows,
                      int nblk, int nb, int w_static, const LaunchCtx &ctx) {
    switch (sh.nv) {
    case 8:
        if constexpr (NW == 8)  // eight vectors always run on 8 warps (pick_shape)
            return launch_stream<SUMS, NW, FUSED, 8>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
        else
            return cudaErrorInvalidValue;
    case 4: return launch_stream<SUMS, NW, FUSED, 4>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    case 2: return launch_stream<SUMS, NW, FUSED, 2>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    default: return launch_stream<SUMS, NW, FUSED, 1>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    }
}

template <bool SUMS, bool FUSED>
cudaError_t run_gemv(const uint8_t *W, const void *act, float *y, int32_t *sums, int64_t rows, int64_t cols,
                     int64_t batch, int w_static, const LaunchCtx &ctx) {
    const int nblk = (int)(cols / QK_K);
    const Shape sh = pick_shape(nblk, batch);
    const int64_t per_launch = sh.ns ? Y_MAX * sh.nv : Y_MAX;
    for (int64_t b0 = 0; b0 < batch; b0 += per_launch) {
        const int nb = (int)std::min<int64_t>(per_launch, batch - b0);
        const void *xb = FUSED ? static_cast<const void *>(static_cast<const float *>(act) + b0 * cols)
                               : static_cast<const void *>(static_cast<const uint8_t *>(act) + b0 * nblk * Q8_K_BYTES);
        float *yb = SUMS ? nullptr : y + b0 * rows;
        int32_t *sb = SUMS ? sums + b0 * rows * nblk * 2 : nullptr;
        cudaError_t e;
        if (sh.ns && sh.nw == 16) {
            e = launch_nv<SUMS, FUSED, 16>(sh, W, xb, yb, sb, rows, nblk, nb, w_static, ctx);
        } else if (sh.ns) {
            e = launch_nv<SUMS, FUSED, 8>(sh, W, xb, yb, sb, rows, nblk, nb, w_static, ctx);
        } else {
            if (FUSED) return cudaErrorInvalidValue;  // one vector does not fit the streaming kernel
            const int64_t gx = (rows + PW - 1) / PW;
            e = launch_pdl(gemv_q5k_plain_kernel<SUMS>, dim3((unsigned)gx, nb), dim3(PW * 32), 0, ctx.stream, W,
                           static_cast<const uint8_t *>(xb), yb, sb, (int)rows, nblk);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// The fused form has no plain-kernel fallback: the whole vector must fit the
// streaming kernel next to a two-stage ring.
bool gemv_q5k_fused_fits(int64_t cols) {
    if (cols < 0 || cols % QK_K != 0 || cols > (int64_t)1 << 20) return false;
    return pick_shape((int)(cols / QK_K), 1).ns > 0;
}

cudaError_t launch_gemv_q5k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t cols,
                            int64_t batch, bool fused, bool w_static, const LaunchCtx &ctx) {
    const uint8_t *w8 = static_cast<const uint8_t *>(W);
    const int ws = w_static ? 1 : 0;
    if (fused)
        return sums ? run_gemv<true, true>(w8, xq, y, sums, rows, cols, batch, ws, ctx)
                    : run_gemv<false, true>(w8, xq, y, sums, rows, cols, batch, ws, ctx);
    return sums ? run_gemv<true, false>(w8, xq, y, sums, rows, cols, batch, ws, ctx)
                : run_gemv<false, false>(w8, xq, y, sums, rows, cols, batch, ws, ctx);
}

}  // namespace gq
