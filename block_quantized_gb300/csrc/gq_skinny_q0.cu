// gq_skinny_q0.cu -- Q4_0 / Q8_0 weights x Q8_0 activations for small
// batches (up to 64 activation vectors per launch) on warp-level tensor-core
// MMAs (mma.sync m16n8k16, fp16 operands, fp32 accumulate): the per-block
// product of "llama.cpp 推理引擎" §5.3-5.4 and §6.4, y = sum over 32-element
// blocks of d_w * d_x * s, s the integer dot of the two blocks' codes.
//
// Between the GEMV (whose dp4a work grows with every vector) and the tcgen05
// kernel for these formats (one tensor-memory accumulator per block, so a
// CTA-wide handshake per pair of blocks), the product is a skinny
// contraction bound by the weight stream.  Each compute warp owns 16 weight
// rows and turns them into MMA A fragments in registers itself; every block
// gets a fresh accumulator in registers (two K = 16 MMAs), which the warp
// scales and adds to its fp32 y right away.
//
// Exactness: A = q - 8 (Q4_0, in [-8, 7]) or the Q8_0 code (in [-128, 127]),
// B = the Q8_0 activation code, all exact fp16 integers; a block dot is at
// most 32 * 128 * 128 = 2^19 in magnitude, so its fp32 accumulation is exact
// in any order and the int32 block sums equal the oracle's.
//
// CTA (96 weight rows, 8 NT activation columns), as the Q4_K warp-level
// kernel: KS groups of six compute warps (group g takes the stages sb = g
// mod KS of the same rows; partial y added in group order at the end), one
// producer warp streaming one 2-D TMA tile per stage (eight blocks = 256 K
// elements of 96 rows: 144 bytes per row for Q4_0, 272 for Q8_0; rows past
// the matrix read as zeros), four converter warps turning the Q8_0 activation
// blocks, KC stages at a time, into fp16 B fragments and column scales in
// shared memory (two chunk buffers).  Every mbarrier wait is bounded and
// reports through the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_mma_sync.cuh"
#include "gq_tc.cuh"

namespace gq {
namespace {

using namespace ms;

constexpr int SQ_PRE = 2;                  // weight tiles requested before the dependency wait (static W)
constexpr int SQ_NW = 6;                   // row tiles of 16 per CTA
constexpr int SQ_ROWS = 16 * SQ_NW;        // weight rows per CTA
constexpr int SQ_SM_SMEM = 233472;         // shared memory per SM (1 KB of it reserved per CTA)

template <int WT, int NT_>
struct SqCfg {
    static constexpr bool Q4 = WT == GQ_Q4_0;
    static constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;  // block bytes
    static constexpr int ROWB = 8 * BB;                      // one stage of one row: 144 / 272 bytes
    static constexpr int STAGE = SQ_ROWS * ROWB;             // 13,824 / 26,112 bytes
    static constexpr int NT = NT_;
    static constexpr int BCOLS = 8 * NT_;
    static constexpr int KS = NT_ == 1 ? 4 : (NT_ <= 4 ? 2 : 1);
    static constexpr int NCW = SQ_NW * KS;
    static constexpr int CW = 4;
    static constexpr int PRODUCER = NCW;
    static constexpr int CONV0 = NCW + 1;
    static constexpr int THREADS = 32 * (NCW + 1 + CW);
    static constexpr int LIMIT = SQ_SM_SMEM - 1024;
    static constexpr int KC = NT_ == 1 ? 8 : (NT_ <= 4 ? 16 / NT_ : 2);  // stages per activation chunk
    static constexpr int PART = (KS - 1) * SQ_NW * 32 * NT_ * 16;      // partial y of groups 1..
    // one activation chunk: B fragments [nt][block of the chunk][lane] (uint4:
    // the two K = 16 steps of the block), column scales [block][column]
    static constexpr int BFRAG = NT_ * KC * 8 * 32 * 16;
    static constexpr int COLF = KC * 8 * BCOLS * 4;
    static constexpr int CHUNK = BFRAG + COLF;
    static constexpr int OFF_CHUNK = 0;
    static constexpr int OFF_PART = 2 * CHUNK;
    static constexpr int OFF_RING = (OFF_PART + PART + 127) / 128 * 128;
    static constexpr int FIXED = OFF_RING + 16 + 16 * 8 + 4 * 8 + 16 + 128;
    static constexpr int NS = (LIMIT - FIXED) / STAGE > 8 ? 8 : (LIMIT - FIXED) / STAGE;
    // 16 bytes of slack after the ring: the realigning loads of a row's last
    // block read up to 4 bytes past it
    static constexpr int OFF_BAR = OFF_RING + NS * STAGE + 16;
    static constexpr int OFF_MISC = OFF_BAR + (2 * NS + 4) * 8;
    static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 128;
    static_assert(NS >= 2 && NS >= SQ_PRE, "ring");
    static_assert(THREADS <= 1024, "threads per CTA");
    static_assert(SMEM_ALLOC <= LIMIT, "shared memory budget");
    static_assert(OFF_RING % 128 == 0 && STAGE % 128 == 0, "TMA destinations");
    static_assert(ROWB % 16 == 0, "TMA box rows are 16-byte multiples");
    static_assert(CHUNK % 16 == 0, "fragment alignment");
};

inline int pick_nt(int64_t batch) { return batch <= 8 ? 1 : batch <= 16 ? 2 : batch <= 32 ? 4 : 8; }

// Eight bytes starting `off` bytes into shared memory (off even), as two
// words: aligned loads and a funnel shift by 0 or 16 bits.
__device__ __forceinline__ uint2 load8_even(const uint8_t *base, uint32_t off) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(base + (off & ~3u));
    const uint32_t sh = (off & 2u) * 8u;
    const uint32_t v0 = w[0], v1 = w[1], v2 = w[2];
    return make_uint2(__funnelshift_r(v0, v1, sh), __funnelshift_r(v1, v2, sh));
}

// Four bytes starting `off` bytes into shared memory (off even).
__device__ __forceinline__ uint32_t load4_even(const uint8_t *base, uint32_t off) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(base + (off & ~3u));
    return __funnelshift_r(w[0], w[1], (off & 2u) * 8u);
}

// Activation chunk c (stages c KC .. + kc - 1, i.e. blocks 8 c KC ..) into
// buffer `buf`, by the converter warps (thread tid of CW * 32).  Every global
// load of the chunk is issued before any value is converted.  Columns past
// the batch are zeros.
//   B fragments: item (nt, jj, lane), jj a block of the chunk: the eight
//     codes 8 t .. 8 t + 7 of column 8 nt + lane / 4 as four fp16 pairs;
//   column scales: item (jj, column): d_x of the block as fp32.
// Q8_0 blocks are 34 bytes, so their fields are read with 16-bit loads.
template <class C>
__device__ void convert_chunk_q0(uint8_t *buf, const uint8_t *__restrict__ xq, int c, int kc, int nblk,
                                 int batch, int tid) {
    constexpr int NTH = 32 * C::CW;
    constexpr int JB = 8 * C::KC;  // blocks per chunk
    constexpr int NB = C::NT * JB * 32, UB = (NB + NTH - 1) / NTH;
    constexpr int NCI = JB * C::BCOLS, UC = (NCI + NTH - 1) / NTH;
    uint4 *bf = reinterpret_cast<uint4 *>(buf);
    float *cf = reinterpret_cast<float *>(buf + C::BFRAG);
    auto block_of = [&](int n, int jj) { return xq + ((size_t)n * nblk + (size_t)c * JB + jj) * Q8_0_BYTES; };
    uint32_t w0[UB], w1[UB];
    uint16_t dh[UC];
#pragma unroll
    for (int u = 0; u < UB; ++u) {
        const int i = tid + u * NTH;
        const int ln = i & 31, jj = (i >> 5) % JB, nt = (i >> 5) / JB;
        const int n = 8 * nt + (ln >> 2), t = ln & 3;
        w0[u] = w1[u] = 0u;
        if (i < NB && jj < 8 * kc && n < batch) {
            const uint16_t *p = reinterpret_cast<const uint16_t *>(block_of(n, jj) + 2 + 8 * t);
            w0[u] = (uint32_t)__ldg(p) | ((uint32_t)__ldg(p + 1) << 16);
            w1[u] = (uint32_t)__ldg(p + 2) | ((uint32_t)__ldg(p + 3) << 16);
        }
    }
#pragma unroll
    for (int u = 0; u < UC; ++u) {
        const int i = tid + u * NTH;
        const int jj = i / C::BCOLS, n = i % C::BCOLS;
        dh[u] = 0;
        if (i < NCI && jj < 8 * kc && n < batch) dh[u] = __ldg(reinterpret_cast<const uint16_t *>(block_of(n, jj)));
    }
#pragma unroll
    for (int u = 0; u < UB; ++u) {
        const int i = tid + u * NTH;
        if (i < NB) bf[i] = i8x8_to_f16(w0[u], w1[u]);  // zero codes convert to zeros
    }
#pragma unroll
    for (int u = 0; u < UC; ++u) {
        const int i = tid + u * NTH;
        if (i < NCI) cf[i] = half_bits_to_float(dh[u]);
    }
}

template <int WT, int NT, bool SUMS>
__global__ void __launch_bounds__(SqCfg<WT, NT>::THREADS, 1) skinny_q0_kernel(
    const __grid_constant__ CUtensorMap tmap_w, const uint8_t *__restrict__ xq, float *__restrict__ y,
    int32_t *__restrict__ sums, int rows, int nsb, int batch, int w_static, uint32_t *__restrict__ status) {
    using C = SqCfg<WT, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::NS;
    uint64_t *cfull = empty + C::NS;  // activation chunk buffer b converted (one arrival per converter warp)
    uint64_t *cempty = cfull + 2;     // activation chunk buffer b read (one arrival per compute warp)
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * SQ_ROWS;
    const int nblk = nsb * 8;
    const int nchunks = (nsb + C::KC - 1) / C::KC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, SQ_NW);  // the six warps of the stage's group
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(cfull + i, C::CW);
            mbar_init(cempty + i, C::NCW);
        }
        *abort = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // one 2-D TMA tile (eight blocks of the CTA's 96 rows) into ring slot `slot`
    auto issue_tile = [&](int sb, int slot) {
        mbar_arrive_expect_tx(full + slot, C::STAGE);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + C::OFF_RING + slot * C::STAGE)),
            "l"(reinterpret_cast<uint64_t>(&tmap_w)), "r"(sb * (C::ROWB / 2)), "r"(row0), "r"(smem_u32(full + slot))
            : "memory");
    };
    // Static weights (no kernel in flight writes W): the first SQ_PRE tiles
    // are requested before the dependency wait.
    const int pre = w_static ? min(SQ_PRE, nsb) : 0;
    if (warp == C::PRODUCER && lane == 0)
        for (int sb = 0; sb < pre; ++sb) issue_tile(sb, sb);
    pdl_wait();  // the activations (and W, unless static) may come from the preceding kernel

    if (warp >= C::CONV0) {
        for (int c = 0; c < nchunks; ++c) {
            const int bi = c & 1;
            if (c >= 2 && !tc::wait_warp(cempty + bi, (uint32_t)((c - 2) >> 1) & 1u, abort)) break;
            convert_chunk_q0<C>(smem + C::OFF_CHUNK + bi * C::CHUNK, xq, c, min(C::KC, nsb - c * C::KC), nblk,
                                batch, threadIdx.x - 32 * C::CONV0);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(cfull + bi);
        }
    } else if (warp == C::PRODUCER) {
        tc::RingPos rp(C::NS);
        int last[8];
        for (int i = 0; i < 8; ++i) last[i] = -1;
        for (int sb = 0; sb < pre; ++sb) {
            last[rp.idx] = (int)rp.phase;
            rp.next();
        }
        bool ok = true;
        for (int sb = pre; sb < nsb; ++sb) {
            if (!(ok = tc::wait_warp(empty + rp.idx, rp.phase ^ 1u, abort))) break;
            if (lane == 0) issue_tile(sb, rp.idx);
            __syncwarp();
            last[rp.idx] = (int)rp.phase;
            rp.next();
        }
        if (!ok)
            for (int i = 0; i < C::NS; ++i)
                if (last[i] >= 0) mbar_wait_bounded(full + i, (uint32_t)last[i]);
    } else {
        // compute warps: row tile rw of the CTA, stages sb = kg (mod KS)
        const int rw = warp % SQ_NW, kg = warp / SQ_NW;
        const int g = lane >> 2, t = lane & 3;
        // Q4_0: nibble e to the fp16 e - 8 (low nibbles: 1024 + e - 1032;
        // high nibbles: (1024 + 16 e) / 16 - 72)
        const uint4 k40 = make_uint4(pack_h2(1.0f, 1.0f), pack_h2(-1032.0f, -1032.0f), pack_h2(0.0625f, 0.0625f),
                                     pack_h2(-72.0f, -72.0f));
        float yacc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) yacc[n][e] = 0.0f;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int kc = min(C::KC, nsb - c * C::KC);
            if (!(ok = tc::wait_warp(cfull + (c & 1), (uint32_t)(c >> 1) & 1u, abort))) break;
            const uint8_t *buf = smem + C::OFF_CHUNK + (c & 1) * C::CHUNK;
            const uint4 *bf = reinterpret_cast<const uint4 *>(buf);
            const float *cf = reinterpret_cast<const float *>(buf + C::BFRAG);
            for (int sbk = 0; sbk < kc && ok; ++sbk) {
                const int sb = c * C::KC + sbk;
                if (sb % C::KS != kg) continue;
                const int si = sb % C::NS;
                if (!(ok = tc::wait_warp(full + si, (uint32_t)(sb / C::NS) & 1u, abort))) break;
                const uint8_t *rg = smem + C::OFF_RING + si * C::STAGE + (16 * rw + g) * C::ROWB;
                const uint8_t *rh = rg + 8 * C::ROWB;
#pragma unroll 2
                for (int j = 0; j < 8; ++j) {
                    const uint32_t ob = (uint32_t)(j * C::BB);
                    uint4 ag, ah;
                    if (C::Q4) {
                        ag = nib8_to_f16(load4_even(rg, ob + 2 + 4 * t), k40);
                        ah = nib8_to_f16(load4_even(rh, ob + 2 + 4 * t), k40);
                    } else {
                        const uint2 cg = load8_even(rg, ob + 2 + 8 * t), ch = load8_even(rh, ob + 2 + 8 * t);
                        ag = i8x8_to_f16(cg.x, cg.y);
                        ah = i8x8_to_f16(ch.x, ch.y);
                    }
                    const float dg = half_bits_to_float(*reinterpret_cast<const uint16_t *>(rg + ob));
                    const float dh = half_bits_to_float(*reinterpret_cast<const uint16_t *>(rh + ob));
                    const int jj = sbk * 8 + j;  // block of the chunk
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint4 b = bf[(n * C::KC * 8 + jj) * 32 + lane];
                        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        mma16816(s, ag.x, ah.x, ag.y, ah.y, b.x, b.y);
                        mma16816(s, ag.z, ah.z, ag.w, ah.w, b.z, b.w);
                        const float2 dx = *reinterpret_cast<const float2 *>(cf + jj * C::BCOLS + 8 * n + 2 * t);
                        if (SUMS) {
                            const int rr[2] = {row0 + 16 * rw + g, row0 + 16 * rw + g + 8};
                            const int kb = sb * 8 + j;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int row = rr[e >> 1], bcol = 8 * n + 2 * t + (e & 1);
                                if (row < rows && bcol < batch)
                                    sums[((size_t)bcol * rows + row) * nblk + kb] = (int32_t)s[e];
                            }
                        } else {
                            yacc[n][0] = fmaf(dg * dx.x, s[0], yacc[n][0]);
                            yacc[n][1] = fmaf(dg * dx.y, s[1], yacc[n][1]);
                            yacc[n][2] = fmaf(dh * dx.x, s[2], yacc[n][2]);
                            yacc[n][3] = fmaf(dh * dx.y, s[3], yacc[n][3]);
                        }
                    }
                }
                // the stage is read; release it to the producer
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(empty + si);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(cempty + (c & 1));
        }
        if (!SUMS) {
            if (C::KS > 1) {
                // groups 1.. hand their partial y to group 0, which adds them
                // in group order; every compute warp reaches the barrier
                float4 *part = reinterpret_cast<float4 *>(smem + C::OFF_PART);
                if (kg > 0)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        part[(((kg - 1) * SQ_NW + rw) * NT + n) * 32 + lane] =
                            make_float4(yacc[n][0], yacc[n][1], yacc[n][2], yacc[n][3]);
                asm volatile("bar.sync 1, %0;" ::"r"(32 * C::NCW) : "memory");
                if (kg == 0)
                    for (int k = 1; k < C::KS; ++k)
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            const float4 v = part[(((k - 1) * SQ_NW + rw) * NT + n) * 32 + lane];
                            yacc[n][0] += v.x;
                            yacc[n][1] += v.y;
                            yacc[n][2] += v.z;
                            yacc[n][3] += v.w;
                        }
            }
            if (kg == 0 && !*abort) {
                const int rg = row0 + 16 * rw + g;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int row = rg + 8 * (e >> 1), bcol = 8 * n + 2 * t + (e & 1);
                        if (row < rows && bcol < batch) y[(size_t)bcol * rows + row] = yacc[n][e];
                    }
            }
        }
    }
    pdl_launch_dependents();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) atomicOr(status, STATUS_MMA_TIMEOUT);
}

template <int WT, int NT>
cudaError_t launch_nt(const CUtensorMap &tmap, const void *xq, float *y, int32_t *sums, int64_t rows, int nsb,
                      int64_t batch, bool w_static, const LaunchCtx &ctx) {
    using C = SqCfg<WT, NT>;
    auto k = sums ? skinny_q0_kernel<WT, NT, true> : skinny_q0_kernel<WT, NT, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((rows + SQ_ROWS - 1) / SQ_ROWS));
    return launch_pdl(k, grid, dim3(C::THREADS), C::SMEM_ALLOC, ctx.stream, tmap,
                      static_cast<const uint8_t *>(xq), y, sums, (int)rows, nsb, (int)batch, w_static ? 1 : 0,
                      ctx.status);
}

template <int WT>
cudaError_t launch_wt(const CUtensorMap &tmap, const void *xq, float *y, int32_t *sums, int64_t rows, int nsb,
                      int64_t batch, bool w_static, const LaunchCtx &ctx) {
    switch (pick_nt(batch)) {
    case 1: return launch_nt<WT, 1>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    case 2: return launch_nt<WT, 2>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    case 4: return launch_nt<WT, 4>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    default: return launch_nt<WT, 8>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    }
}

}  // namespace

bool skinny_q0_supported(int64_t rows, int64_t cols, int64_t batch) {
    return rows >= 1 && batch >= 1 && batch <= 64 && cols >= QK_K && cols % QK_K == 0 &&
           (rows + SQ_ROWS - 1) / SQ_ROWS <= 0x7fffffff;
}

cudaError_t launch_skinny_q0(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                             int64_t cols, int64_t batch, bool w_static, const LaunchCtx &ctx) {
    if (!skinny_q0_supported(rows, cols, batch) || (wtype != GQ_Q4_0 && wtype != GQ_Q8_0))
        return cudaErrorInvalidValue;
    const int nsb = (int)(cols / QK_K);
    const int bb = wtype == GQ_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmap;
    // W as a 2-D tensor of 16-bit elements (a box edge holds at most 256
    // elements; eight Q8_0 blocks are 272 bytes): rows of cols / 32 blocks;
    // box = eight blocks of 96 rows (a multiple of 16 bytes, as is the row
    // pitch for cols % 256 == 0)
    const cuuint64_t gdim[2] = {(cuuint64_t)nsb * 4 * bb, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)nsb * 8 * bb};
    const cuuint32_t box[2] = {(cuuint32_t)(4 * bb), (cuuint32_t)SQ_ROWS};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(W), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return wtype == GQ_Q4_0 ? launch_wt<GQ_Q4_0>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx)
                            : launch_wt<GQ_Q8_0>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
}

}  // namespace gq
