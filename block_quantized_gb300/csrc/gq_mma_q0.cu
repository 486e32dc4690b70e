// gq_mma_q0.cu -- batched Q4_0 / Q8_0 x Q8_0 product on the 5th-generation
// tensor cores, for batches large enough that the product is a dense
// contraction ("llama.cpp 推理引擎" §7.3).
//
// The product is the per-block one of "llama.cpp 推理引擎" §5.3-5.4 / §6.4:
//   y[b][r] = sum_k d_w(r, k) * d_x(b, k) * S(r, b, k),
//   S(r, b, k) = sum_{i < 32} w_i * a_i,
// w_i = c_i - 8 (Q4_0) or the int8 code (Q8_0), a_i the int8 Q8_0 code of
// the activation, d_w and d_x the two blocks' fp16 scales.
//
// Each block's integer dot runs on the fp16 MMA kind (sm_103a has no integer
// kind) with the codes as exactly representable small integers, into an
// accumulator of its own: two K = 16 steps that start from zero, so
// |S| <= 32 * 128 * 128 = 2^19 and the fp32 accumulation is exact in any
// order.  The epilogue applies the two scales in fp32 registers.
//
// No workspace: both operands are converted inside the kernel.  Per stage a
// 2-D TMA load brings 8 blocks (256 elements) of the 128 weight rows and of
// the TN activation columns into shared memory as raw block bytes; builder
// warps turn each pair of blocks into fp16 operands -- the weight codes into
// tensor memory (tcgen05.st, the MMA's A operand), the activation codes into
// a 128-byte-swizzled K-major tile (the B operand) -- and write the two
// blocks' scales for the epilogue.  Within every 8-element group both
// operands use the order (e0, e4, e1, e5, e2, e6, e3, e7), the order in
// which a Q4_0 nibble word unpacks; a block's dot does not depend on it.
//
// CTA tile: 128 weight rows x TN batch columns (TN = 32, 64 or 128, the
// narrowest that covers the batch), 28 warps:
//   warp 0      raw-tile producer (2-D TMA, NRAW stages);
//   warp 1      MMA issuer (one thread) and tensor-memory owner;
//   warps 4-11  builders: warp w converts block (w - 4) / 4 of every pair for
//               tile rows / columns 32 (w % 4) .. + 31;
//   warps 12-27 epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
//               (its rows) and columns 32 h .. + 31, h = (w - 12) / 4, of
//               each block's accumulator (warps whose columns lie past TN
//               idle).
// Tensor memory (512 columns): NOP A buffers of one pair of blocks (64 K as
// fp16 pairs = 32 columns each) at the top, below them NACC accumulators of
// TN columns in a ring, one per block.
//
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// bit and an abort flag that stops all roles of the CTA, which then drains its
// transfers and frees tensor memory before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_tc.cuh"

namespace gq {
namespace {

using namespace tc;

constexpr int TM = 128;         // weight rows per tile (MMA M)
constexpr int G = 8;            // blocks per raw stage (256 elements, 16-byte aligned rows)
constexpr int PPS = G / 2;      // pairs of blocks per raw stage
constexpr int NOP = 3;          // operand buffers (pairs of blocks)
constexpr int NSC = 4;          // scale slots (pairs of blocks)
constexpr int NTHREADS = 896;
constexpr int BLD_WARP0 = 4, BLD_WARPS = 8, EPI_WARP0 = 12;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_A0 = TMEM_COLS - 32u * NOP;  // A buffers at the top of tensor memory
constexpr int SMEM_LIMIT = 232448;                  // opt-in dynamic shared memory per CTA

template <int WT_, int TN_>
struct Cfg {
    static constexpr int WT = WT_, TN = TN_;
    static constexpr int BB = WT_ == GQ_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES;  // weight block bytes
    static constexpr int RAW_W = TM * G * BB;          // raw weight rows of one stage
    static constexpr int RAW_X = TN_ * G * Q8_0_BYTES; // raw activation columns of one stage
    static constexpr int RAW_STAGE = RAW_W + RAW_X;
    static constexpr int OP_B = TN_ * 128;             // B tile of a pair: TN rows x 64 fp16
    // scales of a pair: d_w of both blocks for the 128 rows, then d_x of both
    // blocks for the TN columns (fp32)
    static constexpr int SC_DW = 0, SC_DX = 2 * TM * 4;
    static constexpr int SC_SLOT = 2 * TM * 4 + 2 * TN_ * 4;
    static constexpr int NACC = (int)(COL_A0 / (uint32_t)TN_);
    static constexpr int NBARS_FIXED = 2 * NOP + 2 * NACC + 2 * NSC + 1;
    static constexpr int OFF_B = 0;                                     // NOP x OP_B (1024-aligned)
    static constexpr int OFF_RAW = OFF_B + NOP * OP_B;
    static constexpr int BASE = OFF_RAW + NSC * SC_SLOT + (NBARS_FIXED + 8) * 8 + 16 + 1024;
    // as many raw stages as fit (2 to 4)
    static constexpr int NRAW = BASE + 4 * RAW_STAGE <= SMEM_LIMIT ? 4 : (BASE + 3 * RAW_STAGE <= SMEM_LIMIT ? 3 : 2);
    static constexpr int OFF_SC = OFF_RAW + NRAW * RAW_STAGE;
    static constexpr int OFF_BAR = OFF_SC + NSC * SC_SLOT;
    static constexpr int NBARS = 2 * NRAW + NBARS_FIXED;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for the 1024-byte alignment
    static constexpr int EPI_ACTIVE = 4 * (TN_ / 32);    // epilogue warps that own columns
    static constexpr uint32_t IDESC = idesc_f16(TM, TN_, 0);
    __host__ __device__ static constexpr uint32_t col_acc(int i) { return (uint32_t)(TN_ * i); }
    __host__ __device__ static constexpr uint32_t col_a(int i) { return COL_A0 + 32u * (uint32_t)i; }
    static_assert(TN_ == 32 || TN_ == 64 || TN_ == 128, "tile widths");
    static_assert(NACC >= 2, "accumulator ring");
    static_assert(SMEM_ALLOC <= SMEM_LIMIT, "shared memory budget");
    static_assert(OP_B % 1024 == 0, "SW128 tiles need 1024-byte alignment");
    static_assert(OFF_RAW % 128 == 0 && RAW_W % 128 == 0 && RAW_STAGE % 128 == 0, "TMA destinations");
    static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
};

// Tile width for a batch: the narrowest tile that covers it, 128 beyond 64.
inline int pick_tn(int64_t batch) { return batch <= 32 ? 32 : (batch <= 64 ? 64 : 128); }

struct Bars {
    uint64_t *raw_full, *raw_empty, *op_full, *op_empty, *acc_full, *acc_empty, *sc_full, *sc_empty, *fin;
};

template <class C>
__device__ __forceinline__ Bars bars_at(uint8_t *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    Bars r;
    r.raw_full = b;
    r.raw_empty = r.raw_full + C::NRAW;
    r.op_full = r.raw_empty + C::NRAW;
    r.op_empty = r.op_full + NOP;
    r.acc_full = r.op_empty + NOP;
    r.acc_empty = r.acc_full + C::NACC;
    r.sc_full = r.acc_empty + C::NACC;
    r.sc_empty = r.sc_full + NSC;
    r.fin = r.sc_empty + NSC;
    return r;
}

// ------------------------------------------------------------ conversions

__device__ __forceinline__ __half2 h2_bits(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ uint32_t bits_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Eight int8 codes e0..e3 (bytes of u0) and e4..e7 (bytes of u1) to the fp16
// chunk (e0, e4, e1, e5, e2, e6, e3, e7).  A byte b ^ 0x80 in the mantissa
// of 0x6400 is the exact fp16 value 1024 + (b + 128); subtracting 1152
// leaves b exactly.
__device__ __forceinline__ uint4 i8x8_to_f16(uint32_t u0, uint32_t u1) {
    const uint32_t x0 = __byte_perm(u0, u1, 0x5140) ^ 0x80808080u;  // e0 e4 e1 e5
    const uint32_t x1 = __byte_perm(u0, u1, 0x7362) ^ 0x80808080u;  // e2 e6 e3 e7
    const __half2 bias = __float2half2_rn(-1152.0f);
    return make_uint4(bits_h2(__hadd2(h2_bits(__byte_perm(x0, 0x64646464u, 0x4140)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x0, 0x64646464u, 0x4342)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x1, 0x64646464u, 0x4140)), bias)),
                      bits_h2(__hadd2(h2_bits(__byte_perm(x1, 0x64646464u, 0x4342)), bias)));
}

// Eight Q4_0 codes of one nibble word (byte i: element 2i in the low, 2i + 1
// in the high nibble) to the fp16 chunk (c - 8) in the order (e0, e4, e1,
// e5, e2, e6, e3, e7).  A nibble in mantissa bits 0-3 (4-7) of 0x6400 is the
// exact fp16 1024 + c (1024 + 16 c); one fma with (1, -1032) -- or
// (1/16, -72) -- yields c - 8 exactly.
__device__ __forceinline__ uint4 nib8_to_f16(uint32_t w) {
    const uint32_t w8 = w >> 8;
    const __half2 one = __float2half2_rn(1.0f), sixteenth = __float2half2_rn(0.0625f);
    const __half2 c_lo = __float2half2_rn(-1032.0f), c_hi = __float2half2_rn(-72.0f);
    return make_uint4(bits_h2(__hfma2(h2_bits((w & 0x000F000Fu) | 0x64006400u), one, c_lo)),         // e0, e4
                      bits_h2(__hfma2(h2_bits((w & 0x00F000F0u) | 0x64006400u), sixteenth, c_hi)),   // e1, e5
                      bits_h2(__hfma2(h2_bits((w8 & 0x000F000Fu) | 0x64006400u), one, c_lo)),        // e2, e6
                      bits_h2(__hfma2(h2_bits((w8 & 0x00F000F0u) | 0x64006400u), sixteenth, c_hi)));  // e3, e7
}

// NW consecutive 32-bit words at byte offset OFF (even) of a 16-byte-aligned
// raw row: 16-byte shared loads of the aligned span, then a 16-bit funnel
// shift when OFF is not a multiple of four.  A tile's rows sit 144 or 272
// bytes apart (nine or seventeen 16-byte units), so the 16-byte loads of
// eight consecutive rows fall in distinct bank groups.
template <int NW, int OFF>
__device__ __forceinline__ void load_words(const uint8_t *row, uint32_t (&out)[NW]) {
    constexpr int BASE = OFF & ~15, SH = OFF & 15, WS = SH >> 2;
    constexpr int NCH = (SH + 4 * NW + 15) / 16;  // 16-byte chunks touched
    static_assert(SH % 2 == 0 && 4 * NCH >= WS + NW + ((SH & 2) ? 1 : 0), "span");
    uint32_t w[NCH * 4];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + BASE + 16 * c);
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        if constexpr ((SH & 2) != 0)
            out[i] = __funnelshift_r(w[WS + i], w[WS + i + 1], 16);
        else
            out[i] = w[WS + i];
    }
}

// Block BLK (0..7) of a raw stage for one tile row: its weight codes as
// fp16 chunks and its fp16 scale as fp32.
template <class C, int BLK>
__device__ __forceinline__ float convert_w(const uint8_t *raw_w, uint4 (&a)[4]) {
    if constexpr (C::WT == GQ_Q4_0) {
        uint32_t wd[4];
        load_words<4, BLK * Q4_0_BYTES + 2>(raw_w, wd);
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = nib8_to_f16(wd[m]);
    } else {
        uint32_t wd[8];
        load_words<8, BLK * Q8_0_BYTES + 2>(raw_w, wd);
#pragma unroll
        for (int m = 0; m < 4; ++m) a[m] = i8x8_to_f16(wd[2 * m], wd[2 * m + 1]);
    }
    return __half2float(*reinterpret_cast<const __half *>(raw_w + BLK * C::BB));
}

// The same for one tile column's Q8_0 activation block.
template <int BLK>
__device__ __forceinline__ float convert_x(const uint8_t *raw_x, uint4 (&b)[4]) {
    uint32_t xd[8];
    load_words<8, BLK * Q8_0_BYTES + 2>(raw_x, xd);
#pragma unroll
    for (int m = 0; m < 4; ++m) b[m] = i8x8_to_f16(xd[2 * m], xd[2 * m + 1]);
    return __half2float(*reinterpret_cast<const __half *>(raw_x + BLK * Q8_0_BYTES));
}

template <class C>
__device__ __forceinline__ float convert_w_blk(int blk, const uint8_t *raw_w, uint4 (&a)[4]) {
    switch (blk) {  // warp-uniform
    case 0: return convert_w<C, 0>(raw_w, a);
    case 1: return convert_w<C, 1>(raw_w, a);
    case 2: return convert_w<C, 2>(raw_w, a);
    case 3: return convert_w<C, 3>(raw_w, a);
    case 4: return convert_w<C, 4>(raw_w, a);
    case 5: return convert_w<C, 5>(raw_w, a);
    case 6: return convert_w<C, 6>(raw_w, a);
    default: return convert_w<C, 7>(raw_w, a);
    }
}

__device__ __forceinline__ float convert_x_blk(int blk, const uint8_t *raw_x, uint4 (&b)[4]) {
    switch (blk) {  // warp-uniform
    case 0: return convert_x<0>(raw_x, b);
    case 1: return convert_x<1>(raw_x, b);
    case 2: return convert_x<2>(raw_x, b);
    case 3: return convert_x<3>(raw_x, b);
    case 4: return convert_x<4>(raw_x, b);
    case 5: return convert_x<5>(raw_x, b);
    case 6: return convert_x<6>(raw_x, b);
    default: return convert_x<7>(raw_x, b);
    }
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint4 (&v)[4]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z),
        "r"(v[1].w), "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y),
        "r"(v[3].z), "r"(v[3].w)
        : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes; the
// wait sits in the same statement, so the outputs are complete when used.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// One MMA with the A operand in tensor memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------------------ roles

// Raw-tile producer (warp 0): per stage one 2-D TMA load of the 128 weight
// rows' 8 blocks (rows past the matrix read as zeros) and one of the TN
// activation columns' 8 blocks (columns past the batch read as zeros), onto
// one barrier.  On abort it waits (bounded) for every load it started.
template <class C>
__device__ void role_producer(uint8_t *smem, const Bars &B, const CUtensorMap *tmap_w,
                              const CUtensorMap *tmap_x, int row0, int col0, int nst, int rot,
                              volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    int last[C::NRAW];
    for (int i = 0; i < C::NRAW; ++i) last[i] = -1;
    RingPos rr(C::NRAW);
    bool ok = true;
    for (int i = 0; ok && i < nst; ++i) {
        if (!(ok = wait_warp(B.raw_empty + rr.idx, rr.phase ^ 1u, abort))) break;
        if (lane == 0) {
            const int g = kslot(i, rot, nst);
            uint8_t *dst = smem + C::OFF_RAW + rr.idx * C::RAW_STAGE;
            mbar_arrive_expect_tx(B.raw_full + rr.idx, C::RAW_STAGE);
            // x coordinates in 16-bit elements: 8 blocks of BB (34) bytes per stage
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
                "l"(reinterpret_cast<uint64_t>(tmap_w)), "r"(g * (G * C::BB / 2)), "r"(row0),
                "r"(smem_u32(B.raw_full + rr.idx))
                : "memory");
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst + C::RAW_W)),
                "l"(reinterpret_cast<uint64_t>(tmap_x)), "r"(g * (G * Q8_0_BYTES / 2)), "r"(col0),
                "r"(smem_u32(B.raw_full + rr.idx))
                : "memory");
        }
        __syncwarp();
        last[rr.idx] = (int)rr.phase;
        rr.next();
    }
    if (!ok)
        for (int i = 0; i < C::NRAW; ++i)
            if (last[i] >= 0) mbar_wait_bounded(B.raw_full + i, (uint32_t)last[i]);
}

// Builders (warps 4-11).  Warp w handles block j = (w - 4) / 4 of every pair
// for tile rows t = 32 (w % 4) + lane (its tensor-memory lanes) and, when
// t < TN, tile column t: the row's 32 weight codes as fp16 A columns
// 16 j .. 16 j + 15 of the pair's A buffer, the column's 32 activation codes
// as K groups 4 j .. 4 j + 3 of the pair's B tile, and both scales.
template <class C>
__device__ void role_builder(uint8_t *smem, const Bars &B, uint32_t tmem, int nst, volatile uint32_t *abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = 32 * (warp & 3) + lane, j = (warp - BLD_WARP0) >> 2;
    const bool has_col = t < C::TN;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    RingPos rr(C::NRAW), orr(NOP), sr(NSC);
    for (int i = 0; i < nst; ++i) {
        if (!wait_warp(B.raw_full + rr.idx, rr.phase, abort)) return;
        const uint8_t *raw_w = smem + C::OFF_RAW + rr.idx * C::RAW_STAGE + t * (G * C::BB);
        const uint8_t *raw_x = smem + C::OFF_RAW + rr.idx * C::RAW_STAGE + C::RAW_W + t * (G * Q8_0_BYTES);
#pragma unroll 1
        for (int q = 0; q < PPS; ++q) {
            const int blk = 2 * q + j;  // block of the stage
            // the pair's operand buffers and scale slot are free once the MMAs
            // (op) and the epilogue (scales) of the pair NOP / NSC back are done
            if (!wait_warp(B.op_empty + orr.idx, orr.phase ^ 1u, abort)) return;
            if (!wait_warp(B.sc_empty + sr.idx, sr.phase ^ 1u, abort)) return;
            tc_fence_after();
            uint8_t *sc = smem + C::OFF_SC + sr.idx * C::SC_SLOT;
            {
                uint4 a[4];
                reinterpret_cast<float *>(sc + C::SC_DW)[j * TM + t] = convert_w_blk<C>(blk, raw_w, a);
                tmem_st16(lane_base + C::col_a(orr.idx) + 16u * (uint32_t)j, a);
            }
            if (has_col) {
                uint4 b[4];
                reinterpret_cast<float *>(sc + C::SC_DX)[j * C::TN + t] = convert_x_blk(blk, raw_x, b);
                uint8_t *bt = smem + C::OFF_B + orr.idx * C::OP_B;
#pragma unroll
                for (int m = 0; m < 4; ++m) *reinterpret_cast<uint4 *>(bt + sw128_off(t, 4 * j + m)) = b[m];
            }
            if (q == PPS - 1) {
                // the stage's bytes are all read
                __syncwarp();
                if (lane == 0) mbar_arrive(B.raw_empty + rr.idx);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B.op_full + orr.idx);
                mbar_arrive(B.sc_full + sr.idx);
            }
            orr.next();
            sr.next();
        }
        rr.next();
    }
}

// MMA issuer (warp 1, one thread).  Per pair, once both blocks' operands are
// built: per block, once its accumulator slot is drained, two K = 16 steps
// into it (the first from zero) and a commit that hands the slot to the
// epilogue; then a commit that frees the pair's operand buffers.  Always
// ends with a commit to `fin`.
template <class C>
__device__ void role_mma(uint8_t *smem, const Bars &B, uint32_t tmem, int npairs, volatile uint32_t *abort) {
    RingPos orr(NOP), ar(C::NACC);
    bool ok = true;
    for (int p = 0; ok && p < npairs; ++p) {
        if (!(ok = wait_or_abort(B.op_full + orr.idx, orr.phase, abort))) break;
        const uint64_t b0 = desc_sw128(smem_u32(smem + C::OFF_B + orr.idx * C::OP_B));
        const uint32_t a0 = tmem + C::col_a(orr.idx);
        for (int j = 0; j < 2; ++j) {
            if (!(ok = wait_or_abort(B.acc_empty + ar.idx, ar.phase ^ 1u, abort))) break;
            tc_fence_after();
            const uint32_t d = tmem + C::col_acc(ar.idx);
            // K step s of block j: A columns 16 j + 8 s, B start + 32 (2 j + s) bytes
            mma_f16_ta(d, a0 + 16u * j, b0 + 4u * j, C::IDESC, 0u);
            mma_f16_ta(d, a0 + 16u * j + 8u, b0 + 4u * j + 2u, C::IDESC, 1u);
            mma_commit(B.acc_full + ar.idx);
            ar.next();
        }
        if (!ok) break;
        mma_commit(B.op_empty + orr.idx);
        orr.next();
    }
    mma_commit(B.fin);
}

// Epilogue (warps 12-27): warp w owns rows 32 (w % 4) .. + 31 and columns
// 32 h .. + 31, h = (w - 12) / 4.  Per block: the accumulator into registers,
// the slot released, then y += d_x * (d_w * S) for its 32 columns (or, with
// SUMS, S written out as int32).
template <class C, bool SUMS>
__device__ void role_epilogue(uint8_t *smem, const Bars &B, uint32_t tmem, int row0, int rows, int col0,
                              int nst, int rot, int nblk, int batch, float *__restrict__ y,
                              int32_t *__restrict__ sums, volatile uint32_t *abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lq = warp & 3, h = (warp - EPI_WARP0) >> 2;
    if (32 * h >= C::TN) return;
    const int r = lq * 32 + lane;
    const int row = row0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(32 * h);
    float2 yacc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) yacc[c] = make_float2(0.0f, 0.0f);
    RingPos ar(C::NACC), sr(NSC);
    for (int i = 0; i < nst; ++i) {
        const int g = kslot(i, rot, nst);
        for (int q = 0; q < PPS; ++q) {
            if (!wait_warp(B.sc_full + sr.idx, sr.phase, abort)) return;
            const uint8_t *sc = smem + C::OFF_SC + sr.idx * C::SC_SLOT;
            for (int j = 0; j < 2; ++j) {
                if (!wait_warp(B.acc_full + ar.idx, ar.phase, abort)) return;
                tc_fence_after();
                const int blk = G * g + 2 * q + j;
                // SUMS: element (b, row, blk), column b = col0 + 32 h + c
                int32_t *sbase = SUMS ? sums + ((size_t)(col0 + 32 * h) * rows + row) * nblk + blk : nullptr;
                const size_t sstride = (size_t)rows * nblk;
                const float dw = reinterpret_cast<const float *>(sc + C::SC_DW)[j * TM + r];
                const float4 *dx4 = reinterpret_cast<const float4 *>(sc + C::SC_DX) + (j * C::TN + 32 * h) / 4;
                // the accumulator in two halves of 16 columns; the slot is
                // released once the second half is in registers
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float s[16];
                    tmem_ld16(lane_addr + C::col_acc(ar.idx) + 16u * hf, s);
                    if (hf == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(B.acc_empty + ar.idx);
                    }
                    if constexpr (SUMS) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            if (row < rows && col0 + 32 * h + 16 * hf + c < batch)
                                sbase[(16 * hf + c) * sstride] = (int32_t)s[c];
                    } else {
                        // y += d_x * (d_w * S), two fp32 lanes per instruction
                        // (each lane rounded as its scalar form)
                        const float2 dw2 = make_float2(dw, dw);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const float4 dx = dx4[4 * hf + c4];
                            const int k = 8 * hf + 2 * c4;
                            yacc[k] = __ffma2_rn(make_float2(dx.x, dx.y), __fmul2_rn(make_float2(s[4 * c4], s[4 * c4 + 1]), dw2),
                                           yacc[k]);
                            yacc[k + 1] = __ffma2_rn(make_float2(dx.z, dx.w),
                                               __fmul2_rn(make_float2(s[4 * c4 + 2], s[4 * c4 + 3]), dw2), yacc[k + 1]);
                        }
                    }
                }
                ar.next();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B.sc_empty + sr.idx);
            sr.next();
        }
    }
    if constexpr (!SUMS) {
        if (row >= rows) return;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int b = col0 + 32 * h + 2 * c;
            if (b < batch) y[(size_t)b * rows + row] = yacc[c].x;
            if (b + 1 < batch) y[(size_t)(b + 1) * rows + row] = yacc[c].y;
        }
    }
}

template <int WT, int TN, bool SUMS>
__global__ void __launch_bounds__(NTHREADS, 1) mma_q0_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                             const __grid_constant__ CUtensorMap tmap_x,
                                                             float *__restrict__ y, int32_t *__restrict__ sums,
                                                             int rows, int nblk, int batch,
                                                             uint32_t *__restrict__ status) {
    using C = Cfg<WT, TN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Bars B = bars_at<C>(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // column tiles vary fastest, so the CTAs that read the same weight rows
    // run together and share them through L2
    const int row0 = blockIdx.y * TM, col0 = blockIdx.x * TN;
    const int nst = nblk / G;
    const int rot = (int)(blockIdx.y % (unsigned)nst);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NRAW; ++i) {
            mbar_init(B.raw_full + i, 1);
            mbar_init(B.raw_empty + i, BLD_WARPS);
        }
        for (int i = 0; i < NOP; ++i) {
            mbar_init(B.op_full + i, BLD_WARPS);
            mbar_init(B.op_empty + i, 1);
        }
        for (int i = 0; i < C::NACC; ++i) {
            mbar_init(B.acc_full + i, 1);
            mbar_init(B.acc_empty + i, C::EPI_ACTIVE);
        }
        for (int i = 0; i < NSC; ++i) {
            mbar_init(B.sc_full + i, BLD_WARPS);
            mbar_init(B.sc_empty + i, C::EPI_ACTIVE);
        }
        mbar_init(B.fin, 1);
        *abort = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the activations (and W) may come from the preceding kernel

    if (warp == 0) {
        role_producer<C>(smem, B, &tmap_w, &tmap_x, row0, col0, nst, rot, abort);
    } else if (warp == 1) {
        if (lane == 0) role_mma<C>(smem, B, tmem, nst * PPS, abort);
        __syncwarp();
    } else if (warp >= BLD_WARP0 && warp < BLD_WARP0 + BLD_WARPS) {
        role_builder<C>(smem, B, tmem, nst, abort);
    } else if (warp >= EPI_WARP0) {
        role_epilogue<C, SUMS>(smem, B, tmem, row0, rows, col0, nst, rot, nblk, batch, y, sums, abort);
    }
    pdl_launch_dependents();

    // teardown: every MMA has completed once `fin` fired (bounded wait), then
    // tensor memory is freed by the warp that allocated it
    if (warp == 1) {
        if (lane == 0) mbar_wait_bounded(B.fin, 0u);
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) atomicOr(status, STATUS_MMA_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// 2-D map of a matrix of `nrows` rows of nblk blocks of `bb` bytes, as
// 16-bit elements; box = 8 blocks x `box_rows` rows.
bool encode_map(CUtensorMap *map, const void *base, int64_t nrows, int64_t nblk, int bb, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)(nblk * bb / 2), (cuuint64_t)nrows};
    const cuuint64_t gstride[1] = {(cuuint64_t)(nblk * bb)};
    const cuuint32_t box[2] = {(cuuint32_t)(G * bb / 2), (cuuint32_t)box_rows};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WT, int TN>
cudaError_t launch_tiles(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t nblk,
                         int64_t batch, const LaunchCtx &ctx) {
    using C = Cfg<WT, TN>;
    CUtensorMap tw, tx;
    if (!encode_map(&tw, W, rows, nblk, C::BB, TM) || !encode_map(&tx, xq, batch, nblk, Q8_0_BYTES, TN))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((batch + TN - 1) / TN), (unsigned)((rows + TM - 1) / TM));
    auto k = sums ? mma_q0_kernel<WT, TN, true> : mma_q0_kernel<WT, TN, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, grid, dim3(NTHREADS), C::SMEM_ALLOC, ctx.stream, tw, tx, y, sums, (int)rows, (int)nblk,
                      (int)batch, ctx.status);
}

template <int WT>
cudaError_t launch_type(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t nblk,
                        int64_t batch, const LaunchCtx &ctx) {
    switch (pick_tn(batch)) {
    case 32: return launch_tiles<WT, 32>(W, xq, y, sums, rows, nblk, batch, ctx);
    case 64: return launch_tiles<WT, 64>(W, xq, y, sums, rows, nblk, batch, ctx);
    default: return launch_tiles<WT, 128>(W, xq, y, sums, rows, nblk, batch, ctx);
    }
}

}  // namespace

bool mma_q0_supported(int64_t rows, int64_t cols, int64_t batch) {
    return rows >= 1 && batch >= 1 && cols >= 256 && cols % 256 == 0 && (rows + TM - 1) / TM <= 65535 &&
           (batch + 31) / 32 <= 0x7fffffff;
}

cudaError_t launch_mma_q0(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                          int64_t cols, int64_t batch, const LaunchCtx &ctx) {
    if (!mma_q0_supported(rows, cols, batch)) return cudaErrorInvalidValue;
    const int64_t nblk = cols / 32;
    if (wtype == GQ_Q4_0) return launch_type<GQ_Q4_0>(W, xq, y, sums, rows, nblk, batch, ctx);
    if (wtype == GQ_Q8_0) return launch_type<GQ_Q8_0>(W, xq, y, sums, rows, nblk, batch, ctx);
    return cudaErrorInvalidValue;
}

}  // namespace gq

