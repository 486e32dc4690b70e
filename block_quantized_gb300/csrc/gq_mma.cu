// gq_mma.cu -- batched Q4_K x Q8_K product on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), for batches large enough that
// the product is a dense contraction ("llama.cpp 推理引擎" §7.3: prompt
// processing is compute-bound, token generation bandwidth-bound).
//
// sm_103a has no integer MMA kind, so the contraction runs on the fp16 kind
// with operands that are small integers, exactly representable in fp16:
//   A[r][k] = sc_j(r) * q_k(r) - 512  (in [-512, 433])
//   B[b][k] = a_k(b)                  (|a| <= 127, the Q8_K code)
// Every product is exact (|A * B| <= 65024) and every partial sum of one
// 256-element super-block is an integer of magnitude at most
// 256 * 512 * 127 = 16,646,144 < 2^24, so the fp32 accumulation is exact in
// any order.  (Without the offset, sc * q * a reaches 945 * 127 and a
// super-block sum 3.07e7 > 2^24, where fp32 keeps only even integers.)  The
// epilogue restores the integer S1 = sum_j sc_j * s_j of "llama.cpp 推理引擎"
// §5.5's two-level scheme as
//   S1 = S1' + 512 * asum(b),   asum(b) = sum of the super-block's 256 codes,
// asum being stored per column and super-block by the pack kernel
// (|S1| <= 3.07e7: one int32 add, or one fp32 fma that rounds the exact S1
// once).  The min-term integer S2 = sum_j m_j * t_j (t_j the activation
// sub-block sums) is one more K=16 step per super-block, with t_j split
// exactly as t_lo + 64 t_hi:
//   A2[r] = [m_0..m_7 | 64 m_0..64 m_7]   B2[b] = [t_lo_0..t_lo_7 | t_hi_0..t_hi_7]
// (all exact in fp16, |S2| < 2^21).  Per super-block the epilogue promotes
// both exact integers:
//   y[b][r] += dx(b) * (d(r) * S1 - dmin(r) * S2)      (fp32, in registers)
//
// CTA tile: 128 weight rows x TN batch columns, one super-block (K = 256) per
// step, 28 warps:
//   warps 0, 3 activation producers: one bulk copy each per super-block of
//              the packed unit's half 0 (B stages 0-1) or half 1 (stages 2-3
//              and the min-term B tile) into a ring of NBSB super-blocks
//              (4 / 3 / 2 for TN = 32 / 64 / 128);
//   warp 1     MMA issuer (one thread) and tensor-memory owner;
//   warp 2     weight producer: one 2-D tiled TMA load per super-block of
//              the raw Q4_K rows into a ring of NRAW stages (box 144 bytes x
//              128 rows; rows past the matrix read as zeros);
//   warps 4-11 A builders: two threads per weight row, each turning half of
//              the raw super-block into fp16 sc*q - 512 and storing it straight
//              from registers into tensor memory (tcgen05.st), where the MMA
//              reads the A operand; then the min-term row (first half) or
//              the row scales, column scales and column code sums
//              (second half);
//   warps 12-27 epilogue: four threads per row, 32 columns each (the warps
//              whose columns lie past TN idle).
// Per super-block a ready barrier (A and min-term rows built, the S1 buffer
// of its parity released by the epilogue) and a done
// barrier (one commit after its MMAs, which frees its S1/S2 for the
// epilogue and its activation slots and min-term rows for reuse), in a ring.
// Tensor memory (512 columns): the S1 accumulator, double-buffered by
// super-block, and two or three buffers of the A operand.  The min-term step
// writes S2 over the A buffer its super-block has just consumed, so the
// builders run one or two super-blocks ahead of the MMAs and the MMAs a
// super-block ahead of the epilogue.
// The tile width TN (32, 64 or 128 batch columns) is chosen per call: the
// narrowest that covers the batch, 128 beyond 64.
// The activation operand is packed once per call by pack_kernel into a
// caller-provided workspace, already in the swizzled shared-memory image, so
// each operand tile is a single 1-D bulk copy.
//
// Every mbarrier wait is bounded; a wait that gives up sets the device status
// bit and an abort flag that stops all roles of the CTA, which then drains its
// transfers and frees tensor memory before exiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_mma_sync.cuh"
#include "gq_tc.cuh"

namespace gq {
namespace {

using namespace tc;

constexpr int TM = 128;   // weight rows per tile (MMA M)
constexpr int KS = 64;    // K per B operand stage (one 128-byte swizzle atom)
constexpr int NKS = 4;    // B operand stages per super-block
constexpr int KMIN = 16;  // min-term K per super-block (8 mins, two halves of t)
constexpr int NSM = 4;    // ring depth of the per-super-block scales and min-term A rows
constexpr int NF = 4;     // ring of per-super-block ready / done barriers (= NSM)
static_assert(NF == NSM, "the min-term rows share the ready/done ring");
constexpr int MIN_A = TM * KMIN * 2;           // 4 KB min-term A rows
constexpr int RAW_STAGE = TM * Q4_K_BYTES;     // 18 KB raw weight rows
constexpr int NTHREADS = 896;
constexpr int EPI_WARP0 = 12, EPI_WARPS = 16, BLD_WARP0 = 4, BLD_THREADS = 256;

// Tensor memory (512 columns): the S1 accumulator double-buffered by
// super-block parity (2 x TN columns from 0), and NA buffers of the A operand
// (one super-block, 256 K as fp16 pairs = 128 columns each) from column
// COL_A0, used in turn.  Once the sixteen S1 steps of a super-block have read
// its A buffer, the min-term step writes S2 over it (the tensor core executes
// one thread's MMAs in issue order), and the epilogue frees the buffer for
// the builders when it has read S2.  Tiles of up to 64 columns leave room for
// a third A buffer, so the builders may run two super-blocks ahead of the
// MMAs.
constexpr uint32_t TMEM_COLS = 512;

// ------------------------------------------------------------ tcgen05 helpers

// Shared-memory matrix descriptor, K-major, no swizzle: 8x16-byte core
// matrices, `lbo` bytes apart along K and `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// Tile-width configuration.  A CTA computes TM weight rows x TN batch
// columns (MMA N = TN).  Per (column tile, super-block) the workspace holds
// one unit: the four B stage images (TN x 64 K fp16, 128-byte swizzled), the
// min-term B tile, the column scales and the column code sums (fp32),
// contiguous.  Each unit arrives as two bulk copies, issued by two producer
// warps (a warp completes about one bulk copy per half microsecond however
// large, so one copy per warp per super-block keeps the copies off the
// critical path): half 0 = stages 0-1; half 1 = stages 2-3 and the min-term
// B tile.  The column scales and code sums are fetched by builder threads
// with plain loads.  Narrow tiles (small batches) move
// little activation data per super-block, so their period is set by the
// weight rows; they get deeper activation (NBSB super-blocks) and weight
// (NRAW) rings to cover the copy latency.
template <int TN_>
struct Cfg {
    static constexpr int TN = TN_;
    static constexpr int NBSB = TN_ == 32 ? 4 : (TN_ == 64 ? 3 : 2);
    static constexpr int NBS = 2 * NBSB;   // B ring slots: two halves per super-block
    static constexpr int NRAW = TN_ == 32 ? 6 : (TN_ == 64 ? 4 : 3);
    // tensor memory: S1 buffers at 0 and TN, A buffers from COL_A0
    static constexpr int NA = TN_ <= 64 ? 3 : 2;
    static constexpr uint32_t COL_A0 = TN_ <= 64 ? 128u : 256u;
    static constexpr int OP_B = TN * KS * 2;                       // one B stage
    static constexpr int MIN_B = TN * KMIN * 2;
    static constexpr size_t WS_B = (size_t)NKS * OP_B;
    static constexpr size_t WS_MIN = MIN_B;
    static constexpr size_t WS_DX = TN * 4;
    static constexpr size_t WS_AS = TN * 4;   // per column: sum of the super-block's 256 codes
    static constexpr size_t WS_UNIT = WS_B + WS_MIN + WS_DX + WS_AS;
    static constexpr int HALF0_BYTES = 2 * OP_B;
    static constexpr int HALF1_BYTES = 2 * OP_B + MIN_B;
    static constexpr int SLOT_B = (HALF1_BYTES + 1023) / 1024 * 1024;  // ring slot stride
    static constexpr int SLOT_MIN = 2 * OP_B;                          // inside a half-1 slot
    // per super-block scales: d and dmin per row; per column the pair
    // (dx, 512 * code sum) (all fp32; 512 times a code sum is an integer
    // below 2^24 in magnitude, exact)
    static constexpr int META_D = 0, META_DMIN = TM * 4, META_COL = 2 * TM * 4;
    static constexpr int META_STAGE = 2 * TM * 4 + 2 * TN * 4;
    // Shared-memory layout (bytes from a 1024-aligned base).  The A operand
    // lives in tensor memory, not here.
    static constexpr int OFF_B = 0;                               // NBS x SLOT_B
    static constexpr int OFF_MINA = OFF_B + NBS * SLOT_B;         // NSM x 4 KB min-term A rows
    static constexpr int OFF_RAW = OFF_MINA + NSM * MIN_A;        // NRAW x 18 KB
    static constexpr int OFF_META = OFF_RAW + NRAW * RAW_STAGE;   // NSM scale stages
    static constexpr int OFF_BAR = OFF_META + NSM * META_STAGE;
    // per super-block ready (A and min-term rows built, S1 buffer free) and
    // done (all its MMAs complete), A empty, B tx, raw full/empty, meta
    // full/empty, final.
    static constexpr int NBARS = 2 * NF + NA + NBS + 2 * NRAW + 2 * NSM + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for the 1024-byte alignment
    // epilogue warps that own columns (four per 32 columns)
    static constexpr int EPI_ACTIVE = 4 * (TN / 32);
    // epilogue warps with no columns: they pack the activations when there is
    // no workspace (tiles of up to 64 columns)
    static constexpr int NPACK = 16 - EPI_ACTIVE;
    static constexpr int PACK_COLS = NPACK > 0 ? (TN + NPACK - 1) / NPACK : 1;  // columns per packing warp
    static_assert(COL_A0 + 128u * NA <= TMEM_COLS && 2 * TN <= (int)COL_A0, "tensor-memory columns");
    __host__ __device__ static constexpr uint32_t col_s1(int p) { return (uint32_t)(TN * p); }
    __host__ __device__ static constexpr uint32_t col_a(int i) { return COL_A0 + 128u * (uint32_t)i; }
    static constexpr uint32_t IDESC = idesc_f16(TM, TN, 0);
    static_assert(TN == 32 || TN == 64 || TN == 128, "tile widths");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(SLOT_B % 1024 == 0 && OP_B % 1024 == 0, "SW128 tiles need 1024-byte alignment");
    static_assert(OFF_RAW % 128 == 0 && RAW_STAGE % 128 == 0, "tiled TMA destinations are 128-byte aligned");
    static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
    static_assert(WS_UNIT % 16 == 0 && HALF0_BYTES % 16 == 0 && HALF1_BYTES % 16 == 0 && SLOT_MIN % 16 == 0,
                  "bulk copies move 16-byte units");
};

// Tile width for a batch: the narrowest tile that covers it, 128 beyond 64.
inline int pick_tn(int64_t batch) { return batch <= 32 ? 32 : (batch <= 64 ? 64 : 128); }

// One MMA with the A operand in tensor memory (lane = row, K along the
// columns, two fp16 per 32-bit column with the lower K in the low half).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
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

// Two runs of 8 consecutive fp32 columns of this warp's 32 tensor-memory
// lanes, both loads in flight before one wait.
__device__ __forceinline__ void tmem_ld8x2(uint32_t ta, uint32_t tb, float (&va)[8], float (&vb)[8]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(ta), "r"(tb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[8 + i]);
    }
}

// Byte offset of K group g (0 or 1) of tile row r in the no-swizzle min-term
// tile (core matrices 128 bytes apart along K, 8-row groups 256 bytes apart).
__device__ __forceinline__ uint32_t plain_off(int r, int g) {
    return (uint32_t)((r >> 3) * 256 + g * 128 + (r & 7) * 16);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// ----------------------------------------------------------------- packing

// One CTA per (super-block, column tile); warp w packs columns w, w+8, ...
// Lane l owns codes 8l..8l+7 (K group l of the super-block) and writes them
// as fp16 in the group order (a0,a4, a1,a5, a2,a6, a3,a7) -- the order in
// which the A builders emit the weight nibbles -- into the 128-byte-swizzled
// image of operand stage l / 8.  Lanes 0..7 also write the sub-block sum t_j
// split exactly as t_lo = t mod 64 (K position j) and t_hi = floor(t / 64)
// (K position 8 + j) of the min-term tile, and lane 0 the column scale dx
// and the column's code sum (the sum of the eight t_j).  Columns past the
// batch are zero.
// What lane l of a warp reads of one column's Q8_K block: codes 8l..8l+7
// and, lanes 0..7, the sub-block sum t_l (zeros for a column past the batch).
struct PackIn {
    uint32_t w0, w1;
    int t;
};

__device__ __forceinline__ PackIn pack_load(const uint8_t *__restrict__ src, bool valid) {
    const int lane = threadIdx.x & 31;
    PackIn in{0u, 0u, 0};
    if (valid) {
        in.w0 = __ldg(reinterpret_cast<const uint32_t *>(src + 4 + 8 * lane));
        in.w1 = __ldg(reinterpret_cast<const uint32_t *>(src + 8 + 8 * lane));
        if (lane < 8) in.t = __ldg(reinterpret_cast<const int16_t *>(src + 260) + lane);
    }
    return in;
}

// Column c of one unit (a warp, lane l): the operand stages go to st01
// (stages 0, 1) and st23 (stages 2, 3, then the min-term tile); with SUM,
// returns the column's code sum in every lane.
template <class C, bool SUM = true>
__device__ __forceinline__ int pack_store(const PackIn &in, int c, uint8_t *st01, uint8_t *st23) {
    const int lane = threadIdx.x & 31;
    // the codes as exact fp16 pairs (a0, a4), (a1, a5), (a2, a6), (a3, a7)
    const uint4 chunk = ms::i8x8_to_f16(in.w0, in.w1);
    const int stage = lane >> 3;
    uint8_t *st = stage < 2 ? st01 + stage * C::OP_B : st23 + (stage - 2) * C::OP_B;
    *reinterpret_cast<uint4 *>(st + sw128_off(c, lane & 7)) = chunk;
    const int t = in.t;
    if (lane < 8) {
        const int thi = t >> 6;          // floor(t / 64), in [-64, 63]
        const int tlo = t - 64 * thi;    // in [0, 63]
        uint8_t *mb = st23 + 2 * C::OP_B;
        *reinterpret_cast<__half *>(mb + plain_off(c, 0) + 2 * lane) = __int2half_rn(tlo);
        *reinterpret_cast<__half *>(mb + plain_off(c, 1) + 2 * lane) = __int2half_rn(thi);
    }
    if constexpr (!SUM) return 0;
    // code sum of the column's super-block: lanes 0..7 hold t_0..t_7, the
    // other lanes zero
    int asum = t;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) asum += __shfl_xor_sync(0xffffffffu, asum, o);
    return __shfl_sync(0xffffffffu, asum, 0);
}

template <class C>
__device__ __forceinline__ int pack_column(const uint8_t *__restrict__ src, bool valid, int c, uint8_t *st01,
                                           uint8_t *st23) {
    return pack_store<C>(pack_load(src, valid), c, st01, st23);
}

template <int TN>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ xq,
                                                   uint8_t *__restrict__ ws, int nsb, int batch) {
    using C = Cfg<TN>;
    const int sb = blockIdx.x, ct = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *unit = ws + ((size_t)ct * nsb + sb) * C::WS_UNIT;
    pdl_launch_dependents();
    pdl_wait();
    for (int c = warp; c < TN; c += 8) {
        const int b = ct * TN + c;
        const bool valid = b < batch;
        const uint8_t *src = xq + ((size_t)(valid ? b : 0) * nsb + sb) * Q8_K_BYTES;
        const int asum = pack_column<C>(src, valid, c, unit, unit + 2 * C::OP_B);
        if (lane == 0) {
            float *cs = reinterpret_cast<float *>(unit + C::WS_B + C::WS_MIN);
            cs[c] = valid ? __ldg(reinterpret_cast<const float *>(src)) : 0.0f;
            cs[TN + c] = (float)asum;  // exact: |asum| <= 256 * 127
        }
    }
}

// ------------------------------------------------------------- main kernel

// Barriers.  b_tx and raw_full complete when a copy has landed (their only
// arrival is the producer's expect-tx).  Per super-block sb, in a ring of NF:
//   sb_full[sb % NF]: its A operand (one arrival per builder warp) and its
//                     min-term A rows (one per hh = 0 builder warp) are in
//                     place, and the S1 buffer of its parity is free (one
//                     arrival per active epilogue warp after it read S1 of
//                     sb - 2; made at initialization for sb = 0, 1);
//   sb_done[sb % NF]: every MMA of sb has completed (one commit) -- its S1 and
//                     S2 may be read, and its two B slots and min-term rows
//                     reused.
// A waiter on sb_done for super-block x uses parity (x / NF) & 1; the ring
// cannot run a lap ahead of it, since super-block x + NF needs, through the
// waiter itself, a resource that x releases.
struct Bars {
    uint64_t *sb_full, *sb_done, *a_empty, *b_tx, *raw_full, *raw_empty;
    uint64_t *meta_full, *meta_empty, *fin;
};

template <class C>
__device__ __forceinline__ Bars bars_at(uint8_t *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    Bars r;
    r.sb_full = b;
    r.sb_done = r.sb_full + NF;
    r.a_empty = r.sb_done + NF;
    r.b_tx = r.a_empty + C::NA;
    r.raw_full = r.b_tx + C::NBS;
    r.raw_empty = r.raw_full + C::NRAW;
    r.meta_full = r.raw_empty + C::NRAW;
    r.meta_empty = r.meta_full + NSM;
    r.fin = r.meta_empty + NSM;
    return r;
}

// B ring slot of half h of super-block step sb; it is reused every NBSB-th
// step, so the parity of its current use is that of sb / NBSB.
template <class C>
__device__ __forceinline__ int b_slot(int sb, int h) { return 2 * (sb % C::NBSB) + h; }
template <class C>
__device__ __forceinline__ uint32_t b_phase(int sb) { return (uint32_t)(sb / C::NBSB) & 1u; }

// Producer of half h of the activation units (warps 0 and 3): one bulk copy
// per super-block into the B ring.  On abort it waits (bounded) for every
// copy it started before the CTA may exit.
template <class C>
__device__ void role_producer_b(uint8_t *smem, const Bars &B, const uint8_t *__restrict__ ws, int nsb,
                                int ct, int rot, int h, volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    const uint32_t bytes = h ? (uint32_t)C::HALF1_BYTES : (uint32_t)C::HALF0_BYTES;
    int last[C::NBSB];
    for (int i = 0; i < C::NBSB; ++i) last[i] = -1;
    bool ok = true;
    for (int sb = 0; ok && sb < nsb; ++sb) {
        const int s = b_slot<C>(sb, h);
        const uint32_t ph = b_phase<C>(sb);
        const int prev = sb - C::NBSB;  // the super-block that last used this slot
        if (prev >= 0 && !(ok = wait_warp(B.sb_done + prev % NF, (uint32_t)(prev / NF) & 1u, abort))) break;
        if (lane == 0) {
            const uint8_t *src =
                ws + ((size_t)ct * nsb + kslot(sb, rot, nsb)) * C::WS_UNIT + (h ? C::HALF0_BYTES : 0);
            mbar_arrive_expect_tx(B.b_tx + s, bytes);
            bulk_g2s(smem + C::OFF_B + s * C::SLOT_B, src, bytes, B.b_tx + s);
        }
        last[sb % C::NBSB] = (int)ph;
    }
    if (!ok)
        for (int i = 0; i < C::NBSB; ++i)
            if (last[i] >= 0) mbar_wait_bounded(B.b_tx + 2 * i + h, (uint32_t)last[i]);
}

// Producer of the raw weight rows (warp 2): one 2-D tiled TMA load per
// super-block (box 144 bytes x 128 rows; rows past the matrix read as
// zeros), NRAW - 1 super-blocks ahead of the builders.
template <class C>
__device__ void role_producer_w(uint8_t *smem, const Bars &B, const CUtensorMap *tmap_w, int row0, int nsb,
                                int rot, volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    int raw_last[C::NRAW];
    for (int i = 0; i < C::NRAW; ++i) raw_last[i] = -1;
    RingPos rr(C::NRAW);
    bool ok = true;
    for (int sb = 0; ok && sb < nsb; ++sb) {
        if (!(ok = wait_warp(B.raw_empty + rr.idx, rr.phase ^ 1u, abort))) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(B.raw_full + rr.idx, RAW_STAGE);
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + C::OFF_RAW + rr.idx * RAW_STAGE)),
                "l"(reinterpret_cast<uint64_t>(tmap_w)), "r"(kslot(sb, rot, nsb) * Q4_K_BYTES), "r"(row0),
                "r"(smem_u32(B.raw_full + rr.idx))
                : "memory");
        }
        __syncwarp();
        raw_last[rr.idx] = (int)rr.phase;
        rr.next();
    }
    if (!ok)
        for (int i = 0; i < C::NRAW; ++i)
            if (raw_last[i] >= 0) mbar_wait_bounded(B.raw_full + i, (uint32_t)raw_last[i]);
}

// fp16x2 value of the two halves of an integer-coded word (bit pattern).
__device__ __forceinline__ __half2 h2_bits(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ uint32_t bits_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// One packed nibble word (elements e0..e7 in nibbles 0..7) to the fp16 chunk
// (v e0, v e4, v e1, v e5, v e2, v e6, v e3, v e7), v e = sc e - 512.  A nibble
// placed in mantissa bits 0-3 (4-7) of 0x6400 gives the exact fp16 value
// 1024 + e (1024 + 16 e); one fma with (sc, -512 (2 sc + 1)) -- or
// (sc / 16, -64 (sc + 8)) -- yields sc e - 512 exactly: both addends have at
// most 7 significant bits, and the fused result, an integer in [-512, 433],
// is representable.
__device__ __forceinline__ uint4 nibbles_to_f16(uint32_t w, __half2 s1, __half2 c1, __half2 s16,
                                                __half2 c16) {
    const uint32_t w8 = w >> 8;
    const __half2 p0 = h2_bits((w & 0x000F000Fu) | 0x64006400u);
    const __half2 p1 = h2_bits((w & 0x00F000F0u) | 0x64006400u);
    const __half2 p2 = h2_bits((w8 & 0x000F000Fu) | 0x64006400u);
    const __half2 p3 = h2_bits((w8 & 0x00F000F0u) | 0x64006400u);
    return make_uint4(bits_h2(__hfma2(p0, s1, c1)), bits_h2(__hfma2(p1, s16, c16)),
                      bits_h2(__hfma2(p2, s1, c1)), bits_h2(__hfma2(p3, s16, c16)));
}

// A builders (warps 4-11): warp w builds tile rows 32 (w % 4) .. + 31 (its
// tensor-memory lanes; row t = 32 (w % 4) + lane) for half hh = (w - 4) / 4
// of every super-block, i.e. sub-blocks 4hh .. 4hh + 3 = K 128hh .. + 127 =
// A columns 64hh .. + 63 of the buffer of the super-block's parity.  Each
// sub-block is 16 columns, written by one tcgen05.st from registers; the
// buffer is free again once the epilogue has read the S2 written over it.
// Then the hh = 0 threads write row t's min-term A row, the hh = 1 threads
// row t's scales d, dmin and (t < TN) column t's scale dx and code sum (read
// from the workspace, requested before the raw weights are waited for).
template <class C, bool WS>
__device__ void role_builder(uint8_t *smem, const Bars &B, uint32_t tmem, const uint8_t *__restrict__ ws,
                             const uint8_t *__restrict__ xq, int batch, int ct, int rot, int nvalid, int nsb,
                             volatile uint32_t *abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = 32 * (warp & 3) + lane, hh = (warp - BLD_WARP0) >> 2;
    const bool valid = t < nvalid;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    RingPos rr(C::NRAW), mr(NSM);
    for (int sb = 0; sb < nsb; ++sb) {
        const int ai = sb % C::NA;                              // A buffer
        const uint32_t aph = (uint32_t)(sb / C::NA) & 1u;       // parity of its use
        float dx = 0.0f, as = 0.0f;
        if (hh == 1 && t < C::TN) {
            if constexpr (WS) {
                const uint8_t *unit = ws + ((size_t)ct * nsb + kslot(sb, rot, nsb)) * C::WS_UNIT;
                const float *cs = reinterpret_cast<const float *>(unit + C::WS_B + C::WS_MIN);
                dx = __ldg(cs + t);
                as = __ldg(cs + C::TN + t);
            } else if (ct * C::TN + t < batch) {
                // no workspace: the column's scale and code sum straight from
                // its Q8_K block (the eight sub-block sums added, exact)
                const uint8_t *src = xq + ((size_t)(ct * C::TN + t) * nsb + kslot(sb, rot, nsb)) * Q8_K_BYTES;
                dx = __ldg(reinterpret_cast<const float *>(src));
                // Q8_K blocks are 276 bytes: only 4-byte alignment holds
                const uint32_t *bs = reinterpret_cast<const uint32_t *>(src + 260);
                int a = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t w = __ldg(bs + k);
                    a += (int)(int16_t)(w & 0xffffu) + (int)(int16_t)(w >> 16);
                }
                as = (float)a;
            }
        }
        if (!wait_warp(B.raw_full + rr.idx, rr.phase, abort)) return;
        const uint8_t *raw = smem + C::OFF_RAW + rr.idx * RAW_STAGE + t * Q4_K_BYTES;
        uint4 h = make_uint4(0, 0, 0, 0), q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) q[j] = make_uint4(0, 0, 0, 0);
        if (valid) {
            h = *reinterpret_cast<const uint4 *>(raw);
#pragma unroll
            for (int j = 0; j < 4; ++j) q[j] = *reinterpret_cast<const uint4 *>(raw + 16 + 16 * (4 * hh + j));
        }
        mbar_arrive(B.raw_empty + rr.idx);
        rr.next();

        // this half of the A operand: sc_j * q - 512 for sub-blocks 4hh .. 4hh + 3
        if (!wait_warp(B.a_empty + ai, aph ^ 1u, abort)) return;
        tc_fence_after();
        const uint64_t lo64 = (uint64_t)h.y | ((uint64_t)h.z << 32);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float sc = (float)(int)((lo64 >> (6 * (4 * hh + j))) & 63);
            const __half2 s1 = __float2half2_rn(sc), c1 = __float2half2_rn(-512.0f * (2.0f * sc + 1.0f));
            const __half2 s16 = __float2half2_rn(sc * 0.0625f), c16 = __float2half2_rn(-64.0f * (sc + 8.0f));
            uint4 v[4];
            v[0] = nibbles_to_f16(q[j].x, s1, c1, s16, c16);
            v[1] = nibbles_to_f16(q[j].y, s1, c1, s16, c16);
            v[2] = nibbles_to_f16(q[j].z, s1, c1, s16, c16);
            v[3] = nibbles_to_f16(q[j].w, s1, c1, s16, c16);
            tmem_st16(lane_base + C::col_a(ai) + 64u * hh + 16u * j, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.sb_full + sb % NF);

        // then (off the MMA's critical path) the hh = 1 threads write the
        // epilogue's scales (row t's d and dmin, column t's dx), the hh = 0
        // threads row t's min-term A row [m_0..m_7 | 64 m_0..64 m_7] (fp16, exact)
        if (hh == 1) {
            if (!wait_warp(B.meta_empty + mr.idx, mr.phase ^ 1u, abort)) return;
            uint8_t *meta = smem + C::OFF_META + mr.idx * C::META_STAGE;
            reinterpret_cast<float *>(meta + C::META_D)[t] = half_bits_to_float(h.x);
            reinterpret_cast<float *>(meta + C::META_DMIN)[t] = half_bits_to_float(h.x >> 16);
            if (t < C::TN) {
                reinterpret_cast<float2 *>(meta + C::META_COL)[t] = make_float2(dx, 512.0f * as);
            }
            mbar_arrive(B.meta_full + mr.idx);
        } else {
            const uint64_t hi64 = (uint64_t)h.z | ((uint64_t)h.w << 32);  // header bits 32..95
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const float m0 = (float)(int)((hi64 >> (6 * j + 16)) & 63);
                const float m1 = (float)(int)((hi64 >> (6 * (j + 1) + 16)) & 63);
                lo[j >> 1] = pack_h2(m0, m1);
                hi[j >> 1] = pack_h2(64.0f * m0, 64.0f * m1);
            }
            // the min-term rows of sb - NF (same slot) have been consumed
            if (sb >= NF && !wait_warp(B.sb_done + sb % NF, (uint32_t)(sb / NF - 1) & 1u, abort)) return;
            uint8_t *ma = smem + C::OFF_MINA + mr.idx * MIN_A;
            *reinterpret_cast<uint4 *>(ma + plain_off(t, 0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4 *>(ma + plain_off(t, 1)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.sb_full + sb % NF);
        }
        mr.next();
    }
}

// Eight K=16 steps into accumulator d, the A operand of step i at tensor
// memory column a[i] and its B operand at descriptor b[i], in one asm block
// whose operands are all computed beforehand.  Issued back to back this way
// one thread feeds the tensor core about one M=128 step per 60 clocks; with
// each step's addresses and predicate formed just before it, about one per
// 100-150.  Only the first step may start a fresh accumulation
// (accumulate == 0).
__device__ __forceinline__ void mma8_ta(uint32_t d, const uint32_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t"
        "setp.ne.b32 p, %18, 0;\n\t"
        "setp.eq.b32 t, %18, %18;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, t;\n\t}" ::"r"(d),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]),
        "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc),
        "r"(accumulate)
        : "memory");
}


// MMA issuer (warp 1, one thread).  Per super-block: once its A operand and
// min-term rows are built and the S1 buffer of its parity is drained (both
// counted by sb_full) and the first B half has landed, eight K=16 steps of
// the S1 product (A from
// the super-block's tensor-memory buffer, B from the ring), then after the
// second half has landed eight more, then one K=16 step of the min-term
// product S2 written over the consumed A buffer; then a single commit
// (sb_done) that the epilogue, the B producers and the min-term builders all
// wait on.  A wait or a commit costs the issuing thread about as much as one
// to two MMAs, so the super-block has as few of them as its dependencies
// allow.  Always ends with a commit to `fin` so the teardown can wait for
// every MMA to finish.
template <class C>
__device__ void role_mma(uint8_t *smem, const Bars &B, uint32_t tmem, int nsb, volatile uint32_t *abort) {
    constexpr uint64_t OPB16 = C::OP_B >> 4;  // one B stage in descriptor address units
    bool ok = true;
    for (int sb = 0; ok && sb < nsb; ++sb) {
        const int p = sb & 1;                                   // S1 buffer
        const int ai = sb % C::NA;                              // A buffer
        const int f = sb % NF;                                  // ready / done ring, min-term rows
        if (!(ok = wait_or_abort(B.sb_full + f, (uint32_t)(sb / NF) & 1u, abort))) break;
        for (int h = 0; h < 2; ++h) {
            const int sl = b_slot<C>(sb, h);
            if (!(ok = wait_or_abort(B.b_tx + sl, b_phase<C>(sb), abort))) break;
            if (h == 0) tc_fence_after();
            const uint64_t b0 = desc_sw128(smem_u32(smem + C::OFF_B + sl * C::SLOT_B));
            const uint32_t a0 = tmem + C::col_a(ai) + 64u * h;
            uint32_t av[8];
            uint64_t bv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // stage i / 4 of the half, K step i % 4
                av[i] = a0 + 32u * (i >> 2) + 8u * (i & 3);
                bv[i] = b0 + OPB16 * (uint64_t)(i >> 2) + 2u * (uint64_t)(i & 3);
            }
            mma8_ta(tmem + C::col_s1(p), av, bv, C::IDESC, (uint32_t)h);
        }
        if (!ok) break;
        const uint32_t a2 = smem_u32(smem + C::OFF_MINA + f * MIN_A);
        const uint32_t b2 = smem_u32(smem + C::OFF_B + b_slot<C>(sb, 1) * C::SLOT_B + C::SLOT_MIN);
        mma_f16(tmem + C::col_a(ai), desc_plain(a2, 128, 256), desc_plain(b2, 128, 256), C::IDESC, 0u);
        mma_commit(B.sb_done + f);  // S1 and S2 ready; both B slots and the min-term rows free
    }
    mma_commit(B.fin);
}

// Without a workspace (tiles of up to 64 columns): the epilogue warps whose
// columns lie past TN pack the activation operand into the B ring themselves,
// the work pack_kernel does into the workspace.  Per super-block they wait
// until the MMAs of the super-block NBSB steps back have released the slot
// pair, convert their columns (warp w of NP takes columns w, w + NP, ...),
// make the stores visible to the tensor core and arrive on both halves'
// barriers (NP arrivals complete each).
template <class C>
__device__ void role_pack(uint8_t *smem, const Bars &B, const uint8_t *__restrict__ xq, int batch, int ct,
                          int rot, int nsb, int pw, volatile uint32_t *abort) {
    constexpr int KMAX = C::PACK_COLS;
    const int lane = threadIdx.x & 31;
    // the reads of super-block sb + 1 are in flight while sb waits for its
    // slots and is converted
    PackIn cur[KMAX], nxt[KMAX];
    auto load_sb = [&](int sb, PackIn (&in)[C::PACK_COLS]) {
        const int ks = kslot(sb, rot, nsb);
#pragma unroll
        for (int k = 0; k < C::PACK_COLS; ++k) {
            const int c = pw + k * C::NPACK, b = ct * C::TN + c;
            const bool valid = c < C::TN && b < batch;
            in[k] = pack_load(xq + ((size_t)(valid ? b : 0) * nsb + ks) * Q8_K_BYTES, valid);
        }
    };
    load_sb(0, cur);
    for (int sb = 0; sb < nsb; ++sb) {
        if (sb + 1 < nsb) load_sb(sb + 1, nxt);
        const int prev = sb - C::NBSB;  // the super-block that last used these slots
        if (prev >= 0 && !wait_warp(B.sb_done + prev % NF, (uint32_t)(prev / NF) & 1u, abort)) return;
        uint8_t *h0 = smem + C::OFF_B + b_slot<C>(sb, 0) * C::SLOT_B;
        uint8_t *h1 = smem + C::OFF_B + b_slot<C>(sb, 1) * C::SLOT_B;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int c = pw + k * C::NPACK;
            if (c < C::TN) pack_store<C, false>(cur[k], c, h0, h1);  // the builders add the sums
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B.b_tx + b_slot<C>(sb, 0));
            mbar_arrive(B.b_tx + b_slot<C>(sb, 1));
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) cur[k] = nxt[k];
    }
}

// Epilogue (warps 12-27): warp w reads tensor-memory lanes 32 (w % 4) .. + 31
// (its 32 rows) and columns 32 h .. + 31, h = (w - 12) / 4, of S1 and of the
// S2 written over the A buffer.  It frees both as soon as they are in
// registers and promotes them while the tensor core runs the next
// super-block.  Warps whose columns lie past TN have nothing to do (the
// barriers count EPI_ACTIVE warps).
template <class C, bool SUMS>
__device__ void role_epilogue(uint8_t *smem, const Bars &B, uint32_t tmem, int row0, int rows, int ct,
                              int nsb, int rot, int batch, float *__restrict__ y,
                              int32_t *__restrict__ sums, volatile uint32_t *abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lq = warp & 3, h = (warp - EPI_WARP0) >> 2;
    if (32 * h >= C::TN) return;
    constexpr int TN = C::TN;
    const int r = lq * 32 + lane;
    const int row = row0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(32 * h);
    float yacc[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) yacc[c] = 0.0f;
    bool ok = true;
    for (int sb = 0; sb < nsb; ++sb) {
        const int p = sb & 1;
        const uint32_t ph = (uint32_t)(sb >> 1) & 1u;
        const int ai = sb % C::NA;
        const int mi = sb % NSM;
        const uint32_t mph = (uint32_t)(sb / NSM) & 1u;
        if (!(ok = wait_warp(B.meta_full + mi, mph, abort))) break;
        if (!(ok = wait_warp(B.sb_done + sb % NF, (uint32_t)(sb / NF) & 1u, abort))) break;
        tc_fence_after();
        const uint8_t *meta = smem + C::OFF_META + mi * C::META_STAGE;
        const float d = reinterpret_cast<const float *>(meta + C::META_D)[r];
        const float dmin = reinterpret_cast<const float *>(meta + C::META_DMIN)[r];
        const float2 *col = reinterpret_cast<const float2 *>(meta + C::META_COL) + 32 * h;
        // eight columns at a time: S1 and S2 of the group, plus the column
        // pairs, stay within the register budget next to the 32 accumulators
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 8) {
            float s1[8], s2[8];
            tmem_ld8x2(lane_addr + C::col_s1(p) + c0, lane_addr + C::col_a(ai) + c0, s1, s2);
            if (c0 == 24) {
                // all of S1 and S2 is in registers: S1 and the A buffer may be reused
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // S1 buffer p is next accumulated by super-block sb + 2: its
                    // ready barrier counts this release
                    if (sb + 2 < nsb) mbar_arrive(B.sb_full + (sb + 2) % NF);
                    mbar_arrive(B.a_empty + ai);
                }
            }
            if (SUMS) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int b = ct * TN + 32 * h + c0 + i;
                    if (row < rows && b < batch) {
                        int32_t *o = sums + (((size_t)b * rows + row) * nsb + kslot(sb, rot, nsb)) * 2;
                        o[0] = (int32_t)s1[i] + (int32_t)col[c0 + i].y;
                        o[1] = (int32_t)s2[i];
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 cv = col[c0 + i];   // (dx, 512 * code sum)
                    const float S1 = s1[i] + cv.y;   // the exact S1, rounded once
                    yacc[c0 + i] = fmaf(cv.x, d * S1 - dmin * s2[i], yacc[c0 + i]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(B.meta_empty + mi);
    }
    if (!ok || SUMS) return;
    if (row < rows) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int b = ct * TN + 32 * h + c;
            if (b < batch) y[(size_t)b * rows + row] = yacc[c];
        }
    }
}

// WS: the activation operand comes packed in the workspace (bulk copies by
// warps 0 and 3); otherwise the idle epilogue warps pack it from xq in the
// CTA (TN <= 64).
template <int TN, bool SUMS, bool WS>
__global__ void __launch_bounds__(NTHREADS, 1) mma_q4k_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                              const uint8_t *__restrict__ ws,
                                                              const uint8_t *__restrict__ xq,
                                                              float *__restrict__ y,
                                                              int32_t *__restrict__ sums, int rows,
                                                              int nsb, int batch,
                                                              uint32_t *__restrict__ status) {
    using C = Cfg<TN>;
    static_assert(WS || C::NPACK > 0, "packing in the CTA needs idle epilogue warps");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Bars B = bars_at<C>(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // column tiles vary fastest, so the CTAs that read the same weight rows
    // run together and share them through L2
    const int row0 = blockIdx.y * TM, ct = blockIdx.x;
    const int rot = (int)(blockIdx.y % (unsigned)nsb);
    const int nvalid = min(TM, rows - row0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NF; ++i) {
            // one arrival per builder warp (A), per hh = 0 builder warp (min-term
            // rows) and per active epilogue warp (the S1 buffer of the
            // super-block's parity released by super-block sb - 2)
            mbar_init(B.sb_full + i, BLD_THREADS / 32 + 4 + C::EPI_ACTIVE);
            mbar_init(B.sb_done + i, 1);
        }
        // super-blocks 0 and 1 find their S1 buffers free
        for (int i = 0; i < 2; ++i)
            for (int k = 0; k < C::EPI_ACTIVE; ++k) mbar_arrive(B.sb_full + i);
        for (int i = 0; i < C::NA; ++i) mbar_init(B.a_empty + i, C::EPI_ACTIVE);  // S2 over it read
        // a slot's operand half: one expect-tx arrival for its bulk copy, or
        // one arrival per packing warp
        for (int i = 0; i < C::NBS; ++i) mbar_init(B.b_tx + i, WS ? 1 : C::NPACK);
        for (int i = 0; i < C::NRAW; ++i) {
            mbar_init(B.raw_full + i, 1);
            mbar_init(B.raw_empty + i, BLD_THREADS);
        }
        for (int i = 0; i < NSM; ++i) {
            mbar_init(B.meta_full + i, BLD_THREADS / 2);  // every hh = 1 builder thread
            mbar_init(B.meta_empty + i, C::EPI_ACTIVE);
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
    pdl_wait();  // the packed activations come from the preceding kernel

    if (warp == 0 || warp == 3) {
        if (WS) role_producer_b<C>(smem, B, ws, nsb, ct, rot, warp == 3 ? 1 : 0, abort);
    } else if (warp == 2) {
        role_producer_w<C>(smem, B, &tmap_w, row0, nsb, rot, abort);
    } else if (warp == 1) {
        if (lane == 0) role_mma<C>(smem, B, tmem, nsb, abort);
        __syncwarp();
    } else if (warp >= BLD_WARP0 && warp < EPI_WARP0) {
        role_builder<C, WS>(smem, B, tmem, ws, xq, batch, ct, rot, nvalid, nsb, abort);
    } else if (warp >= EPI_WARP0) {
        const int ew = warp - EPI_WARP0;  // epilogue warps with columns come first
        if constexpr (!WS) {
            if (ew >= C::EPI_ACTIVE)
                role_pack<C>(smem, B, xq, batch, ct, rot, nsb, ew - C::EPI_ACTIVE, abort);
            else
                role_epilogue<C, SUMS>(smem, B, tmem, row0, rows, ct, nsb, rot, batch, y, sums, abort);
        } else {
            role_epilogue<C, SUMS>(smem, B, tmem, row0, rows, ct, nsb, rot, batch, y, sums, abort);
        }
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

}  // namespace

bool mma_supported(int64_t rows, int64_t cols, int64_t batch) {
    return rows >= 1 && batch >= 1 && cols >= QK_K && cols % QK_K == 0;
}

size_t mma_workspace_bytes(int64_t rows, int64_t cols, int64_t batch) {
    (void)rows;
    if (cols % QK_K != 0 || batch < 1) return 0;
    const int tn = pick_tn(batch);
    const size_t unit = tn == 32 ? Cfg<32>::WS_UNIT : (tn == 64 ? Cfg<64>::WS_UNIT : Cfg<128>::WS_UNIT);
    return (size_t)((batch + tn - 1) / tn) * (size_t)(cols / QK_K) * unit;
}

// Static scratch for callers that cannot allocate device memory (see
// gq_matmul_noalloc in gq.h).  It is module-scope device memory: every GPU
// that loads this library holds these bytes until the process exits.  Host
// code must never hand the symbol itself to a kernel -- on the host it only
// names the array; the device address comes from cudaGetSymbolAddress.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)16 << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
struct ScratchSlot {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *ptr = nullptr;
};
ScratchSlot g_scratch_slot[NOALLOC_MAX_DEVICES];

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// dependency on the driver library); shared with gq_mma_q0.cu.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int TN, bool WS>
cudaError_t launch_tiles(const CUtensorMap &tmap, const void *xq, float *y, int32_t *sums, int64_t rows,
                         int nsb, int64_t batch, uint8_t *ws, const LaunchCtx &ctx) {
    using C = Cfg<TN>;
    const int ctiles = (int)((batch + TN - 1) / TN);
    const int rtiles = (int)((rows + TM - 1) / TM);
    cudaError_t e = cudaSuccess;
    if (WS) {
        e = launch_pdl(pack_kernel<TN>, dim3(nsb, ctiles), dim3(256), 0, ctx.stream,
                       static_cast<const uint8_t *>(xq), ws, nsb, (int)batch);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((unsigned)ctiles, (unsigned)rtiles);
    auto k = sums ? mma_q4k_kernel<TN, true, WS> : mma_q4k_kernel<TN, false, WS>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, grid, dim3(NTHREADS), C::SMEM_ALLOC, ctx.stream, tmap, (const uint8_t *)ws,
                      static_cast<const uint8_t *>(xq), y, sums, (int)rows, nsb, (int)batch, ctx.status);
}

cudaError_t launch_mma_q4k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                           int64_t cols, int64_t batch, void *workspace, const LaunchCtx &ctx) {
    const int nsb = (int)(cols / QK_K);
    const int rtiles = (int)((rows + TM - 1) / TM);
    if (rtiles > 65535) return cudaErrorInvalidConfiguration;
    // W as a 2-D byte tensor: rows of nsb * 144 bytes; box = one super-block
    // (144 bytes) of 128 rows
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)nsb * Q4_K_BYTES, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)nsb * Q4_K_BYTES};
    const cuuint32_t box[2] = {(cuuint32_t)Q4_K_BYTES, (cuuint32_t)TM};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (!ws) {
        // no workspace: tiles of at most 64 columns, packed in the CTA
        if (batch <= 32) return launch_tiles<32, false>(tmap, xq, y, sums, rows, nsb, batch, nullptr, ctx);
        return launch_tiles<64, false>(tmap, xq, y, sums, rows, nsb, batch, nullptr, ctx);
    }
    switch (pick_tn(batch)) {
    case 32: return launch_tiles<32, true>(tmap, xq, y, sums, rows, nsb, batch, ws, ctx);
    case 64: return launch_tiles<64, true>(tmap, xq, y, sums, rows, nsb, batch, ws, ctx);
    default: return launch_tiles<128, true>(tmap, xq, y, sums, rows, nsb, batch, ws, ctx);
    }
}

size_t mma_noalloc_scratch_bytes() { return NOALLOC_SCRATCH_BYTES; }

// Device address of the static scratch on the current device, resolved once
// per device (with that device current) on the first call there.
cudaError_t mma_noalloc_scratch(int device, void **ptr) {
    if (device < 0 || device >= NOALLOC_MAX_DEVICES) return cudaErrorInvalidDevice;
    ScratchSlot &slot = g_scratch_slot[device];
    std::call_once(slot.once, [&slot]() {
        void *p = nullptr;
        slot.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        slot.ptr = p;
    });
    *ptr = slot.ptr;
    return slot.err;
}

}  // namespace gq
