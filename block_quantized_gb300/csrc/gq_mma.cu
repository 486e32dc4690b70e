// gq_mma.cu -- batched Q4_K x Q8_K product on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), for batches large enough that
// the product is a dense contraction ("llama.cpp 推理引擎" §7.3: prompt
// processing is compute-bound, token generation bandwidth-bound).
//
// sm_103a has no integer MMA kind, so the contraction runs on the fp16 kind
// with operands that are small integers, exactly representable in fp16:
//   A[r][k] = sc_j(r) * q_k(r)        (<= 63 * 15 = 945)
//   B[b][k] = a_k(b)                  (|a| <= 127, the Q8_K code)
// Every product is exact and the fp32 accumulation of one 256-element
// super-block is exact while partial sums stay below 2^24, so the tensor core
// returns the integer S1 = sum_j sc_j * s_j of "llama.cpp 推理引擎" §5.5's
// two-level scheme.  The min-term integer S2 = sum_j m_j * t_j (t_j the
// activation sub-block sums) is one more K=16 step per super-block into a
// second accumulator, with t_j split exactly as t_lo + 64 t_hi:
//   A2[r] = [m_0..m_7 | 64 m_0..64 m_7]   B2[b] = [t_lo_0..t_lo_7 | t_hi_0..t_hi_7]
// (all exact in fp16, |S2| < 2^21).  Per super-block the epilogue promotes
// both exact integers:
//   y[b][r] += dx(b) * (d(r) * S1 - dmin(r) * S2)      (fp32, in registers)
//
// CTA tile: 128 weight rows x 128 batch columns, one super-block (K = 256) per
// step, 28 warps:
//   warp 0     activation producer: 1-D bulk copies of the packed B tiles
//              into their own 6-slot ring (1.5 super-blocks ahead);
//   warp 1     MMA issuer (one thread) and tensor-memory owner;
//   warp 2     weight producer: one 2-D tiled TMA load per super-block of
//              the raw Q4_K rows (box 144 bytes x 128 rows; rows past the
//              matrix read as zeros), the min-term B tile and the scales;
//   warps 4-11 A builders: two threads per weight row, each turning half of
//              the raw super-block into two fp16 A stages (128-byte swizzled
//              K-major); the first half also writes the min-term row and the
//              row scales d, dmin;
//   warps 12-27 epilogue: four threads per row, 32 columns each.
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

namespace gq {
namespace {

constexpr int TM = 128;   // weight rows per tile (MMA M)
constexpr int TN = 128;   // batch columns per tile (MMA N)
constexpr int KS = 64;    // K per operand stage (one 128-byte swizzle atom)
constexpr int NOP = 4;    // A operand stages (= one super-block)
constexpr int NBR = 6;    // B operand stages (1.5 super-blocks of lookahead)
constexpr int NRAW = 2;   // raw weight stages
constexpr int KMIN = 16;  // min-term K per super-block (8 mins, two halves of t)

// Shared-memory layout (bytes from a 1024-aligned base).
constexpr int OP_A = TM * KS * 2;                 // 16 KB
constexpr int OP_B = TN * KS * 2;                 // 16 KB
constexpr int MIN_A = TM * KMIN * 2;              // 4 KB
constexpr int MIN_B = TN * KMIN * 2;              // 4 KB
constexpr int MIN_STAGE = MIN_A + MIN_B;          // 8 KB
constexpr int RAW_STAGE = TM * Q4_K_BYTES;        // 18 KB
// per super-block scales: d and dmin per row, dx per column (all fp32)
constexpr int META_D = 0, META_DMIN = TM * 4, META_DX = 2 * TM * 4;
constexpr int META_STAGE = 2 * TM * 4 + TN * 4;

constexpr int OFF_A = 0;                                  // NOP x 16 KB
constexpr int OFF_B = OFF_A + NOP * OP_A;                 // NBR x 16 KB
constexpr int OFF_MIN = OFF_B + NBR * OP_B;
constexpr int OFF_RAW = OFF_MIN + 2 * MIN_STAGE;          // 163840
constexpr int OFF_META = OFF_RAW + NRAW * RAW_STAGE;      // 200704
constexpr int OFF_BAR = OFF_META + 2 * META_STAGE;        // 202752
// A: full (builders), empty; B: full-tx (producer), empty; min: full
// (builders), full-tx, empty; raw: full, empty; meta: full (builders),
// full-tx, empty; acc: full, empty; final.
constexpr int NBARS = 2 * NOP + 2 * NBR + 3 * 2 + 2 * NRAW + 3 * 2 + 2 * 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM_USED = OFF_MISC + 16;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for the 1024-byte alignment
static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
static_assert(OFF_A % 1024 == 0 && OFF_B % 1024 == 0 && OP_A % 1024 == 0 && OP_B % 1024 == 0,
              "SW128 tiles need 1024-byte alignment");

// Workspace (packed activations) per (column tile, super-block).
constexpr size_t WS_B = (size_t)NOP * OP_B;   // 64 KB, the four B stage images
constexpr size_t WS_MIN = MIN_B;              // 4 KB
constexpr size_t WS_DX = TN * 4;              // 512 B
constexpr size_t WS_UNIT = WS_B + WS_MIN + WS_DX;

// Tensor-memory columns: S1 and S2 accumulators, each double-buffered by
// super-block parity.
constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t col_s1(int p) { return 128u * (uint32_t)p; }
__host__ __device__ constexpr uint32_t col_s2(int p) { return 256u + 128u * (uint32_t)p; }

constexpr int NTHREADS = 896;
constexpr int EPI_WARP0 = 12, EPI_WARPS = 16, BLD_WARP0 = 4, BLD_THREADS = 256;

// ------------------------------------------------------------ tcgen05 helpers

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row groups
// 1024 bytes apart; K advances inside the swizzle atom by moving the start
// address (32 bytes per 16 fp16).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Shared-memory matrix descriptor, K-major, no swizzle: 8x16-byte core
// matrices, `lbo` bytes apart along K and `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t desc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulate, A/B fp16 (fmt 0) or
// bf16 (fmt 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, uint32_t fmt) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait that also gives up as soon as another role of the CTA set
// the abort flag.  Returns false (and raises the flag) when it gives up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    return false;
}

// The same for a whole warp: every lane polls, and the warp gives up together
// if any lane did, so no lane leaves a warp-synchronous section alone.
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    const bool ok = wait_or_abort(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Ring position: stage index and the parity of its current use.
struct RingPos {
    int n, idx;
    uint32_t phase;
    __device__ explicit RingPos(int stages) : n(stages), idx(0), phase(0) {}
    __device__ void next() {
        if (++idx == n) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// Byte offset of the 16-byte chunk holding K group g (8 elements) of tile
// row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int g) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((g ^ (r & 7)) << 4));
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
// (K position 8 + j) of the min-term tile, and lane 0 the column scale dx.
// Columns past the batch are zero.
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ xq,
                                                   uint8_t *__restrict__ ws, int nsb, int batch) {
    const int sb = blockIdx.x, ct = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *unit = ws + ((size_t)ct * nsb + sb) * WS_UNIT;
    pdl_launch_dependents();
    pdl_wait();
    for (int c = warp; c < TN; c += 8) {
        const int b = ct * TN + c;
        const bool valid = b < batch;
        const uint8_t *src = xq + ((size_t)(valid ? b : 0) * nsb + sb) * Q8_K_BYTES;
        uint32_t w0 = 0, w1 = 0;
        if (valid) {
            w0 = __ldg(reinterpret_cast<const uint32_t *>(src + 4 + 8 * lane));
            w1 = __ldg(reinterpret_cast<const uint32_t *>(src + 8 + 8 * lane));
        }
        float a[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[i] = (float)(int8_t)(w0 >> (8 * i));
            a[4 + i] = (float)(int8_t)(w1 >> (8 * i));
        }
        const uint4 chunk = make_uint4(pack_h2(a[0], a[4]), pack_h2(a[1], a[5]), pack_h2(a[2], a[6]),
                                       pack_h2(a[3], a[7]));
        *reinterpret_cast<uint4 *>(unit + (lane >> 3) * OP_B + sw128_off(c, lane & 7)) = chunk;
        if (lane < 8) {
            int t = 0;
            if (valid) t = __ldg(reinterpret_cast<const int16_t *>(src + 260) + lane);
            const int thi = t >> 6;          // floor(t / 64), in [-64, 63]
            const int tlo = t - 64 * thi;    // in [0, 63]
            uint8_t *mb = unit + WS_B;
            *reinterpret_cast<__half *>(mb + plain_off(c, 0) + 2 * lane) = __int2half_rn(tlo);
            *reinterpret_cast<__half *>(mb + plain_off(c, 1) + 2 * lane) = __int2half_rn(thi);
        }
        if (lane == 0)
            reinterpret_cast<float *>(unit + WS_B + WS_MIN)[c] =
                valid ? __ldg(reinterpret_cast<const float *>(src)) : 0.0f;
    }
}

// ------------------------------------------------------------- main kernel

constexpr uint32_t IDESC_F16 = idesc_f16(TM, TN, 0);
constexpr uint32_t IDESC_BF16 = idesc_f16(TM, TN, 1);

// Barriers whose only arrival is a transfer's transaction count (the *_tx
// ones and raw_full) tell the producer that a copy has landed; the builders
// arrive on the plain *_full ones.
struct Bars {
    uint64_t *a_full, *a_empty, *b_tx, *b_empty, *min_full, *min_tx, *min_empty, *raw_full, *raw_empty;
    uint64_t *meta_full, *meta_tx, *meta_empty, *acc_full, *acc_empty, *fin;
};

__device__ __forceinline__ Bars bars_at(uint8_t *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    Bars r;
    r.a_full = b;
    r.a_empty = r.a_full + NOP;
    r.b_tx = r.a_empty + NOP;
    r.b_empty = r.b_tx + NBR;
    r.min_full = r.b_empty + NBR;
    r.min_tx = r.min_full + 2;
    r.min_empty = r.min_tx + 2;
    r.raw_full = r.min_empty + 2;
    r.raw_empty = r.raw_full + NRAW;
    r.meta_full = r.raw_empty + NRAW;
    r.meta_tx = r.meta_full + 2;
    r.meta_empty = r.meta_tx + 2;
    r.acc_full = r.meta_empty + 2;
    r.acc_empty = r.acc_full + 2;
    r.fin = r.acc_empty + 2;
    return r;
}

// Producer of the activation operand (warp 0): the four B stage images of
// every super-block, through a ring of NBR slots.  On abort it waits
// (bounded) for every copy it started before the CTA may exit.
__device__ void role_producer_b(uint8_t *smem, const Bars &B, const uint8_t *__restrict__ ws, int nsb,
                                int ct, volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    int last[NBR];
    for (int i = 0; i < NBR; ++i) last[i] = -1;
    RingPos br(NBR);
    bool ok = true;
    for (int sb = 0; ok && sb < nsb; ++sb) {
        const uint8_t *unit = ws + ((size_t)ct * nsb + sb) * WS_UNIT;
        for (int q = 0; q < NOP; ++q) {
            if (!(ok = wait_warp(B.b_empty + br.idx, br.phase ^ 1u, abort))) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(B.b_tx + br.idx, OP_B);
                bulk_g2s(smem + OFF_B + br.idx * OP_B, unit + (size_t)q * OP_B, OP_B, B.b_tx + br.idx);
            }
            last[br.idx] = (int)br.phase;
            br.next();
        }
    }
    if (!ok)
        for (int i = 0; i < NBR; ++i)
            if (last[i] >= 0) mbar_wait_bounded(B.b_tx + i, (uint32_t)last[i]);
}

// Producer of the weight side and the small per-super-block operands
// (warp 2): the raw Q4_K rows one super-block ahead (one 2-D tiled TMA load,
// box 144 bytes x 128 rows; rows past the matrix read as zeros), then the
// min-term B tile and the column scales of the current super-block.
__device__ void role_producer_w(uint8_t *smem, const Bars &B, const CUtensorMap *tmap_w,
                                const uint8_t *__restrict__ ws, int row0, int nsb, int ct,
                                volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    int raw_last[NRAW], min_last[2], meta_last[2];
    for (int i = 0; i < NRAW; ++i) raw_last[i] = -1;
    for (int i = 0; i < 2; ++i) min_last[i] = meta_last[i] = -1;
    RingPos rr(NRAW), mr(2);

    auto issue_raw = [&](int sb) -> bool {
        if (!wait_warp(B.raw_empty + rr.idx, rr.phase ^ 1u, abort)) return false;
        if (lane == 0) {
            mbar_arrive_expect_tx(B.raw_full + rr.idx, RAW_STAGE);
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + OFF_RAW + rr.idx * RAW_STAGE)),
                "l"(reinterpret_cast<uint64_t>(tmap_w)), "r"(sb * Q4_K_BYTES), "r"(row0),
                "r"(smem_u32(B.raw_full + rr.idx))
                : "memory");
        }
        __syncwarp();
        raw_last[rr.idx] = (int)rr.phase;
        rr.next();
        return true;
    };

    bool ok = issue_raw(0);
    for (int sb = 0; ok && sb < nsb; ++sb) {
        if (sb + 1 < nsb && !(ok = issue_raw(sb + 1))) break;
        const uint8_t *unit = ws + ((size_t)ct * nsb + sb) * WS_UNIT;
        if (!(ok = wait_warp(B.min_empty + mr.idx, mr.phase ^ 1u, abort))) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(B.min_tx + mr.idx, MIN_B);
            bulk_g2s(smem + OFF_MIN + mr.idx * MIN_STAGE + MIN_A, unit + WS_B, MIN_B, B.min_tx + mr.idx);
        }
        min_last[mr.idx] = (int)mr.phase;
        mr.next();
        const int mp = sb & 1;
        const uint32_t mph = (uint32_t)(sb >> 1) & 1u;
        if (!(ok = wait_warp(B.meta_empty + mp, mph ^ 1u, abort))) break;
        if (lane == 0) {
            mbar_arrive_expect_tx(B.meta_tx + mp, TN * 4);
            bulk_g2s(smem + OFF_META + mp * META_STAGE + META_DX, unit + WS_B + WS_MIN, TN * 4,
                     B.meta_tx + mp);
        }
        meta_last[mp] = (int)mph;
    }
    if (!ok) {
        for (int i = 0; i < NRAW; ++i)
            if (raw_last[i] >= 0) mbar_wait_bounded(B.raw_full + i, (uint32_t)raw_last[i]);
        for (int i = 0; i < 2; ++i) {
            if (min_last[i] >= 0) mbar_wait_bounded(B.min_tx + i, (uint32_t)min_last[i]);
            if (meta_last[i] >= 0) mbar_wait_bounded(B.meta_tx + i, (uint32_t)meta_last[i]);
        }
    }
}

// fp16x2 value of the two halves of an integer-coded word (bit pattern).
__device__ __forceinline__ __half2 h2_bits(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ uint32_t bits_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// One packed nibble word (elements e0..e7 in nibbles 0..7) to the fp16 chunk
// (sc e0, sc e4, sc e1, sc e5, sc e2, sc e6, sc e3, sc e7).  A nibble placed in
// mantissa bits 0-3 (4-7) of 0x6400 gives the exact fp16 value 1024 + e
// (1024 + 16 e); one fma with (sc, -1024 sc) -- or (sc / 16, -64 sc) --
// yields sc * e exactly (every operand and result is representable).
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

// A builders (warps 4-11): thread idx -> tile row t = idx % 128 and half
// hh = idx / 128, which builds operand stages 2hh and 2hh + 1 (sub-blocks
// 4hh .. 4hh + 3).  Stage q of every super-block uses ring slot q, so each
// half owns its two slots; the ring parity is the super-block's.
__device__ void role_builder(uint8_t *smem, const Bars &B, int idx, int nvalid, int nsb,
                             volatile uint32_t *abort) {
    const int lane = threadIdx.x & 31;
    const int t = idx & (TM - 1), hh = idx >> 7;
    const bool valid = t < nvalid;
    RingPos rr(NRAW), mr(2);
    for (int sb = 0; sb < nsb; ++sb) {
        const int mp = sb & 1;
        const uint32_t par = (uint32_t)sb & 1u;
        const uint32_t mph = (uint32_t)(sb >> 1) & 1u;
        if (!wait_warp(B.raw_full + rr.idx, rr.phase, abort)) return;
        const uint8_t *raw = smem + OFF_RAW + rr.idx * RAW_STAGE + t * Q4_K_BYTES;
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

        if (hh == 0) {
            // row scales and the min-term row [m_0..m_7 | 64 m_0..64 m_7] (fp16, exact)
            const uint64_t hi64 = (uint64_t)h.z | ((uint64_t)h.w << 32);
            int mn[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mn[j] = (int)((hi64 >> (6 * j + 16)) & 63);
            if (!wait_warp(B.meta_empty + mp, mph ^ 1u, abort)) return;
            uint8_t *meta = smem + OFF_META + mp * META_STAGE;
            reinterpret_cast<float *>(meta + META_D)[t] = half_bits_to_float(h.x);
            reinterpret_cast<float *>(meta + META_DMIN)[t] = half_bits_to_float(h.x >> 16);
            mbar_arrive(B.meta_full + mp);
            if (!wait_warp(B.min_empty + mr.idx, mr.phase ^ 1u, abort)) return;
            uint8_t *ma = smem + OFF_MIN + mr.idx * MIN_STAGE;
            if (valid) {
                uint32_t lo[4], hi[4];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    lo[j >> 1] = pack_h2((float)mn[j], (float)mn[j + 1]);
                    hi[j >> 1] = pack_h2(64.0f * (float)mn[j], 64.0f * (float)mn[j + 1]);
                }
                *reinterpret_cast<uint4 *>(ma + plain_off(t, 0)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(ma + plain_off(t, 1)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.min_full + mr.idx);
            mr.next();
        }

        // this half's two operand stages of 64 K (two sub-blocks each)
        const uint64_t lo64 = (uint64_t)h.y | ((uint64_t)h.z << 32);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int slot = 2 * hh + k;
            if (!wait_warp(B.a_empty + slot, par ^ 1u, abort)) return;
            uint8_t *A = smem + OFF_A + slot * OP_A;
            if (valid) {
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = 2 * k + jj;  // sub-block within this half
                    const float sc = (float)(int)((lo64 >> (6 * (4 * hh + j))) & 63);
                    const __half2 s1 = __float2half2_rn(sc), c1 = __float2half2_rn(-1024.0f * sc);
                    const __half2 s16 = __float2half2_rn(sc * 0.0625f), c16 = __float2half2_rn(-64.0f * sc);
                    const uint32_t wd[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4 *>(A + sw128_off(t, 4 * jj + i)) =
                            nibbles_to_f16(wd[i], s1, c1, s16, c16);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.a_full + slot);
        }
    }
}

// MMA issuer (warp 1, one thread).  Per super-block: sixteen K=16 steps into
// the S1 accumulator of this super-block's parity, committed to the stage
// barriers and to acc_full; then two K=16 bf16 steps into the min-term
// accumulator.  Always ends with a commit to `fin` so the epilogue (and the
// teardown) can wait for every MMA to finish.
__device__ void role_mma(uint8_t *smem, const Bars &B, uint32_t tmem, int nsb, volatile uint32_t *abort) {
    RingPos orr(NOP), br(NBR), mr(2);
    bool ok = true;
    for (int sb = 0; ok && sb < nsb; ++sb) {
        const int p = sb & 1;
        const uint32_t ph = (uint32_t)(sb >> 1) & 1u;
        if (!(ok = wait_or_abort(B.acc_empty + p, ph ^ 1u, abort))) break;
        tc_fence_after();
        for (int qq = 0; qq < NOP; ++qq) {
            if (!(ok = wait_or_abort(B.a_full + orr.idx, orr.phase, abort))) break;
            if (!(ok = wait_or_abort(B.b_tx + br.idx, br.phase, abort))) break;
            tc_fence_after();
            const uint32_t a = smem_u32(smem + OFF_A + orr.idx * OP_A);
            const uint32_t b = smem_u32(smem + OFF_B + br.idx * OP_B);
#pragma unroll
            for (int kk = 0; kk < KS / 16; ++kk)
                mma_f16(tmem + col_s1(p), desc_sw128(a + 32 * kk), desc_sw128(b + 32 * kk), IDESC_F16,
                        (qq | kk) != 0);
            mma_commit(B.a_empty + orr.idx);  // both slots free once these MMAs complete
            mma_commit(B.b_empty + br.idx);
            orr.next();
            br.next();
        }
        if (!ok) break;
        if (!(ok = wait_or_abort(B.min_full + mr.idx, mr.phase, abort))) break;
        if (!(ok = wait_or_abort(B.min_tx + mr.idx, mr.phase, abort))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + OFF_MIN + mr.idx * MIN_STAGE);
        mma_f16(tmem + col_s2(p), desc_plain(a, 128, 256), desc_plain(a + MIN_A, 128, 256), IDESC_F16, 0u);
        mma_commit(B.min_empty + mr.idx);
        mr.next();
        mma_commit(B.acc_full + p);  // S1 and S2 of this super-block are ready
    }
    mma_commit(B.fin);
}

// Epilogue (warps 12-27): warp w reads tensor-memory lanes 32 (w % 4) .. + 31
// (its 32 rows) and columns 32 h .. + 31, h = (w - 12) / 4.
template <bool SUMS>
__device__ void role_epilogue(uint8_t *smem, const Bars &B, uint32_t tmem, int row0, int rows, int ct,
                              int nsb, int batch, float *__restrict__ y, int32_t *__restrict__ sums,
                              const uint8_t *__restrict__ xq, volatile uint32_t *abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lq = warp & 3, h = (warp - EPI_WARP0) >> 2;
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
        if (!(ok = wait_warp(B.acc_full + p, ph, abort))) break;
        if (!(ok = wait_warp(B.meta_full + p, ph, abort))) break;
        if (!(ok = wait_warp(B.meta_tx + p, ph, abort))) break;
        tc_fence_after();
        const uint8_t *meta = smem + OFF_META + p * META_STAGE;
        const float d = reinterpret_cast<const float *>(meta + META_D)[r];
        const float dmin = reinterpret_cast<const float *>(meta + META_DMIN)[r];
        const float *dx = reinterpret_cast<const float *>(meta + META_DX) + 32 * h;
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 16) {
            float s1[16], s2[16];
            tmem_ld16(lane_addr + col_s1(p) + c0, s1);
            tmem_ld16(lane_addr + col_s2(p) + c0, s2);
            if (SUMS) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int b = ct * TN + 32 * h + c0 + i;
                    if (row < rows && b < batch) {
                        int32_t *o = sums + (((size_t)b * rows + row) * nsb + sb) * 2;
                        o[0] = (int32_t)s1[i];
                        o[1] = (int32_t)s2[i];
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    yacc[c0 + i] = fmaf(dx[c0 + i], d * s1[i] - dmin * s2[i], yacc[c0 + i]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(B.acc_empty + p);
            mbar_arrive(B.meta_empty + p);
        }
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

template <bool SUMS>
__global__ void __launch_bounds__(NTHREADS, 1) mma_q4k_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                              const uint8_t *__restrict__ ws,
                                                              const uint8_t *__restrict__ xq,
                                                              float *__restrict__ y,
                                                              int32_t *__restrict__ sums, int rows,
                                                              int nsb, int batch,
                                                              uint32_t *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Bars B = bars_at(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // column tiles vary fastest, so the CTAs that read the same weight rows
    // run together and share them through L2
    const int row0 = blockIdx.y * TM, ct = blockIdx.x;
    const int nvalid = min(TM, rows - row0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NOP; ++i) {
            mbar_init(B.a_full + i, 4);
            mbar_init(B.a_empty + i, 1);
        }
        for (int i = 0; i < NBR; ++i) {
            mbar_init(B.b_tx + i, 1);
            mbar_init(B.b_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B.min_full + i, 4);
            mbar_init(B.min_tx + i, 1);
            mbar_init(B.min_empty + i, 1);
            mbar_init(B.meta_full + i, TM);
            mbar_init(B.meta_tx + i, 1);
            mbar_init(B.meta_empty + i, EPI_WARPS);
            mbar_init(B.acc_full + i, 1);
            mbar_init(B.acc_empty + i, EPI_WARPS);
        }
        for (int i = 0; i < NRAW; ++i) {
            mbar_init(B.raw_full + i, 1);
            mbar_init(B.raw_empty + i, BLD_THREADS);
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

    if (warp == 0) {
        role_producer_b(smem, B, ws, nsb, ct, abort);
    } else if (warp == 2) {
        role_producer_w(smem, B, &tmap_w, ws, row0, nsb, ct, abort);
    } else if (warp == 1) {
        if (lane == 0) role_mma(smem, B, tmem, nsb, abort);
        __syncwarp();
    } else if (warp >= BLD_WARP0 && warp < EPI_WARP0) {
        role_builder(smem, B, threadIdx.x - 32 * BLD_WARP0, nvalid, nsb, abort);
    } else if (warp >= EPI_WARP0) {
        role_epilogue<SUMS>(smem, B, tmem, row0, rows, ct, nsb, batch, y, sums, xq, abort);
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
    return (size_t)((batch + TN - 1) / TN) * (size_t)(cols / QK_K) * WS_UNIT;
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
// dependency on the driver library).
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

cudaError_t launch_mma_q4k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                           int64_t cols, int64_t batch, void *workspace, const LaunchCtx &ctx) {
    const int nsb = (int)(cols / QK_K);
    const int ctiles = (int)((batch + TN - 1) / TN);
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
    cudaError_t e = launch_pdl(pack_kernel, dim3(nsb, ctiles), dim3(256), 0, ctx.stream,
                               static_cast<const uint8_t *>(xq), ws, nsb, (int)batch);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)ctiles, (unsigned)rtiles);
    if (sums) {
        auto k = mma_q4k_kernel<true>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        return launch_pdl(k, grid, dim3(NTHREADS), SMEM_ALLOC, ctx.stream, tmap, (const uint8_t *)ws,
                          static_cast<const uint8_t *>(xq), y, sums, (int)rows, nsb, (int)batch, ctx.status);
    }
    auto k = mma_q4k_kernel<false>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, grid, dim3(NTHREADS), SMEM_ALLOC, ctx.stream, tmap, (const uint8_t *)ws,
                      static_cast<const uint8_t *>(xq), y, sums, (int)rows, nsb, (int)batch, ctx.status);
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
