// gq_skinny.cu -- Q4_K (and Q5_K) x Q8_K for small batches (up to 64
// activation vectors per launch, 32 for Q5_K): the per-super-block product of
// "llama.cpp 推理引擎" §5.5 on warp-level tensor-core MMAs (mma.sync
// m16n8k16, fp16 operands, fp32 accumulate).
//
// Between the GEMV (one pass over W per eight vectors, its dp4a work growing
// with every vector) and the tcgen05 kernel (a CTA-wide pipeline whose
// per-super-block handshakes cost more than the MMAs at these widths) lies a
// band where the product is a skinny contraction bound by the weight stream.
// Here every compute warp owns 16 weight rows and does its own work: it turns
// the rows' nibbles into MMA A fragments in registers and issues the MMAs
// itself, with no hand-off to another role per super-block.
//
// Exactness (the integer sums of the tcgen05 kernel, same argument):
//   A = sc_j * q - 512 in [-512, 433], B = a in [-128, 127] (fp16, exact);
//   S1' = sum over the super-block of A * B, |S1'| <= 256 * 512 * 128 = 2^24,
//   so every partial sum is an exactly representable integer, and
//   S1 = S1' + 512 * asum with asum = sum of the column's 256 codes;
//   S2 = sum_j m_j * t_j by one more K = 16 step, t_j split exactly as
//   t_lo + 64 t_hi: A2 = [m | 64 m], B2 = [t_lo | t_hi] (|S2| < 2^21).
//   y += d_x * (d * S1 - dmin * S2) per super-block, in fp32.
// Q5_K (5-bit codes, the fifth bits in their own plane) uses A = sc_j * q -
// 1024 in [-1024, 929]: |S1'| reaches 2^25, so the even and odd sub-blocks
// accumulate apart (each within 2^24, exact) and S1 = S1'(even) + S1'(odd) +
// 1024 * asum is formed in int32.
//
// Operand order: within each 8-element group of a 32-element sub-block both
// operands use (e0, e4, e1, e5, e2, e6, e3, e7) -- the order in which a
// nibble word unpacks with the 0x6400 trick -- so lane (g, t) of the
// fragment takes elements 32 j + 8 t + 0..7 of its rows and columns.
//
// CTA (96 weight rows, 8 NT activation columns):
//   compute warps  KS groups of six (KS = 4 for 8 columns, 2 up to 32, else 1); group
//                  g takes the super-blocks sb = g (mod KS) of the 96 rows,
//                  and the groups' partial y are added in group order at the
//                  end (the int32 block sums are per super-block, exact);
//   producer warp  one 2-D TMA tile per super-block (144 or 176 bytes x 96 rows;
//                  rows past the matrix read as zeros) through a ring of NS;
//   converter warps (four) turn the Q8_K activation blocks, KC super-blocks
//                  at a time, into fp16 B fragments, min-term fragments and
//                  column scales in shared memory (two chunk buffers).
// Every mbarrier wait is bounded and reports through the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_tc.cuh"
#include "gq_mma_sync.cuh"


namespace gq {
namespace {

using namespace ms;

// Weight tiles requested before the dependency wait when W is static: two
// (more delay the activation loads queued behind them; 14336 x 4096: 11.9 /
// 15.6 / 22.1 us at batch 1 / 16 / 32 against 12.1 / 16.0 / 22.6 without and
// 12.6 / 15.9 / 22.3 with eight)
constexpr int SK_PRE = 2;
constexpr int SK_NW = 6;                   // row tiles of 16 per CTA
constexpr int SK_ROWS = 16 * SK_NW;        // weight rows per CTA
constexpr int SK_SM_SMEM = 233472;         // shared memory per SM (1 KB of it reserved per CTA)

// WT: Q4_K or Q5_K weights (the same super-block, 5-bit codes with a
// fifth-bit plane for Q5_K).
template <int WT, int NT_>
struct SkCfg {
    static constexpr bool Q5 = WT == GQ_Q5_K;
    static constexpr int BB = Q5 ? Q5_K_BYTES : Q4_K_BYTES;  // super-block bytes
    static constexpr int STAGE = SK_ROWS * BB;                // one ring stage: 13,824 / 16,896 bytes
    // A = sc q - OFFSET keeps every operand an fp16 integer below 1024 in
    // magnitude; S1 = S1' + OFFSET * asum
    static constexpr int OFFSET = Q5 ? 1024 : 512;
    // Q4_K: |S1'| <= 256 * 512 * 128 = 2^24 per super-block, one accumulator
    // is exact (two for narrow tiles, for the latency).  Q5_K: 2^25, so the
    // even and odd sub-blocks always accumulate apart (each <= 2^24, exact)
    // and meet in int32.
    static constexpr bool DUAL = Q5 || NT_ <= 2;
    static constexpr int NT = NT_;                       // 8-column N tiles
    static constexpr int BCOLS = 8 * NT_;
    // Tiles up to 32 columns split the super-blocks between KS groups of six
    // compute warps (group g takes the super-blocks sb = g mod KS of the same
    // 96 rows), so more independent warps cover the latency of each warp's
    // conversion and MMA chain; their partial y meet at the end.  Four groups
    // (64 registers a thread) pay off only for 8-column tiles: 12.8 vs 13.3 us
    // at 14336 x 4096 x 8, but 17.1 vs 16.7 us at 16 columns.
    static constexpr int KS = NT_ == 1 ? 4 : (NT_ <= 4 ? 2 : 1);
    static constexpr int NCW = SK_NW * KS;                 // compute warps
    static constexpr int CW = 4;                           // activation converter warps
    static constexpr int PRODUCER = NCW;                   // warp index of the weight producer
    static constexpr int CONV0 = NCW + 1;                  // first converter warp
    static constexpr int THREADS = 32 * (NCW + 1 + CW);
    static constexpr int MINB = 1;
    static constexpr int LIMIT = SK_SM_SMEM - 1024;
    // super-blocks per activation chunk: one L2 round trip of the converters
    // per chunk, so larger chunks for narrow tiles (eight: 12.0 vs 12.4 us at
    // batch 1, 16.0 vs 16.7 at 16, 22.6 vs 23.2 at 32 on 14336 x 4096)
    static constexpr int KC = NT_ == 1 ? 8 : (NT_ <= 4 ? 16 / NT_ : 2);
    static constexpr int PART = (KS - 1) * SK_NW * 32 * NT_ * 16;  // partial y of groups 1.. (float4 per lane and tile)
    // one activation chunk: B fragments [nt][sub-block of the chunk][lane]
    // (uint4: the two K = 16 steps of the sub-block), min-term B fragments
    // [nt][super-block of the chunk][lane] (uint2), column pairs (dx,
    // 512 * asum) [super-block of the chunk][column] (float2)
    static constexpr int BFRAG = NT_ * KC * 8 * 32 * 16;
    static constexpr int TFRAG = NT_ * KC * 32 * 8;
    static constexpr int COLF = KC * BCOLS * 8;
    static constexpr int CHUNK = BFRAG + TFRAG + COLF;
    static constexpr int OFF_CHUNK = 0;                  // 2 x CHUNK
    static constexpr int OFF_SCT = 2 * CHUNK;            // 64 x uint4 scale constants
    static constexpr int OFF_PART = OFF_SCT + 64 * 16;   // partial y of groups 1.. (KS > 1)
    static constexpr int OFF_RING = OFF_PART + PART;     // NS x STAGE
    static constexpr int FIXED = OFF_RING + 16 * 8 + 4 * 8 + 16 + 128;
    static constexpr int NS = (LIMIT - FIXED) / STAGE > 8 ? 8 : (LIMIT - FIXED) / STAGE;
    static constexpr int OFF_BAR = OFF_RING + NS * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + (2 * NS + 4) * 8;  // ring full / empty, chunk full / empty
    static constexpr int SMEM_ALLOC = OFF_MISC + 16 + 128;  // slack for the 128-byte alignment
    static_assert(NS >= 2, "ring");
    static_assert(THREADS <= 1024, "threads per CTA");
    static_assert(SMEM_ALLOC <= LIMIT, "shared memory budget");
    static_assert(OFF_RING % 128 == 0 && STAGE % 128 == 0, "TMA destinations");
    static_assert(!Q5 || NT_ <= 4, "Q5_K tiles hold at most 32 columns (registers of the dual accumulators)");
    static_assert(CHUNK % 16 == 0, "fragment alignment");
};

inline int pick_nt(int64_t batch) { return batch <= 8 ? 1 : batch <= 16 ? 2 : batch <= 32 ? 4 : 8; }

// One Q5_K nibble word w (byte i: element 2i low, 2i + 1 high) of lane t
// with its sub-block's fifth-bit word F (bit 2t + p of byte i: the fifth bit
// of element 2i + p of the lane's eight) to the fp16 pairs (v e0, v e4),
// (v e1, v e5), (v e2, v e6), (v e3, v e7), v e = sc q - 1024.  Every 5-bit
// code is placed in mantissa bits 4-8 of 0x6400 (fp16 1024 + 16 q) and one fma
// with k = (sc / 16, -64 sc - 1024) maps it exactly (a 1024 + q form would
// need the constant -1024 (sc + 1), below the fp16 range at sc = 63).
__device__ __forceinline__ uint4 nib5x8_to_f16(uint32_t w, uint32_t F, int t, uint4 k) {
    const uint32_t w8 = w >> 8, f = F >> (2 * t);
    const __half2 s16 = h2_bits(k.x), c = h2_bits(k.y);
    const uint32_t e04 = ((w << 4) & 0x00F000F0u) | ((f & 0x00010001u) << 8);
    const uint32_t e15 = (w & 0x00F000F0u) | (((f >> 1) & 0x00010001u) << 8);
    const uint32_t e26 = ((w8 << 4) & 0x00F000F0u) | (((f >> 8) & 0x00010001u) << 8);
    const uint32_t e37 = (w8 & 0x00F000F0u) | (((f >> 9) & 0x00010001u) << 8);
    return make_uint4(bits_h2(__hfma2(h2_bits(e04 | 0x64006400u), s16, c)),
                      bits_h2(__hfma2(h2_bits(e15 | 0x64006400u), s16, c)),
                      bits_h2(__hfma2(h2_bits(e26 | 0x64006400u), s16, c)),
                      bits_h2(__hfma2(h2_bits(e37 | 0x64006400u), s16, c)));
}

// 6-bit field f (0..15) of a Q4_K header's twelve scale bytes (words y, z, w).
__device__ __forceinline__ uint32_t field6(const uint4 &hd, int f) {
    const uint64_t lo = (uint64_t)hd.y | ((uint64_t)hd.z << 32);
    const int bit = 6 * f;
    if (bit + 6 <= 64) return (uint32_t)(lo >> bit) & 63u;
    const uint64_t hi = (uint64_t)hd.z | ((uint64_t)hd.w << 32);
    return (uint32_t)(hi >> (bit - 32)) & 63u;
}

// Activation chunk c (super-blocks c KC .. + kc - 1) into buffer `buf`, by the
// converter warps (thread tid of CW * 32).  Every global load of the chunk
// is issued before any value is converted, so a chunk costs one round trip
// to L2.  Columns past the batch are zeros.
//   B fragments: item (nt, jj, lane), jj a sub-block of the chunk: the eight
//     codes 32 j + 8 t .. + 7 of column 8 nt + lane / 4 as four fp16 pairs;
//   min-term B fragments: item (nt, sbk, lane): (t_lo, t_lo) and (t_hi, t_hi)
//     of sub-blocks 2t, 2t + 1 of that column;
//   column pairs (dx, 512 * asum): item (sbk, column).
template <class C>
__device__ void convert_chunk(uint8_t *buf, const uint8_t *__restrict__ xq, int c, int kc, int nsb, int batch,
                              int tid) {
    constexpr int NTH = 32 * C::CW;
    constexpr int NB = C::NT * C::KC * 8 * 32, UB = (NB + NTH - 1) / NTH;
    constexpr int NTI = C::NT * C::KC * 32, UT = (NTI + NTH - 1) / NTH;
    constexpr int NCI = C::KC * C::BCOLS, UC = (NCI + NTH - 1) / NTH;
    uint4 *bf = reinterpret_cast<uint4 *>(buf);
    uint2 *tf = reinterpret_cast<uint2 *>(buf + C::BFRAG);
    float2 *cf = reinterpret_cast<float2 *>(buf + C::BFRAG + C::TFRAG);
    auto block_of = [&](int n, int sbk) { return xq + ((size_t)n * nsb + c * C::KC + sbk) * Q8_K_BYTES; };
    uint32_t w0[UB], w1[UB], tw[UT], cw[UC][5];
#pragma unroll
    for (int u = 0; u < UB; ++u) {
        const int i = tid + u * NTH;
        const int ln = i & 31, jj = (i >> 5) % (C::KC * 8), nt = (i >> 5) / (C::KC * 8);
        const int n = 8 * nt + (ln >> 2), t = ln & 3;
        w0[u] = w1[u] = 0u;
        if (i < NB && jj < 8 * kc && n < batch) {
            const uint32_t *p = reinterpret_cast<const uint32_t *>(block_of(n, jj >> 3) + 4 + 32 * (jj & 7) + 8 * t);
            w0[u] = __ldg(p);
            w1[u] = __ldg(p + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < UT; ++u) {
        const int i = tid + u * NTH;
        const int ln = i & 31, sbk = (i >> 5) % C::KC, nt = (i >> 5) / C::KC;
        const int n = 8 * nt + (ln >> 2), t = ln & 3;
        tw[u] = 0u;
        if (i < NTI && sbk < kc && n < batch)
            tw[u] = __ldg(reinterpret_cast<const uint32_t *>(block_of(n, sbk) + 260 + 4 * t));
    }
#pragma unroll
    for (int u = 0; u < UC; ++u) {
        const int i = tid + u * NTH;
        const int sbk = i / C::BCOLS, n = i % C::BCOLS;
#pragma unroll
        for (int q = 0; q < 5; ++q) cw[u][q] = 0u;
        if (i < NCI && sbk < kc && n < batch) {
            const uint32_t *p = reinterpret_cast<const uint32_t *>(block_of(n, sbk));
            cw[u][0] = __ldg(p);  // dx
#pragma unroll
            for (int q = 0; q < 4; ++q) cw[u][1 + q] = __ldg(p + 65 + q);  // bsums (bytes 260..275)
        }
    }
#pragma unroll
    for (int u = 0; u < UB; ++u) {
        const int i = tid + u * NTH;
        if (i < NB) bf[i] = i8x8_to_f16(w0[u], w1[u]);  // zero codes convert to zeros
    }
#pragma unroll
    for (int u = 0; u < UT; ++u) {
        const int i = tid + u * NTH;
        if (i < NTI) {
            const int t0 = (int)(int16_t)(tw[u] & 0xffffu), t1 = (int)(int16_t)(tw[u] >> 16);
            const int h0 = t0 >> 6, h1 = t1 >> 6;  // floor(t / 64)
            tf[i] = make_uint2(pack_h2((float)(t0 - 64 * h0), (float)(t1 - 64 * h1)), pack_h2((float)h0, (float)h1));
        }
    }
#pragma unroll
    for (int u = 0; u < UC; ++u) {
        const int i = tid + u * NTH;
        if (i < NCI) {
            int asum = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) asum += (int)(int16_t)(cw[u][1 + q] & 0xffffu) + (int)(int16_t)(cw[u][1 + q] >> 16);
            // Q4_K: 512 asum as fp32 (below 2^24, exact); Q5_K: asum itself
            // (the int32 bits), since 1024 asum can exceed 2^24
            cf[i] = make_float2(__uint_as_float(cw[u][0]), C::Q5 ? __int_as_float(asum) : 512.0f * (float)asum);
        }
    }
}

template <int WT, int NT, bool SUMS>
__global__ void __launch_bounds__(SkCfg<WT, NT>::THREADS, SkCfg<WT, NT>::MINB) skinny_q4k_kernel(
    const __grid_constant__ CUtensorMap tmap_w, const uint8_t *__restrict__ xq, float *__restrict__ y,
    int32_t *__restrict__ sums, int rows, int nsb, int batch, int w_static, uint32_t *__restrict__ status) {
    using C = SkCfg<WT, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::NS;
    uint64_t *cfull = empty + C::NS;    // activation chunk buffer b converted (one arrival per converter warp)
    uint64_t *cempty = cfull + 2;       // activation chunk buffer b read (one arrival per compute warp)
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + C::OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * SK_ROWS;
    const int nchunks = (nsb + C::KC - 1) / C::KC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, SK_NW);  // the six warps of the super-block's group
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(cfull + i, C::CW);
            mbar_init(cempty + i, C::NCW);
        }
        *abort = 0u;
        fence_mbar_init();
    }
    // per-scale fma constants: Q4_K (nib8_to_f16) (sc, -512 (2 sc + 1),
    // sc / 16, -64 (sc + 8)); Q5_K (nib5x8_to_f16) (sc / 16, -64 sc - 1024)
    if (threadIdx.x < 64) {
        const float sc = (float)threadIdx.x;
        reinterpret_cast<uint4 *>(smem + C::OFF_SCT)[threadIdx.x] =
            C::Q5 ? make_uint4(pack_h2(sc * 0.0625f, sc * 0.0625f),
                               pack_h2(-64.0f * sc - 1024.0f, -64.0f * sc - 1024.0f), 0u, 0u)
                  : make_uint4(pack_h2(sc, sc), pack_h2(-512.0f * (2.0f * sc + 1.0f), -512.0f * (2.0f * sc + 1.0f)),
                               pack_h2(sc * 0.0625f, sc * 0.0625f), pack_h2(-64.0f * (sc + 8.0f), -64.0f * (sc + 8.0f)));
    }
    __syncthreads();
    // one 2-D TMA tile (the super-block's 96 rows) into ring slot `slot`
    auto issue_tile = [&](int sb, int slot) {
        mbar_arrive_expect_tx(full + slot, C::STAGE);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem + C::OFF_RING + slot * C::STAGE)),
            "l"(reinterpret_cast<uint64_t>(&tmap_w)), "r"(sb * C::BB), "r"(row0), "r"(smem_u32(full + slot))
            : "memory");
    };
    // Static weights (no kernel in flight writes W): the producer requests the
    // first SK_PRE tiles before the dependency wait, so the weight stream
    // starts during the preceding kernel's tail.
    const int pre = w_static ? min(SK_PRE, nsb) : 0;
    if (warp == C::PRODUCER && lane == 0)
        for (int sb = 0; sb < pre; ++sb) issue_tile(sb, sb);
    pdl_wait();  // the activations (and W, unless static) may come from the preceding kernel

    if (warp >= C::CONV0) {
        // converters: activation chunk c into buffer c & 1, once the compute
        // warps have released what it held (chunk c - 2)
        for (int c = 0; c < nchunks; ++c) {
            const int bi = c & 1;
            if (c >= 2 && !tc::wait_warp(cempty + bi, (uint32_t)((c - 2) >> 1) & 1u, abort)) break;
            convert_chunk<C>(smem + C::OFF_CHUNK + bi * C::CHUNK, xq, c, min(C::KC, nsb - c * C::KC), nsb, batch,
                             threadIdx.x - 32 * C::CONV0);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(cfull + bi);
        }
    } else if (warp == C::PRODUCER) {
        // producer: one 2-D TMA tile per super-block (the first `pre` are
        // already requested)
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
        // compute warps: row tile rw of the CTA, super-blocks sb = kg (mod KS)
        const int rw = warp % SK_NW, kg = warp / SK_NW;
        const int g = lane >> 2, t = lane & 3;
        const uint4 *sct = reinterpret_cast<const uint4 *>(smem + C::OFF_SCT);
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
            const uint2 *tf = reinterpret_cast<const uint2 *>(buf + C::BFRAG);
            const float4 *cf = reinterpret_cast<const float4 *>(buf + C::BFRAG + C::TFRAG);
            for (int sbk = 0; sbk < kc && ok; ++sbk) {
                const int sb = c * C::KC + sbk;
                if (sb % C::KS != kg) continue;
                const int si = sb % C::NS;
                if (!(ok = tc::wait_warp(full + si, (uint32_t)(sb / C::NS) & 1u, abort))) break;
                const uint8_t *rg = smem + C::OFF_RING + si * C::STAGE + (16 * rw + g) * C::BB;
                const uint8_t *rh = rg + 8 * C::BB;
                const uint4 hg = *reinterpret_cast<const uint4 *>(rg), hh = *reinterpret_cast<const uint4 *>(rh);
                // odd sub-blocks accumulate apart (C::DUAL): two MMA chains
                // side by side, both partial sums exact integers
                constexpr bool DUAL = C::DUAL;
                float s1[NT][4], s1b[NT][4], s2[NT][4];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s1[n][e] = s1b[n][e] = s2[n][e] = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t wg = *reinterpret_cast<const uint32_t *>(rg + 16 + 16 * j + 4 * t);
                    const uint32_t wh = *reinterpret_cast<const uint32_t *>(rh + 16 + 16 * j + 4 * t);
                    uint4 ag, ah;
                    if constexpr (C::Q5) {
                        const uint32_t fg = *reinterpret_cast<const uint32_t *>(rg + 144 + 4 * j);
                        const uint32_t fh = *reinterpret_cast<const uint32_t *>(rh + 144 + 4 * j);
                        ag = nib5x8_to_f16(wg, fg, t, sct[field6(hg, j)]);
                        ah = nib5x8_to_f16(wh, fh, t, sct[field6(hh, j)]);
                    } else {
                        ag = nib8_to_f16(wg, sct[field6(hg, j)]);
                        ah = nib8_to_f16(wh, sct[field6(hh, j)]);
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        const uint4 b = bf[(n * C::KC * 8 + sbk * 8 + j) * 32 + lane];
                        float(&acc)[4] = (DUAL && (j & 1)) ? s1b[n] : s1[n];
                        mma16816(acc, ag.x, ah.x, ag.y, ah.y, b.x, b.y);
                        mma16816(acc, ag.z, ah.z, ag.w, ah.w, b.z, b.w);
                    }
                }
                if (DUAL && !C::Q5) {
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) s1[n][e] += s1b[n][e];
                }
                // min term: A2 = [m_2t, m_2t+1 | 64 m_2t, 64 m_2t+1] per row
                const float mg0 = (float)field6(hg, 8 + 2 * t), mg1 = (float)field6(hg, 9 + 2 * t);
                const float mh0 = (float)field6(hh, 8 + 2 * t), mh1 = (float)field6(hh, 9 + 2 * t);
                const uint32_t a0 = pack_h2(mg0, mg1), a1 = pack_h2(mh0, mh1);
                const uint32_t a2 = pack_h2(64.0f * mg0, 64.0f * mg1), a3 = pack_h2(64.0f * mh0, 64.0f * mh1);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint2 b = tf[(n * C::KC + sbk) * 32 + lane];
                    mma16816(s2[n], a0, a1, a2, a3, b.x, b.y);
                }
                const float dg = half_bits_to_float(hg.x), dming = half_bits_to_float(hg.x >> 16);
                const float dh = half_bits_to_float(hh.x), dminh = half_bits_to_float(hh.x >> 16);
                // the stage is read; release it to the producer
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(empty + si);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    // columns 8 n + 2 t and + 1: (dx, 512 asum) of both
                    const float4 cv = cf[(sbk * C::BCOLS + 8 * n + 2 * t) / 2];
                    if constexpr (C::Q5) {
                        // S1 in int32: the two exact halves plus 1024 asum
                        int S1[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            S1[e] = __float2int_rn(s1[n][e]) + __float2int_rn(s1b[n][e]) +
                                    C::OFFSET * __float_as_int((e & 1) ? cv.w : cv.y);
                        if (SUMS) {
                            const int rr[2] = {row0 + 16 * rw + g, row0 + 16 * rw + g + 8};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int row = rr[e >> 1], b = 8 * n + 2 * t + (e & 1);
                                if (row < rows && b < batch) {
                                    int32_t *o = sums + (((size_t)b * rows + row) * nsb + sb) * 2;
                                    o[0] = S1[e];
                                    o[1] = (int32_t)s2[n][e];
                                }
                            }
                        } else {
                            yacc[n][0] = fmaf(cv.x, dg * (float)S1[0] - dming * s2[n][0], yacc[n][0]);
                            yacc[n][1] = fmaf(cv.z, dg * (float)S1[1] - dming * s2[n][1], yacc[n][1]);
                            yacc[n][2] = fmaf(cv.x, dh * (float)S1[2] - dminh * s2[n][2], yacc[n][2]);
                            yacc[n][3] = fmaf(cv.z, dh * (float)S1[3] - dminh * s2[n][3], yacc[n][3]);
                        }
                    } else if (SUMS) {
                        const int rr[2] = {row0 + 16 * rw + g, row0 + 16 * rw + g + 8};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = rr[e >> 1], b = 8 * n + 2 * t + (e & 1);
                            if (row < rows && b < batch) {
                                int32_t *o = sums + (((size_t)b * rows + row) * nsb + sb) * 2;
                                o[0] = (int32_t)s1[n][e] + (int32_t)((e & 1) ? cv.w : cv.y);
                                o[1] = (int32_t)s2[n][e];
                            }
                        }
                    } else {
                        yacc[n][0] = fmaf(cv.x, dg * (s1[n][0] + cv.y) - dming * s2[n][0], yacc[n][0]);
                        yacc[n][1] = fmaf(cv.z, dg * (s1[n][1] + cv.w) - dming * s2[n][1], yacc[n][1]);
                        yacc[n][2] = fmaf(cv.x, dh * (s1[n][2] + cv.y) - dminh * s2[n][2], yacc[n][2]);
                        yacc[n][3] = fmaf(cv.z, dh * (s1[n][3] + cv.w) - dminh * s2[n][3], yacc[n][3]);
                    }
                }
            }
            // this warp is done with the chunk's buffer
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(cempty + (c & 1));
        }
        if (!SUMS) {
            if (C::KS > 1) {
                // groups 1.. hand their partial y to group 0, which adds them
                // in group order; every compute warp reaches both barriers
                float4 *part = reinterpret_cast<float4 *>(smem + C::OFF_PART);
                if (kg > 0)
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        part[(((kg - 1) * SK_NW + rw) * NT + n) * 32 + lane] =
                            make_float4(yacc[n][0], yacc[n][1], yacc[n][2], yacc[n][3]);
                asm volatile("bar.sync 1, %0;" ::"r"(32 * C::NCW) : "memory");
                if (kg == 0)
                    for (int k = 1; k < C::KS; ++k)
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            const float4 v = part[(((k - 1) * SK_NW + rw) * NT + n) * 32 + lane];
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
                        const int row = rg + 8 * (e >> 1), b = 8 * n + 2 * t + (e & 1);
                        if (row < rows && b < batch) y[(size_t)b * rows + row] = yacc[n][e];
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
    using C = SkCfg<WT, NT>;
    auto k = sums ? skinny_q4k_kernel<WT, NT, true> : skinny_q4k_kernel<WT, NT, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((rows + SK_ROWS - 1) / SK_ROWS));
    return launch_pdl(k, grid, dim3(C::THREADS), C::SMEM_ALLOC, ctx.stream, tmap,
                      static_cast<const uint8_t *>(xq), y, sums, (int)rows, nsb, (int)batch, w_static ? 1 : 0,
                      ctx.status);
}

}  // namespace

int skinny_max_batch(gq_type wtype) { return wtype == GQ_Q5_K ? 32 : 64; }

bool skinny_supported(int64_t rows, int64_t cols, int64_t batch) {
    return rows >= 1 && batch >= 1 && batch <= 64 && cols >= QK_K && cols % QK_K == 0 &&
           (rows + SK_ROWS - 1) / SK_ROWS <= 0x7fffffff;
}

cudaError_t launch_skinny_q4k(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                              int64_t cols, int64_t batch, bool w_static, const LaunchCtx &ctx) {
    if (!skinny_supported(rows, cols, batch) || batch > skinny_max_batch(wtype) ||
        (wtype != GQ_Q4_K && wtype != GQ_Q5_K))
        return cudaErrorInvalidValue;
    const int nsb = (int)(cols / QK_K);
    const int bb = wtype == GQ_Q5_K ? Q5_K_BYTES : Q4_K_BYTES;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap tmap;
    // W as a 2-D byte tensor: rows of nsb super-blocks; box = one super-block
    // (144 or 176 bytes, both 16-byte multiples) of 96 rows
    const cuuint64_t gdim[2] = {(cuuint64_t)nsb * bb, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)nsb * bb};
    const cuuint32_t box[2] = {(cuuint32_t)bb, (cuuint32_t)SK_ROWS};
    const cuuint32_t estride[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (wtype == GQ_Q5_K) {
        switch (pick_nt(batch)) {
        case 1: return launch_nt<GQ_Q5_K, 1>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
        case 2: return launch_nt<GQ_Q5_K, 2>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
        default: return launch_nt<GQ_Q5_K, 4>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
        }
    }
    switch (pick_nt(batch)) {
    case 1: return launch_nt<GQ_Q4_K, 1>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    case 2: return launch_nt<GQ_Q4_K, 2>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    case 4: return launch_nt<GQ_Q4_K, 4>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    default: return launch_nt<GQ_Q4_K, 8>(tmap, xq, y, sums, rows, nsb, batch, w_static, ctx);
    }
}

}  // namespace gq
