// gq_kv.cu -- quantized KV cache: the int8 dot of a query with every cached
// key.  "llama.cpp 推理引擎" §3.7.3 (KV Cache 量化) stores the attention keys
// and values as Q8_0 or Q4_0 blocks to cut long-context memory; the
// attention scores are then block dot products of the cached key codes with
// the query quantized to Q8_0 -- the same per-block integer dot, scaled by
// both block scales, as the GEMV (§5.1, §6.4), with cache positions as rows.
//
// Cache layout: [n_heads][capacity][head_dim / 32] blocks; key row (h, p) is
// head_dim / 32 consecutive blocks, rows of a head are consecutive.
//
// Work split: one CTA per (8 x PW positions, head); each warp takes PW
// consecutive positions (PW = 32, or 64 when 32 rows are under 4 KB and the
// capacity is a multiple of 64), whose key rows are one contiguous span (PW
// rows x row_bytes, a multiple of 16 bytes).  The warp copies the span into
// shared memory -- one bulk copy (TMA) when it is at least 4 KB, else
// coalesced 16-byte loads -- then lane l computes the dots of rows l, l + 32,
// ... of the span.  The query is quantized once per CTA (warp j: block j)
// with the standalone quantizer's arithmetic, so its codes equal
// gq_quantize_rows'.
#include <atomic>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr int KV_WARPS = 8;
constexpr int KV_POS = 32;     // positions per warp
constexpr int KV_MAX_NB = 8;   // head_dim <= 256

// Test switch for the timeout path (set by gq_debug_kv_timeout, passed to
// the kernel as an argument): warp 0 of every CTA arms its transfer barrier
// for its span but issues no copy, so the barrier never completes and its
// bounded wait -- shortened to DEBUG_WAIT_LIMIT polls -- runs out.  No copy
// is in flight when the warp gives up and leaves; nothing faults or hangs.
std::atomic<int> g_kv_debug_timeout{0};
constexpr uint32_t DEBUG_WAIT_LIMIT = 4096;

__device__ __forceinline__ float warp_max32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

// Two bytes at a 2-byte aligned shared-memory address.
__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p) {
    return *reinterpret_cast<const uint16_t *>(p);
}

// The NW 32-bit words starting at the 2-byte aligned shared-memory address
// p, read as NW + 1 aligned words and funnel-shifted into place (reads up to
// 4 bytes past the last word: the staging area carries a tail pad).
template <int NW>
__device__ __forceinline__ void lds_words_a2(const uint8_t *p, uint32_t (&w)[NW]) {
    const uint32_t *a = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(p) & 3u) * 8u;  // 0 or 16
    uint32_t r[NW + 1];
#pragma unroll
    for (int i = 0; i <= NW; ++i) r[i] = a[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) w[i] = __funnelshift_r(r[i], r[i + 1], sh);
}

// 32 bits at byte offset O of a row held as 64-bit words (O a compile-time
// constant once the loops are unrolled).
template <int O, int N64>
__device__ __forceinline__ uint32_t row_u32(const uint64_t (&r)[N64]) {
    constexpr int W = O / 8, B = O % 8;
    if (B <= 4) return (uint32_t)(r[W] >> (8 * B));
    return (uint32_t)((r[W] >> (8 * B)) | (r[W + 1] << (64 - 8 * B)));
}

// Dot of the key row (NB blocks, held as 64-bit words) with the query codes.
template <int WT, int NB, int J = 0, int N64>
__device__ __forceinline__ float row_dot(const uint64_t (&r)[N64], const int8_t (*qc)[32], const float *qd,
                                         const int *qsum, float acc) {
    if constexpr (J == NB) {
        return acc;
    } else {
        constexpr int BB = WT == GQ_Q8_0 ? Q8_0_BYTES : Q4_0_BYTES;
        constexpr int O = J * BB;
        const float dk = half_bits_to_float(row_u32<O, N64>(r) & 0xffffu);
        const int *qw = reinterpret_cast<const int *>(qc[J]);
        int s = 0;
        if constexpr (WT == GQ_Q8_0) {
            s = dp4a((int)row_u32<O + 2, N64>(r), qw[0], s);
            s = dp4a((int)row_u32<O + 6, N64>(r), qw[1], s);
            s = dp4a((int)row_u32<O + 10, N64>(r), qw[2], s);
            s = dp4a((int)row_u32<O + 14, N64>(r), qw[3], s);
            s = dp4a((int)row_u32<O + 18, N64>(r), qw[4], s);
            s = dp4a((int)row_u32<O + 22, N64>(r), qw[5], s);
            s = dp4a((int)row_u32<O + 26, N64>(r), qw[6], s);
            s = dp4a((int)row_u32<O + 30, N64>(r), qw[7], s);
        } else {
            const uint32_t w0 = row_u32<O + 2, N64>(r), w1 = row_u32<O + 6, N64>(r);
            const uint32_t w2 = row_u32<O + 10, N64>(r), w3 = row_u32<O + 14, N64>(r);
            s = dp4a_us(w0 & NIB, qw[0], s);
            s = dp4a_us((w0 >> 4) & NIB, qw[1], s);
            s = dp4a_us(w1 & NIB, qw[2], s);
            s = dp4a_us((w1 >> 4) & NIB, qw[3], s);
            s = dp4a_us(w2 & NIB, qw[4], s);
            s = dp4a_us((w2 >> 4) & NIB, qw[5], s);
            s = dp4a_us(w3 & NIB, qw[6], s);
            s = dp4a_us((w3 >> 4) & NIB, qw[7], s);
            s -= 8 * qsum[J];
        }
        acc = fmaf(dk * qd[J], (float)s, acc);
        return row_dot<WT, NB, J + 1>(r, qc, qd, qsum, acc);
    }
}

// WT = GQ_Q8_0 or GQ_Q4_0 key blocks.  Q4_0 codes are c - 8 with c the stored
// nibble (element 2j low, 2j + 1 high in byte j), so the block sum is
// sum c a - 8 sum a; the query codes are kept split per group of eight as
// (a0, a2, a4, a6 | a1, a3, a5, a7) so a nibble word feeds dp4a directly.
// NBC = 4 or 8 (head_dim 128 or 256): rows are 8-byte aligned and each lane
// reads its row with 64-bit shared-memory loads (conflict-free at 128),
// block fields extracted by compile-time shifts; NBC = 0: any head_dim, block
// fields read as funnel-shifted 32-bit words.
template <int WT, int NBC, int PW>
__global__ void __launch_bounds__(KV_WARPS * 32) kv_scores_kernel(const uint8_t *__restrict__ cache,
                                                                  const float *__restrict__ q,
                                                                  float *__restrict__ scores, int nb,
                                                                  int capacity, int n_pos,
                                                                  uint32_t *__restrict__ status,
                                                                  int debug_starve) {
    constexpr int BB = WT == GQ_Q8_0 ? Q8_0_BYTES : Q4_0_BYTES;
    constexpr bool SPLIT = WT == GQ_Q4_0;
    extern __shared__ __align__(16) uint8_t kv_smem[];
    __shared__ __align__(16) int8_t qc[KV_MAX_NB][32];
    __shared__ float qd[KV_MAX_NB];
    __shared__ int qsum[KV_MAX_NB];
    __shared__ uint64_t span_bar[KV_WARPS];
    const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_bytes = nb * BB;
    const int p0 = (blockIdx.x * KV_WARPS + warp) * PW;
    const uint32_t span = (uint32_t)(PW * row_bytes);  // a multiple of 16
    const bool bulk = span >= 4096;
    uint8_t *st = kv_smem + (size_t)warp * span;
    if (lane == 0) {
        mbar_init(span_bar + warp, 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_launch_dependents();
    pdl_wait();  // the cache and the query may come from the preceding kernels
    // the PW key rows of positions p0 .. p0 + PW - 1 (inside the cache:
    // capacity is a multiple of PW) into this warp's staging area, one bulk
    // copy
    const bool starve = debug_starve != 0 && warp == 0;
    const uint32_t limit = starve ? DEBUG_WAIT_LIMIT : WAIT_LIMIT;
    if (bulk && lane == 0 && p0 < n_pos) {
        mbar_arrive_expect_tx(span_bar + warp, span);
        if (!starve) bulk_g2s(st, cache + ((size_t)h * capacity + p0) * row_bytes, span, span_bar + warp);
    }

    // query block `warp`: amax, d = fp16(amax / 127), code = roundf(x / d)
    if (warp < nb) {
        const float v = q[((size_t)h * nb + warp) * 32 + lane];
        const float amax = warp_max32(fabsf(v));
        const float d = __half2float(__float2half_rn(__fdiv_rn(amax, 127.0f)));
        float c = d == 0.0f ? 0.0f : roundf(__fdiv_rn(v, d));
        c = c < -127.0f ? -127.0f : (c > 127.0f ? 127.0f : c);
        int ci = (int)c;
        const int e = lane & 7;
        const int pos = SPLIT ? ((lane & ~7) | ((e & 1) ? 4 + (e >> 1) : (e >> 1))) : lane;
        qc[warp][pos] = (int8_t)ci;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ci += __shfl_xor_sync(FULL, ci, o);
        if (lane == 0) {
            qd[warp] = d;
            qsum[warp] = ci;
        }
    }
    __syncthreads();

    if (p0 >= n_pos) return;
    if (bulk) {
        if (!mbar_wait_limit(span_bar + warp, 0u, limit)) {
            // the copy never completed: flag it and leave these scores
            // unwritten.  A real copy still in flight gets one more bounded
            // wait before the CTA may exit (after a timeout the scores and
            // the context are suspect); the test switch issued none.
            if (lane == 0) atomicOr(status, STATUS_KV_TMA_TIMEOUT);
            if (!starve) mbar_wait_limit(span_bar + warp, 0u, limit);
            return;
        }
    } else {
        const uint8_t *src = cache + ((size_t)h * capacity + p0) * row_bytes;
        const int nchunk = (int)(span / 16);
        for (int c0 = 0; c0 < nchunk; c0 += 8 * 32) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < nchunk) v[u] = ldg_nc_v4(src + (size_t)c * 16);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < nchunk) reinterpret_cast<uint4 *>(st)[c] = v[u];
            }
        }
        __syncwarp();
    }

#pragma unroll
    for (int rr = 0; rr < PW / 32; ++rr) {  // lane scores rows lane, lane + 32, ...
        const int pr = lane + 32 * rr;
        const uint8_t *row = st + pr * row_bytes;
        float acc = 0.0f;
        if constexpr (NBC != 0) {
            constexpr int N64 = NBC * BB / 8;
            uint64_t r[N64];
            const uint64_t *rp = reinterpret_cast<const uint64_t *>(row);
#pragma unroll
            for (int i = 0; i < N64; ++i) r[i] = rp[i];
            acc = row_dot<WT, NBC>(r, qc, qd, qsum, 0.0f);
        } else {
            for (int j = 0; j < nb; ++j) {
                const uint8_t *blk = row + j * BB;
                const float dk = half_bits_to_float(lds_u16(blk));
                const int *qw = reinterpret_cast<const int *>(qc[j]);
                int s = 0;
                if (WT == GQ_Q8_0) {
                    uint32_t w[8];
                    lds_words_a2<8>(blk + 2, w);
#pragma unroll
                    for (int k = 0; k < 8; ++k) s = dp4a((int)w[k], qw[k], s);
                } else {
                    uint32_t w[4];
                    lds_words_a2<4>(blk + 2, w);  // word k: elements 8k .. 8k + 7
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        s = dp4a_us(w[k] & NIB, qw[2 * k], s);
                        s = dp4a_us((w[k] >> 4) & NIB, qw[2 * k + 1], s);
                    }
                    s -= 8 * qsum[j];
                }
                acc = fmaf(dk * qd[j], (float)s, acc);
            }
        }
        if (p0 + pr < n_pos) scores[(size_t)h * n_pos + p0 + pr] = acc;
    }
}

template <int WT, int NBC, int PW>
cudaError_t launch_kv1(size_t row_bytes, int64_t n_heads, const LaunchCtx &ctx, const uint8_t *cache,
                       const float *q, float *scores, int nb, int64_t capacity, int64_t n_pos) {
    auto k = kv_scores_kernel<WT, NBC, PW>;
    const size_t smem = (size_t)KV_WARPS * PW * row_bytes + 16;  // + tail pad for the word reads
    const dim3 grid((unsigned)((n_pos + KV_WARPS * PW - 1) / (KV_WARPS * PW)), (unsigned)n_heads);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(k, grid, dim3(KV_WARPS * 32), smem, ctx.stream, cache, q, scores, nb, (int)capacity,
                      (int)n_pos, ctx.status, g_kv_debug_timeout.load());
}

// Positions per warp: 64 when a 32-row span is under 4 KB (so the bulk copy
// applies) and the capacity allows whole 64-row spans, else 32.
template <int WT, int NBC>
cudaError_t launch_kv(size_t row_bytes, int64_t n_heads, const LaunchCtx &ctx, const uint8_t *cache,
                      const float *q, float *scores, int nb, int64_t capacity, int64_t n_pos) {
    if (KV_POS * row_bytes < 4096 && capacity % (2 * KV_POS) == 0)
        return launch_kv1<WT, NBC, 2 * KV_POS>(row_bytes, n_heads, ctx, cache, q, scores, nb, capacity, n_pos);
    return launch_kv1<WT, NBC, KV_POS>(row_bytes, n_heads, ctx, cache, q, scores, nb, capacity, n_pos);
}

}  // namespace

cudaError_t kv_debug_timeout(int on) {
    g_kv_debug_timeout.store(on ? 1 : 0);
    return cudaSuccess;
}

cudaError_t launch_kv_scores(gq_type t, const void *cache, const float *q, float *scores, int64_t n_heads,
                             int64_t head_dim, int64_t capacity, int64_t n_pos, const LaunchCtx &ctx) {
    const int nb = (int)(head_dim / 32);
    if (nb < 1 || nb > KV_MAX_NB || capacity % KV_POS != 0 || n_heads > 65535) return cudaErrorInvalidValue;
    const size_t rb = (size_t)nb * (t == GQ_Q8_0 ? Q8_0_BYTES : Q4_0_BYTES);
    const uint8_t *c8 = static_cast<const uint8_t *>(cache);
    if (t == GQ_Q8_0) {
        if (nb == 4) return launch_kv<GQ_Q8_0, 4>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
        if (nb == 8) return launch_kv<GQ_Q8_0, 8>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
        return launch_kv<GQ_Q8_0, 0>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
    }
    if (t == GQ_Q4_0) {
        if (nb == 4) return launch_kv<GQ_Q4_0, 4>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
        if (nb == 8) return launch_kv<GQ_Q4_0, 8>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
        return launch_kv<GQ_Q4_0, 0>(rb, n_heads, ctx, c8, q, scores, nb, capacity, n_pos);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gq
