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
// Work split: one CTA per (256 positions, head); each warp takes 32
// consecutive positions, whose key rows are one contiguous span (32 rows x
// row_bytes, a multiple of 16 bytes).  The warp copies the span into shared
// memory with coalesced 16-byte loads, then lane l computes the dot of row
// p0 + l.  The query is quantized once per CTA (warp j: block j) with the
// standalone quantizer's arithmetic, so its codes equal gq_quantize_rows'.
#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr int KV_WARPS = 8;
constexpr int KV_POS = 32;     // positions per warp
constexpr int KV_MAX_NB = 8;   // head_dim <= 256

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

// WT = GQ_Q8_0 or GQ_Q4_0 key blocks.  Q4_0 codes are c - 8 with c the stored
// nibble (element 2j low, 2j + 1 high in byte j), so the block sum is
// sum c a - 8 sum a; the query codes are kept split per group of eight as
// (a0, a2, a4, a6 | a1, a3, a5, a7) so a nibble word feeds dp4a directly.
template <int WT>
__global__ void __launch_bounds__(KV_WARPS * 32) kv_scores_kernel(const uint8_t *__restrict__ cache,
                                                                  const float *__restrict__ q,
                                                                  float *__restrict__ scores, int nb,
                                                                  int capacity, int n_pos) {
    constexpr int BB = WT == GQ_Q8_0 ? Q8_0_BYTES : Q4_0_BYTES;
    constexpr bool SPLIT = WT == GQ_Q4_0;
    extern __shared__ __align__(16) uint8_t kv_smem[];
    __shared__ __align__(16) int8_t qc[KV_MAX_NB][32];
    __shared__ float qd[KV_MAX_NB];
    __shared__ int qsum[KV_MAX_NB];
    const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_bytes = nb * BB;
    pdl_launch_dependents();
    pdl_wait();  // the cache and the query may come from the preceding kernels

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

    const int p0 = (blockIdx.x * KV_WARPS + warp) * KV_POS;
    if (p0 >= n_pos) return;
    // the 32 key rows of positions p0 .. p0 + 31 (inside the cache: capacity
    // is a multiple of 32) into this warp's staging area
    const uint8_t *src = cache + ((size_t)h * capacity + p0) * row_bytes;
    uint8_t *st = kv_smem + (size_t)warp * KV_POS * row_bytes;
    const int nchunk = KV_POS * row_bytes / 16;
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

    const uint8_t *row = st + lane * row_bytes;
    float acc = 0.0f;
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
    if (p0 + lane < n_pos) scores[(size_t)h * n_pos + p0 + lane] = acc;
}

}  // namespace

cudaError_t launch_kv_scores(gq_type t, const void *cache, const float *q, float *scores, int64_t n_heads,
                             int64_t head_dim, int64_t capacity, int64_t n_pos, const LaunchCtx &ctx) {
    const int nb = (int)(head_dim / 32);
    if (nb < 1 || nb > KV_MAX_NB || capacity % KV_POS != 0 || n_heads > 65535) return cudaErrorInvalidValue;
    const int bb = t == GQ_Q8_0 ? Q8_0_BYTES : Q4_0_BYTES;
    const size_t smem = (size_t)KV_WARPS * KV_POS * nb * bb + 16;  // + tail pad for the word reads
    const dim3 grid((unsigned)((n_pos + KV_WARPS * KV_POS - 1) / (KV_WARPS * KV_POS)), (unsigned)n_heads);
    const uint8_t *c8 = static_cast<const uint8_t *>(cache);
    if (t == GQ_Q8_0) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kv_scores_kernel<GQ_Q8_0>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(kv_scores_kernel<GQ_Q8_0>, grid, dim3(KV_WARPS * 32), smem, ctx.stream, c8, q, scores,
                          nb, (int)capacity, (int)n_pos);
    }
    if (t == GQ_Q4_0) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kv_scores_kernel<GQ_Q4_0>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(kv_scores_kernel<GQ_Q4_0>, grid, dim3(KV_WARPS * 32), smem, ctx.stream, c8, q, scores,
                          nb, (int)capacity, (int)n_pos);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gq
