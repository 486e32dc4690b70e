// gq_gemv.cu -- memory-bound GEMV kernels (and their small-batch form) for
// Q4_K x Q8_K, Q4_0 x Q8_0 and Q8_0 x Q8_0.
//
// The per-block integer dot of "llama.cpp 推理引擎" (runguoli.com) §6.4 --
// low nibble of byte j pairs with activation 2j, high nibble with 2j+1, the
// block offset of 8 is applied to the integer sum, and the block scales
// multiply the integer result -- done with __dp4a on int8 activations, and
// the two-level Q4_K scales of §5.5 applied per 32-element sub-block in
// integers (sc_j * s_j, m_j * t_j) before one float scaling per super-block.
// Decode is bandwidth-bound ("llama.cpp 推理引擎" §7.3: token generation is
// limited by memory bandwidth), so the design goal is streaming the weights
// once at HBM speed:
//   - one warp per weight row, eight rows per 256-thread CTA;
//   - the CTA's activation vectors are staged once in shared memory, with
//     each group of 8 int8 codes stored as (a0,a2,a4,a6 | a1,a3,a5,a7) so a
//     packed nibble word w feeds dp4a directly as (w & 0x0F0F0F0F) and
//     ((w >> 4) & 0x0F0F0F0F);
//   - Q4_K rows (144-byte blocks, 16-byte aligned) are read with 128-bit
//     non-allocating global loads, issued for the whole first part of the
//     row before the activation staging so the two latencies overlap;
//   - Q4_0 / Q8_0 rows (18 / 34-byte blocks, only 2-byte aligned) are moved
//     into shared memory by the TMA engine (cp.async.bulk, 16-byte aligned
//     chunks of 64 blocks, two stages per warp) and unaligned blocks are
//     read from there with funnel shifts;
//   - warp-shuffle reduction of the per-lane partial sums.
#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr uint32_t NIB = 0x0F0F0F0Fu;
constexpr int WARPS = 8;  // rows per CTA

// ---------------------------------------------------------------- Q4_K x Q8_K

// Activation staging for Q8_K: per vector and super-block, 256 code bytes in
// the (even | odd) order, then the fp32 scale and the eight int32 sums.
struct ActK {
    uint8_t *codes;  // [nb][nsb][256]
    float *dx;       // [nb][nsb]
    int32_t *bsum;   // [nb][nsb][8]
};

__device__ __forceinline__ ActK act_k_layout(uint8_t *smem, int nb, int nsb) {
    ActK a;
    a.codes = smem;
    a.dx = reinterpret_cast<float *>(smem + (size_t)nb * nsb * 256);
    a.bsum = reinterpret_cast<int32_t *>(a.dx + (size_t)nb * nsb);
    return a;
}

__device__ __forceinline__ void stage_q8_k(const ActK &a, const uint8_t *__restrict__ xq,
                                           int nvec, int nsb) {
    const int groups = nvec * nsb * 32;
    for (int g = threadIdx.x; g < groups; g += blockDim.x) {
        const int blk = g >> 5, k = g & 31;
        const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + (size_t)blk * Q8_K_BYTES + 4 + 8 * k);
        const uint32_t a0 = __ldg(src), a1 = __ldg(src + 1);
        uint2 v;
        v.x = __byte_perm(a0, a1, 0x6420);
        v.y = __byte_perm(a0, a1, 0x7531);
        reinterpret_cast<uint2 *>(a.codes + (size_t)blk * 256)[k] = v;
    }
    for (int blk = threadIdx.x; blk < nvec * nsb; blk += blockDim.x) {
        const uint8_t *src = xq + (size_t)blk * Q8_K_BYTES;
        a.dx[blk] = __ldg(reinterpret_cast<const float *>(src));
        const uint32_t *bs = reinterpret_cast<const uint32_t *>(src + 260);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w = __ldg(bs + i);
            a.bsum[blk * 8 + 2 * i] = (int32_t)(int16_t)(w & 0xffffu);
            a.bsum[blk * 8 + 2 * i + 1] = (int32_t)(int16_t)(w >> 16);
        }
    }
}

// Sub-block factors of a Q4_K block header (bytes 0..15 as four words).
__device__ __forceinline__ void q4k_factors(const uint4 &h, int j, int &sc, int &m) {
    const uint64_t lo64 = (uint64_t)h.y | ((uint64_t)h.z << 32);  // header bits 32..95
    const uint64_t hi64 = (uint64_t)h.z | ((uint64_t)h.w << 32);  // header bits 64..127
    sc = (int)((lo64 >> (6 * j)) & 63);
    m = (int)((hi64 >> (6 * j + 16)) & 63);
}

// One lane = one 32-element sub-block j = lane & 7 of super-block
// 4 * iteration + (lane >> 3); a warp covers four super-blocks (576
// contiguous bytes) per iteration.  U iterations are kept in flight.
template <int NB, bool SUMS>
__global__ void __launch_bounds__(256) gemv_q4_k_kernel(const uint8_t *__restrict__ W,
                                                        const uint8_t *__restrict__ xq,
                                                        float *__restrict__ y,
                                                        int32_t *__restrict__ sums, int rows,
                                                        int nsb, int batch) {
    constexpr int U = 4;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * WARPS + warp;
    const int b0 = blockIdx.y * NB;
    const int nvec = min(NB, batch - b0);
    const int j = lane & 7, sbl = lane >> 3;
    const int iters = (nsb + 3) >> 2;
    const bool active = row < rows;
    const uint8_t *wrow = W + (size_t)(active ? row : 0) * nsb * Q4_K_BYTES;

    uint4 hdr[U], qs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int sb = 4 * u + sbl;
        if (active && u < iters && sb < nsb) {
            hdr[u] = ldg_nc_v4(wrow + (size_t)sb * Q4_K_BYTES);
            qs[u] = ldg_nc_v4(wrow + (size_t)sb * Q4_K_BYTES + 16 + 16 * j);
        }
    }

    const ActK act = act_k_layout(smem, NB, nsb);
    pdl_wait();  // activations may come from the preceding kernel
    stage_q8_k(act, xq + (size_t)b0 * nsb * Q8_K_BYTES, nvec, nsb);
    __syncthreads();
    pdl_launch_dependents();
    if (!active) return;

    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;

    for (int it0 = 0; it0 < iters; it0 += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int it = it0 + u;
            const int sb = 4 * it + sbl;
            if (it < iters && sb < nsb) {
                const uint32_t lo0 = qs[u].x & NIB, hi0 = (qs[u].x >> 4) & NIB;
                const uint32_t lo1 = qs[u].y & NIB, hi1 = (qs[u].y >> 4) & NIB;
                const uint32_t lo2 = qs[u].z & NIB, hi2 = (qs[u].z >> 4) & NIB;
                const uint32_t lo3 = qs[u].w & NIB, hi3 = (qs[u].w >> 4) & NIB;
                int sc, m;
                q4k_factors(hdr[u], j, sc, m);
                const float d = half_bits_to_float(hdr[u].x);
                const float dmin = half_bits_to_float(hdr[u].x >> 16);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b < nvec) {
                        const int blk = b * nsb + sb;
                        const int4 *ap = reinterpret_cast<const int4 *>(act.codes + (size_t)blk * 256 + 32 * j);
                        const int4 a0 = ap[0], a1 = ap[1];
                        int s = 0;
                        s = dp4a((int)lo0, a0.x, s);
                        s = dp4a((int)hi0, a0.y, s);
                        s = dp4a((int)lo1, a0.z, s);
                        s = dp4a((int)hi1, a0.w, s);
                        s = dp4a((int)lo2, a1.x, s);
                        s = dp4a((int)hi2, a1.y, s);
                        s = dp4a((int)lo3, a1.z, s);
                        s = dp4a((int)hi3, a1.w, s);
                        const int t = act.bsum[blk * 8 + j];
                        int is1 = sc * s, is2 = m * t;
                        if (SUMS) {
                            // lanes of super-blocks that exist in this iteration
                            const int cnt = min(4, nsb - 4 * it);
                            const unsigned gmask = 0xffffffffu >> (32 - 8 * cnt);
#pragma unroll
                            for (int o = 1; o < 8; o <<= 1) {
                                is1 += __shfl_xor_sync(gmask, is1, o);
                                is2 += __shfl_xor_sync(gmask, is2, o);
                            }
                            if (j == 0) {
                                int32_t *o = sums + (((size_t)(b0 + b) * rows + row) * nsb + sb) * 2;
                                o[0] = is1;
                                o[1] = is2;
                            }
                        } else {
                            acc[b] += act.dx[blk] * (d * (float)is1 - dmin * (float)is2);
                        }
                    }
                }
                // refill this slot with the iteration U ahead
                const int itn = it + U, sbn = 4 * itn + sbl;
                if (itn < iters && sbn < nsb) {
                    hdr[u] = ldg_nc_v4(wrow + (size_t)sbn * Q4_K_BYTES);
                    qs[u] = ldg_nc_v4(wrow + (size_t)sbn * Q4_K_BYTES + 16 + 16 * j);
                }
            }
        }
    }
    if (!SUMS) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < nvec) {
                const float v = warp_sum(acc[b]);
                if (lane == 0) y[(size_t)(b0 + b) * rows + row] = v;
            }
        }
    }
}

// ------------------------------------------------------- Q4_0 / Q8_0 x Q8_0

constexpr int CH_BLOCKS = 64;  // blocks per TMA chunk

struct Act0 {
    uint8_t *codes;  // [nb][nblk][32]
    float *dx;       // [nb][nblk]
    int32_t *asum;   // [nb][nblk]  (sum of the 32 codes, for the Q4_0 offset)
};

__device__ __forceinline__ Act0 act_0_layout(uint8_t *smem, int nb, int nblk) {
    Act0 a;
    a.codes = smem;
    a.dx = reinterpret_cast<float *>(smem + (size_t)nb * nblk * 32);
    a.asum = reinterpret_cast<int32_t *>(a.dx + (size_t)nb * nblk);
    return a;
}

// SPLIT: store each group of 8 codes as (even | odd) for nibble weights.
template <bool SPLIT>
__device__ __forceinline__ void stage_q8_0(const Act0 &a, const uint8_t *__restrict__ xq, int nvec,
                                           int nblk) {
    for (int blk = threadIdx.x; blk < nvec * nblk; blk += blockDim.x) {
        const uint16_t *src = reinterpret_cast<const uint16_t *>(xq + (size_t)blk * Q8_0_BYTES);
        a.dx[blk] = half_bits_to_float(__ldg(src));
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = (uint32_t)__ldg(src + 1 + 2 * i) | ((uint32_t)__ldg(src + 2 + 2 * i) << 16);
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = dp4a((int)w[i], 0x01010101, s);
        a.asum[blk] = s;
        uint4 *dst = reinterpret_cast<uint4 *>(a.codes + (size_t)blk * 32);
        if (SPLIT) {
            dst[0] = make_uint4(__byte_perm(w[0], w[1], 0x6420), __byte_perm(w[0], w[1], 0x7531),
                                __byte_perm(w[2], w[3], 0x6420), __byte_perm(w[2], w[3], 0x7531));
            dst[1] = make_uint4(__byte_perm(w[4], w[5], 0x6420), __byte_perm(w[4], w[5], 0x7531),
                                __byte_perm(w[6], w[7], 0x6420), __byte_perm(w[6], w[7], 0x7531));
        } else {
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

// Integer dot of the weight block that starts `off` bytes into a 4-byte
// aligned shared-memory chunk with the staged activation block `ap`.
template <bool Q4>
__device__ __forceinline__ int block_dot_smem(const uint8_t *chunk, int off, const int4 *ap,
                                              int asum, float &dw) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(chunk + (off & ~3));
    const uint32_t sh = (off & 2) ? 32u : 16u;  // code bytes start 2 or 4 bytes into w[0]
    const int4 a0 = ap[0], a1 = ap[1];
    if (Q4) {
        uint32_t v[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) v[i] = w[i];
        dw = half_bits_to_float((off & 2) ? (v[0] >> 16) : v[0]);
        const uint32_t c0 = __funnelshift_rc(v[0], v[1], sh), c1 = __funnelshift_rc(v[1], v[2], sh);
        const uint32_t c2 = __funnelshift_rc(v[2], v[3], sh), c3 = __funnelshift_rc(v[3], v[4], sh);
        int s = 0;
        s = dp4a((int)(c0 & NIB), a0.x, s);
        s = dp4a((int)((c0 >> 4) & NIB), a0.y, s);
        s = dp4a((int)(c1 & NIB), a0.z, s);
        s = dp4a((int)((c1 >> 4) & NIB), a0.w, s);
        s = dp4a((int)(c2 & NIB), a1.x, s);
        s = dp4a((int)((c2 >> 4) & NIB), a1.y, s);
        s = dp4a((int)(c3 & NIB), a1.z, s);
        s = dp4a((int)((c3 >> 4) & NIB), a1.w, s);
        return s - 8 * asum;
    } else {
        uint32_t v[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) v[i] = w[i];
        dw = half_bits_to_float((off & 2) ? (v[0] >> 16) : v[0]);
        int s = 0;
        s = dp4a((int)__funnelshift_rc(v[0], v[1], sh), a0.x, s);
        s = dp4a((int)__funnelshift_rc(v[1], v[2], sh), a0.y, s);
        s = dp4a((int)__funnelshift_rc(v[2], v[3], sh), a0.z, s);
        s = dp4a((int)__funnelshift_rc(v[3], v[4], sh), a0.w, s);
        s = dp4a((int)__funnelshift_rc(v[4], v[5], sh), a1.x, s);
        s = dp4a((int)__funnelshift_rc(v[5], v[6], sh), a1.y, s);
        s = dp4a((int)__funnelshift_rc(v[6], v[7], sh), a1.z, s);
        s = dp4a((int)__funnelshift_rc(v[7], v[8], sh), a1.w, s);
        return s;
    }
}

// Shared memory of the Q4_0 / Q8_0 kernel: per warp two chunk buffers (plus
// 16 bytes of slack for the last block's over-read) and two mbarriers, then
// the staged activations.
template <int BB>
struct ChunkLayout {
    static constexpr int CHUNK_BYTES = CH_BLOCKS * BB;
    static constexpr int BUF = ((CHUNK_BYTES + 16 + 15) / 16) * 16;
    static constexpr int PER_WARP = 2 * BUF;
    static constexpr int BARS_OFF = WARPS * PER_WARP;
    static constexpr int ACT_OFF = BARS_OFF + WARPS * 2 * 8;
};

template <bool Q4, int NB, bool SUMS>
__global__ void __launch_bounds__(256) gemv_q_0_kernel(const uint8_t *__restrict__ W,
                                                       const uint8_t *__restrict__ xq,
                                                       float *__restrict__ y,
                                                       int32_t *__restrict__ sums, int rows,
                                                       int nblk, int batch,
                                                       uint32_t *__restrict__ status) {
    constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    using L = ChunkLayout<BB>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * WARPS + warp;
    const int b0 = blockIdx.y * NB;
    const int nvec = min(NB, batch - b0);
    const bool active = row < rows;
    const int nchunks = (nblk + CH_BLOCKS - 1) / CH_BLOCKS;
    uint8_t *buf = smem + warp * L::PER_WARP;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::BARS_OFF) + 2 * warp;
    const uint8_t *wrow = W + (size_t)(active ? row : 0) * nblk * BB;

    auto issue = [&](int c) {
        const int nb_c = min(CH_BLOCKS, nblk - c * CH_BLOCKS);
        const uint32_t bytes = (uint32_t)(nb_c * BB);
        uint64_t *b = bar + (c & 1);
        mbar_arrive_expect_tx(b, bytes);
        bulk_g2s(buf + (c & 1) * L::BUF, wrow + (size_t)c * CH_BLOCKS * BB, bytes, b);
    };

    if (active && lane == 0) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        fence_mbar_init();
        issue(0);
        if (nchunks > 1) issue(1);
    }

    const Act0 act = act_0_layout(smem + L::ACT_OFF, NB, nblk);
    pdl_wait();
    stage_q8_0<Q4>(act, xq + (size_t)b0 * nblk * Q8_0_BYTES, nvec, nblk);
    __syncthreads();
    pdl_launch_dependents();
    if (!active) return;

    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.0f;

    for (int c = 0; c < nchunks; ++c) {
        if (!mbar_wait_bounded(bar + (c & 1), (uint32_t)(c >> 1) & 1u)) {
            // A transfer never completed: flag it, let the other stage drain
            // (bounded), and leave this row unwritten.
            if (lane == 0) atomicOr(status, STATUS_GEMV_TMA_TIMEOUT);
            if (c + 1 < nchunks) mbar_wait_bounded(bar + ((c + 1) & 1), (uint32_t)((c + 1) >> 1) & 1u);
            return;
        }
        const uint8_t *chunk = buf + (c & 1) * L::BUF;
        const int nb_c = min(CH_BLOCKS, nblk - c * CH_BLOCKS);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = lane + 32 * h;
            if (k < nb_c) {
                const int blk = c * CH_BLOCKS + k;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b < nvec) {
                        const int ab = b * nblk + blk;
                        float dw;
                        const int s = block_dot_smem<Q4>(
                            chunk, k * BB, reinterpret_cast<const int4 *>(act.codes + (size_t)ab * 32),
                            act.asum[ab], dw);
                        if (SUMS)
                            sums[((size_t)(b0 + b) * rows + row) * nblk + blk] = s;
                        else
                            acc[b] += dw * act.dx[ab] * (float)s;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && c + 2 < nchunks) issue(c + 2);
    }
    if (!SUMS) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < nvec) {
                const float v = warp_sum(acc[b]);
                if (lane == 0) y[(size_t)(b0 + b) * rows + row] = v;
            }
        }
    }
}

// Plain per-block kernel for Q4_0 / Q8_0 rows whose byte length is not a
// multiple of 16 (cols % 256 != 0): warp per row, lane per block, 16-bit
// global loads.
template <bool Q4, bool SUMS>
__global__ void __launch_bounds__(256) gemv_q_0_plain_kernel(const uint8_t *__restrict__ W,
                                                             const uint8_t *__restrict__ xq,
                                                             float *__restrict__ y,
                                                             int32_t *__restrict__ sums, int rows,
                                                             int nblk, int batch) {
    constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * WARPS + warp;
    const int b = blockIdx.y;
    pdl_wait();
    pdl_launch_dependents();
    if (row >= rows || b >= batch) return;
    float acc = 0.0f;
    for (int blk = lane; blk < nblk; blk += 32) {
        const uint16_t *wb = reinterpret_cast<const uint16_t *>(W + ((size_t)row * nblk + blk) * BB);
        const uint16_t *ab = reinterpret_cast<const uint16_t *>(xq + ((size_t)b * nblk + blk) * Q8_0_BYTES);
        int s = 0;
        if (Q4) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w2 = __ldg(wb + 1 + i);        // code bytes 2i, 2i+1
                const uint32_t a01 = __ldg(ab + 1 + 2 * i);   // activations 4i, 4i+1
                const uint32_t a23 = __ldg(ab + 2 + 2 * i);   // activations 4i+2, 4i+3
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

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int NB, bool SUMS>
cudaError_t launch_q4k(const void *W, const void *xq, float *y, int32_t *sums, int rows, int nsb,
                       int batch, const LaunchCtx &ctx) {
    const size_t smem = (size_t)NB * nsb * (256 + 4 + 32);
    auto k = gemv_q4_k_kernel<NB, SUMS>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((rows + WARPS - 1) / WARPS, (batch + NB - 1) / NB);
    return launch_pdl(k, grid, dim3(256), smem, ctx.stream, static_cast<const uint8_t *>(W),
                      static_cast<const uint8_t *>(xq), y, sums, rows, nsb, batch);
}

template <bool Q4, int NB, bool SUMS>
cudaError_t launch_q0(const void *W, const void *xq, float *y, int32_t *sums, int rows, int nblk,
                      int batch, const LaunchCtx &ctx) {
    using L = ChunkLayout<Q4 ? Q4_0_BYTES : Q8_0_BYTES>;
    const size_t smem = L::ACT_OFF + (size_t)NB * nblk * (32 + 4 + 4);
    auto k = gemv_q_0_kernel<Q4, NB, SUMS>;
    cudaError_t e = set_smem(k, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((rows + WARPS - 1) / WARPS, (batch + NB - 1) / NB);
    return launch_pdl(k, grid, dim3(256), smem, ctx.stream, static_cast<const uint8_t *>(W),
                      static_cast<const uint8_t *>(xq), y, sums, rows, nblk, batch, ctx.status);
}

// Batch chunk per launch: the largest NB in {1, 2, 4, 8} not above batch
// (bigger batches run as several chunks of 8 vectors in blockIdx.y).
template <bool SUMS>
cudaError_t dispatch(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums,
                     int rows, int cols, int batch, const LaunchCtx &ctx) {
    const int nb = batch >= 8 ? 8 : batch >= 4 ? 4 : batch >= 2 ? 2 : 1;
    if (wtype == GQ_Q4_K) {
        const int nsb = cols / QK_K;
        switch (nb) {
        case 1: return launch_q4k<1, SUMS>(W, xq, y, sums, rows, nsb, batch, ctx);
        case 2: return launch_q4k<2, SUMS>(W, xq, y, sums, rows, nsb, batch, ctx);
        case 4: return launch_q4k<4, SUMS>(W, xq, y, sums, rows, nsb, batch, ctx);
        default: return launch_q4k<8, SUMS>(W, xq, y, sums, rows, nsb, batch, ctx);
        }
    }
    const int nblk = cols / 32;
    const bool q4 = wtype == GQ_Q4_0;
    if (cols % 256 != 0) {
        dim3 grid((rows + WARPS - 1) / WARPS, batch);
        if (q4)
            return launch_pdl(gemv_q_0_plain_kernel<true, SUMS>, grid, dim3(256), 0, ctx.stream,
                              static_cast<const uint8_t *>(W), static_cast<const uint8_t *>(xq), y,
                              sums, rows, nblk, batch);
        return launch_pdl(gemv_q_0_plain_kernel<false, SUMS>, grid, dim3(256), 0, ctx.stream,
                          static_cast<const uint8_t *>(W), static_cast<const uint8_t *>(xq), y, sums,
                          rows, nblk, batch);
    }
    if (q4) {
        switch (nb) {
        case 1: return launch_q0<true, 1, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
        case 2: return launch_q0<true, 2, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
        case 4: return launch_q0<true, 4, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
        default: return launch_q0<true, 8, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
        }
    }
    switch (nb) {
    case 1: return launch_q0<false, 1, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
    case 2: return launch_q0<false, 2, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
    case 4: return launch_q0<false, 4, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
    default: return launch_q0<false, 8, SUMS>(W, xq, y, sums, rows, nblk, batch, ctx);
    }
}

}  // namespace

cudaError_t launch_gemv(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums,
                        int64_t rows, int64_t cols, int64_t batch, const LaunchCtx &ctx) {
    if (sums)
        return dispatch<true>(wtype, W, xq, y, sums, (int)rows, (int)cols, (int)batch, ctx);
    return dispatch<false>(wtype, W, xq, y, sums, (int)rows, (int)cols, (int)batch, ctx);
}

}  // namespace gq
