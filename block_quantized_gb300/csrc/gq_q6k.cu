// gq_q6k.cu -- Q6_K weights: codec kernels and the Q6_K x Q8_K GEMV.
//
// Q6_K is the 6-bit K-quant as the discosf.com page ("为什么说 llama.cpp
// 是'裸引擎'——从模型加载的每一行代码说起", §4 量化不是"压缩"，而是"精度重分配")
// describes it: K blocks only (the 256-element K-quant block of
// "llama.cpp：一个人、一个周末…" 第二层：量化引擎), no sub-blocks, 6-bit main
// quantization.  The scale follows the symmetric rule of "llama.cpp 推理引擎"
// (runguoli.com) §5.1 with b = 6: d = fp16(max|x| / 31), q = round(x / d)
// clamped to [-32, 31] (half away from zero), stored as c = q + 32; w =
// d * (c - 32).  Block (194 B): fp16 d @0; 128 bytes @2 with the low four
// bits of element 2l (low nibble) and 2l+1 (high nibble) in byte l; 64 bytes
// @130 with the top two bits of elements 4l..4l+3 in byte l (element 4l+k in
// bits 2k..2k+1).  The product pairs Q6_K weights with Q8_K activations:
// per block s = sum_i (c_i - 32) * a_i (int32), y = sum_blocks d_w * d_x * s.
//
// This file is compiled with -fmad=false, and every division is __fdiv_rn,
// so the codec's bytes equal the reference definition's.
//
// GEMV.  Decode is bound by the bytes of W streamed ("llama.cpp 推理引擎"
// §7.3), so the kernel streams each row once:
//   - a persistent grid of at most one CTA per SM, 16 warps (8 when 16
//     two-stage rings do not fit); warp w of the grid owns rows w, w + warps,
//     ...  Each warp streams its rows through a private shared-memory ring of
//     2-4 whole-row stages, one bulk copy (cp.async.bulk, evict-first L2
//     policy) per row completing on an mbarrier; every wait is bounded;
//   - the CTA stages up to eight Q8_K activation vectors (the smallest group
//     of 1, 2, 4 or 8 that covers the batch, fewer when wide vectors leave no
//     room for the rings), so W streams once per group; each vector: codes in
//     128-byte half-super-block units, each 8-code group stored as (a0 a2 a4 a6 |
//     a1 a3 a5 a7) so that the masked low nibbles of a packed word line up
//     with dp4a operands, and the 16-byte pieces of a unit XOR-swizzled by
//     the unit index so that the lanes of a quarter-warp hit distinct banks;
//     then the sum of each unit's 128 codes and the per-block scales;
//   - a lane takes half a block (128 elements): 17 + 9 aligned 32-bit shared
//     loads realigned with funnel shifts (blocks are 194 bytes, so half of
//     them start 2 bytes off a word), the top bits spread into the code bytes
//     with shifts and masks once, 32 dp4a per staged vector; the offset 32 is
//     applied once per half through the code sum (s = sum c a - 32 sum a,
//     exact in int32);
//   - fp32 partial sums per lane and vector, one warp-shuffle reduction per
//     row and vector.  14336 x 4096 at batch 1 / 2 / 4 / 8: 12.1 / 13.5 /
//     17.3 / 24.9 us (one vector per pass: 12.1 / 22.2 / 42.4 / 80.3).
// Rows whose byte length is not a multiple of 16 (cols not a multiple of
// 2048), or too long for a two-stage ring, take a plain warp-per-row kernel
// with byte loads from global memory.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"
#include "gq_quant8.cuh"

namespace gq {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t NIB = 0x0F0F0F0Fu;

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

__device__ __forceinline__ float clamp_f(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// ------------------------------------------------------------------ codecs

// One warp per block; lane l owns elements 8l..8l+7, i.e. low-nibble bytes
// 4l..4l+3 and top-bit bytes 2l, 2l+1 of the block.
__global__ void __launch_bounds__(256) quantize_q6_k_kernel(const float *__restrict__ x,
                                                            uint8_t *__restrict__ dst, int64_t nblocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    pdl_launch_dependents();  // dependents still wait for this grid's completion
    pdl_wait();
    for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblocks; b += warps) {
        const float *src = x + b * QK_K + lane * 8;
        float v[8];
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[k] = src[k];
            amax = fmaxf(amax, fabsf(v[k]));
        }
        amax = warp_max_f(amax);
        const __half dh = __float2half_rn(__fdiv_rn(amax, 31.0f));
        const float d = __half2float(dh);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float q = (d == 0.0f) ? 0.0f : clamp_f(roundf(__fdiv_rn(v[k], d)), -32.0f, 31.0f);
            const uint32_t c = (uint32_t)((int)q + 32);  // 0..63
            lo |= (c & 15u) << (4 * k);                   // element 8l+k: byte 4l + k/2, nibble k&1
            hi |= (c >> 4) << (2 * k);                    // byte 2l + k/4, bits 2(k&3)
        }
        uint8_t *blk = dst + b * Q6_K_BYTES;  // 2-byte aligned
        uint16_t *ql = reinterpret_cast<uint16_t *>(blk + 2 + 4 * lane);
        ql[0] = (uint16_t)(lo & 0xffffu);
        ql[1] = (uint16_t)(lo >> 16);
        *reinterpret_cast<uint16_t *>(blk + 130 + 2 * lane) = (uint16_t)hi;
        if (lane == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(dh);
    }
}

// One thread per element: d * (c - 32), exact in fp32.
__global__ void dequantize_q6_k_kernel(const uint8_t *__restrict__ src, float *__restrict__ dst, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
        const uint8_t *blk = src + (e >> 8) * Q6_K_BYTES;
        const int i = (int)(e & 255);
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
        const int byte = blk[2 + (i >> 1)];
        const int lo = (i & 1) ? (byte >> 4) : (byte & 15);
        const int hi = (blk[130 + (i >> 2)] >> (2 * (i & 3))) & 3;
        dst[e] = __fmul_rn(d, (float)((lo | (hi << 4)) - 32));
    }
}

// ------------------------------------------------------------------- GEMV

// Independent dp4a accumulator chains per lane (1 or 2).
#ifndef GQ_Q6K_CHAINS
#define GQ_Q6K_CHAINS 1
#endif
constexpr int MAX_NS = 4;  // ring stages per warp
// the mbarriers, at the start of shared memory
__host__ __device__ constexpr int bars_bytes(int nw) { return nw * MAX_NS * 8; }

// Shared-memory footprint of one staged Q8_K vector of nblk blocks: codes,
// then one int32 code sum per half block, then one fp32 scale per block.
__host__ __device__ constexpr size_t act_smem_bytes(int nblk) {
    return (size_t)nblk * 256 + (size_t)nblk * 2 * 4 + (size_t)nblk * 4;
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
    int32_t *asum = reinterpret_cast<int32_t *>(act + (size_t)nblk * 256);
    float *dx = reinterpret_cast<float *>(asum + 2 * nblk);
    for (int idx = threadIdx.x; idx < nblk * 16; idx += blockDim.x) {
        const int hb = idx >> 3, u = idx & 7;
        const uint8_t *blk = xq + (size_t)(hb >> 1) * Q8_K_BYTES;  // 4-byte aligned
        const uint32_t *c = reinterpret_cast<const uint32_t *>(blk + 4 + (hb & 1) * 128 + u * 16);
        const uint2 g0 = split8(c[0], c[1]), g1 = split8(c[2], c[3]);
        *reinterpret_cast<uint4 *>(act + (size_t)hb * 128 + ((u ^ (hb & 7)) << 4)) =
            make_uint4(g0.x, g0.y, g1.x, g1.y);
    }
    for (int hb = threadIdx.x; hb < 2 * nblk; hb += blockDim.x) {
        const uint8_t *blk = xq + (size_t)(hb >> 1) * Q8_K_BYTES;
        const int16_t *bs = reinterpret_cast<const int16_t *>(blk + 260) + (hb & 1) * 4;
        asum[hb] = (int32_t)bs[0] + bs[1] + bs[2] + bs[3];
        if ((hb & 1) == 0) dx[hb >> 1] = *reinterpret_cast<const float *>(blk);
    }
}

// The top two bits of 4 elements (nibbles 0..3 of t, two bits each) moved to
// bits 4..5 of bytes 0..3.
__device__ __forceinline__ uint32_t spread_top(uint32_t t) {
    uint32_t x = (t & 0xffu) | ((t & 0xff00u) << 8);
    x = (x & 0x000f000fu) | ((x & 0x00f000f0u) << 4);
    return x << 4;
}

// Integer sums of half block h of the block at `blk` (shared memory, 2-byte
// aligned, at least 4 readable bytes past its end) against the staged codes
// of half-block hb of NV vectors (vector v at act + v * astride):
// sum_i c_i a_i over the 128 elements (offset not applied).  The 6-bit code
// words are built once and serve every vector.
template <int NV>
__device__ __forceinline__ void half_dot(const uint8_t *stage, uint32_t blk_off, int h, const uint8_t *act,
                                         size_t astride, int hb, int (&out)[NV]) {
    const uint32_t offa = blk_off + 2 + 64 * h;    // low-nibble bytes of the half
    const uint32_t offb = blk_off + 130 + 32 * h;  // top-bit bytes of the half
    const uint32_t *wa = reinterpret_cast<const uint32_t *>(stage + (offa & ~3u));
    const uint32_t *wb = reinterpret_cast<const uint32_t *>(stage + (offb & ~3u));
    const uint32_t sha = (offa & 3u) * 8, shb = (offb & 3u) * 8;
    uint32_t va[17], vb[9];
#pragma unroll
    for (int i = 0; i < 17; ++i) va[i] = wa[i];
#pragma unroll
    for (int i = 0; i < 9; ++i) vb[i] = wb[i];
    const uint8_t *ah = act + (size_t)hb * 128;
    const int sw = hb & 7;
    int s[NV], s2[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) s[v] = s2[v] = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const uint32_t top = __funnelshift_rc(vb[u], vb[u + 1], shb);  // top bits of elements 16u..16u+15
        uint32_t ca[2], cb[2];
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
            const int g = 2 * u + g2;
            const uint32_t w = __funnelshift_rc(va[g], va[g + 1], sha);  // low nibbles of elements 8g..8g+7
            const uint32_t t = g2 ? (top >> 16) : (top & 0xffffu);
            ca[g2] = (w & NIB) | spread_top(t & 0x3333u);                // elements 0, 2, 4, 6
            cb[g2] = ((w >> 4) & NIB) | spread_top((t >> 2) & 0x3333u);  // elements 1, 3, 5, 7
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint4 a = *reinterpret_cast<const uint4 *>(ah + (size_t)v * astride + ((u ^ sw) << 4));
            s[v] = dp4a((int)ca[0], (int)a.x, s[v]);
            s[v] = dp4a((int)ca[1], (int)a.z, s[v]);
            if (GQ_Q6K_CHAINS == 2) {
                s2[v] = dp4a((int)cb[0], (int)a.y, s2[v]);
                s2[v] = dp4a((int)cb[1], (int)a.w, s2[v]);
            } else {
                s[v] = dp4a((int)cb[0], (int)a.y, s[v]);
                s[v] = dp4a((int)cb[1], (int)a.w, s[v]);
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) out[v] = s[v] + s2[v];
}

// Streaming kernel: cols a multiple of 2048 (rows are 16-byte multiples);
// NV activation vectors per blockIdx.y (vectors NV y .. NV y + NV - 1 of the
// nvec in this launch), so W streams once per NV vectors.  SUMS: write the
// int32 block sums instead of y.
template <bool SUMS, int GW, bool FUSED, int NV>
__global__ void __launch_bounds__(GW * 32, 1) gemv_q6k_kernel(const uint8_t *__restrict__ W,
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
    const uint32_t row_bytes = (uint32_t)nblk * Q6_K_BYTES;
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
            q8::stage_q8_k_from_f32<2>(act + v * astride, static_cast<const float *>(act_in) + b * nblk * QK_K,
                                       nblk);
        else
            stage_q8_k_vec(act + v * astride, static_cast<const uint8_t *>(act_in) + b * nblk * Q8_K_BYTES, nblk);
    }
    __syncthreads();

    // within a staged vector: the half-block code sums, then the scales
    const size_t asum_off = (size_t)nblk * 256, dx_off = asum_off + (size_t)nblk * 2 * 4;
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
            int s[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) s[v] = 0;
            if (hb < 2 * nblk) {
                const int k = hb >> 1;
                half_dot<NV>(stage, (uint32_t)k * Q6_K_BYTES, hb & 1, act, astride, hb, s);
                const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t *>(stage + k * Q6_K_BYTES));
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const uint8_t *av = act + v * astride;
                    s[v] -= 32 * reinterpret_cast<const int32_t *>(av + asum_off)[hb];
                    if (!SUMS) acc[v] += dw * reinterpret_cast<const float *>(av + dx_off)[k] * (float)s[v];
                }
            }
            if (SUMS) {
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int both = s[v] + __shfl_xor_sync(FULL, s[v], 1);  // the two halves of block hb / 2
                    if (v < nv && hb < 2 * nblk && (hb & 1) == 0)
                        sums[((size_t)(b0 + v) * rows + row) * nblk + (hb >> 1)] = both;
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
__global__ void __launch_bounds__(PW * 32) gemv_q6k_plain_kernel(const uint8_t *__restrict__ W,
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
        int s = 0;
        float scale = 0.0f;
        if (hb < 2 * nblk) {
            const int k = hb >> 1, h = hb & 1;
            const uint8_t *wb = W + ((size_t)row * nblk + k) * Q6_K_BYTES;
            const uint8_t *ab = xq + ((size_t)b * nblk + k) * Q8_K_BYTES;
            for (int e = 128 * h; e < 128 * h + 128; ++e) {
                const int lo = (__ldg(wb + 2 + (e >> 1)) >> (4 * (e & 1))) & 15;
                const int hi = (__ldg(wb + 130 + (e >> 2)) >> (2 * (e & 3))) & 3;
                s += ((lo | (hi << 4)) - 32) * (int)(int8_t)__ldg(ab + 4 + e);
            }
            scale = half_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(wb))) *
                    __ldg(reinterpret_cast<const float *>(ab));
        }
        if (SUMS) {
            const int both = s + __shfl_xor_sync(FULL, s, 1);
            if (hb < 2 * nblk && (hb & 1) == 0) sums[((size_t)b * rows + row) * nblk + (hb >> 1)] = both;
        } else {
            acc += scale * (float)s;
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
    return bars_bytes(nw) + (size_t)nw * ns * ((size_t)nblk * Q6_K_BYTES + 16) + (size_t)nv * act_stride(nblk);
}

// Ring stages per warp for the streaming kernel with nw warps: as many as fit
// (2..4) next to nv staged vectors; 0 when rows are not 16-byte multiples or
// two stages do not fit.
int pick_ns(int nw, int nblk, int nv) {
    if (nblk % 8 != 0) return 0;
    for (int ns = MAX_NS; ns >= 2; --ns)
        if (stream_smem(nw, ns, nblk, nv) <= (size_t)SMEM_LIMIT) return ns;
    return 0;
}

// Launch shape of the streaming kernel for a batch: nv vectors per CTA (the
// smallest of 1, 2, 4, 8 that covers the batch, fewer when their staged
// copies leave no room for a two-stage ring), 16 warps when sixteen rings fit,
// else 8, and the ring depth.  ns == 0: the streaming kernel does not apply.
struct Shape {
    int nv, nw, ns;
};
Shape pick_shape(int nblk, int64_t batch) {
    int nv = batch >= 8 ? 8 : batch >= 4 ? (batch > 4 ? 8 : 4) : batch >= 2 ? (batch > 2 ? 4 : 2) : 1;
    for (; nv >= 1; nv >>= 1) {
        if (int ns = pick_ns(16, nblk, nv)) return {nv, 16, ns};
        if (int ns = pick_ns(8, nblk, nv)) return {nv, 8, ns};
    }
    return {1, 8, 0};
}

template <bool SUMS, int NW, bool FUSED, int NV>
cudaError_t launch_stream(const uint8_t *W, const void *xb, float *yb, int32_t *sb, int64_t rows, int nblk,
                          int nb, int ns, int w_static, const LaunchCtx &ctx) {
    auto k = gemv_q6k_kernel<SUMS, NW, FUSED, NV>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    const int64_t gx = std::min<int64_t>(ctx.num_sms, (rows + NW - 1) / NW);
    return launch_pdl(k, dim3((unsigned)gx, (nb + NV - 1) / NV), dim3(NW * 32), stream_smem(NW, ns, nblk, NV),
                      ctx.stream, W, xb, yb, sb, (int)rows, nblk, ns, nblk * Q6_K_BYTES + 16, nb, w_static,
                      ctx.status);
}

template <bool SUMS, bool FUSED, int NW>
cudaError_t launch_nv(const Shape &sh, const uint8_t *W, const void *xb, float *yb, int32_t *sb, int64_t rows,
                      int nblk, int nb, int w_static, const LaunchCtx &ctx) {
    switch (sh.nv) {
    case 8: return launch_stream<SUMS, NW, FUSED, 8>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    case 4: return launch_stream<SUMS, NW, FUSED, 4>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    case 2: return launch_stream<SUMS, NW, FUSED, 2>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    default: return launch_stream<SUMS, NW, FUSED, 1>(W, xb, yb, sb, rows, nblk, nb, sh.ns, w_static, ctx);
    }
}

int codec_grid(int64_t items, int per_cta, int num_sms) {
    int64_t g = (items + per_cta - 1) / per_cta;
    g = std::min<int64_t>(g, (int64_t)num_sms * 16);
    return (int)std::max<int64_t>(g, 1);
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
        int32_t *sb = SUMS ? sums + b0 * rows * nblk : nullptr;
        cudaError_t e;
        if (sh.ns && sh.nw == 16) {
            e = launch_nv<SUMS, FUSED, 16>(sh, W, xb, yb, sb, rows, nblk, nb, w_static, ctx);
        } else if (sh.ns) {
            e = launch_nv<SUMS, FUSED, 8>(sh, W, xb, yb, sb, rows, nblk, nb, w_static, ctx);
        } else {
            if (FUSED) return cudaErrorInvalidValue;  // one vector does not fit the streaming kernel
            const int64_t gx = (rows + PW - 1) / PW;
            e = launch_pdl(gemv_q6k_plain_kernel<SUMS>, dim3((unsigned)gx, nb), dim3(PW * 32), 0, ctx.stream, W,
                           static_cast<const uint8_t *>(xb), yb, sb, (int)rows, nblk);
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_quantize_q6k(const float *src, void *dst, int64_t n, const LaunchCtx &ctx) {
    const int64_t nb = n / QK_K;
    return launch_pdl(quantize_q6_k_kernel, codec_grid(nb, 8, ctx.num_sms), 256, 0, ctx.stream, src,
                      static_cast<uint8_t *>(dst), nb);
}

cudaError_t launch_dequantize_q6k(const void *src, float *dst, int64_t n, const LaunchCtx &ctx) {
    return launch_pdl(dequantize_q6_k_kernel, codec_grid(n, 256, ctx.num_sms), 256, 0, ctx.stream,
                      static_cast<const uint8_t *>(src), dst, n);
}

// The fused form has no plain-kernel fallback: the whole vector must fit the
// streaming kernel next to a two-stage ring.
bool gemv_q6k_fused_fits(int64_t cols) {
    if (cols < 0 || cols % QK_K != 0 || cols > (int64_t)1 << 20) return false;
    return pick_shape((int)(cols / QK_K), 1).ns > 0;
}

cudaError_t launch_gemv_q6k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t cols,
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
