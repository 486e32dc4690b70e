// gq_internal.h -- host-side interface between the API translation unit and
// the kernel translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gq.h"

namespace gq {

struct LaunchCtx;

// Launch with programmatic stream serialization allowed, so a kernel's
// prologue (weight prefetch) may overlap the tail of the previous kernel in
// the stream; every kernel calls griddepcontrol.wait before it touches data
// another kernel may produce or consume.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_quantize(gq_type t, const float *src, void *dst, int64_t n,
                            const LaunchCtx &ctx);
cudaError_t launch_dequantize(gq_type t, const void *src, float *dst, int64_t n,
                              const LaunchCtx &ctx);
// The error-minimizing Q4_K / Q5_K encoder (GQ_QUANT_ERRMIN).
cudaError_t launch_quantize_k_errmin(gq_type t, const float *src, void *dst, int64_t n, const LaunchCtx &ctx);
// Q8_0 / Q4_0 quantize of `rows` rows of row_blocks blocks each, destination
// rows dst_row_stride blocks apart (the KV-cache append).
cudaError_t launch_quantize_rows_strided(gq_type t, const float *src, void *dst, int64_t rows,
                                         int64_t row_blocks, int64_t dst_row_stride, const LaunchCtx &ctx);

// Quantized KV cache: scores[h][p] = dot of key row (h, p) of the cache with
// the Q8_0-quantized query q[h], for p < n_pos.
// Test switch of the scores kernel's timeout path (see gq_debug_kv_timeout).
cudaError_t kv_debug_timeout(int on);
cudaError_t launch_kv_scores(gq_type t, const void *cache, const float *q, float *scores, int64_t n_heads,
                             int64_t head_dim, int64_t capacity, int64_t n_pos, const LaunchCtx &ctx);

// dp4a GEMV family.  sums != nullptr selects the block-sum diagnostic output
// instead of y.  fused_f32: `act` is fp32 activations quantized inside the
// kernel (cols % 256 == 0 required); otherwise `act` holds quantized blocks.
// w_static: W may be fetched before the dependency wait on the previous
// kernel in the stream.
cudaError_t launch_gemv(gq_type wtype, const void *W, const void *act, float *y, int32_t *sums,
                        int64_t rows, int64_t cols, int64_t batch, bool fused_f32, bool w_static,
                        const LaunchCtx &ctx);
// True when one activation vector of `cols` fits the GEMV's shared memory.
bool gemv_fits(gq_type wtype, int64_t cols);

// Q6_K weights (gq_q6k.cu): codecs, and the Q6_K x Q8_K GEMV (any batch,
// one pass over W per group of up to eight activation vectors; sums != nullptr selects the int32
// block sums, one per 256-element block, instead of y; fused_f32 and
// w_static as for launch_gemv: with fused_f32 xq holds fp32 activations,
// quantized to Q8_K in the CTA, and the activation vector must fit the
// streaming kernel's shared memory, which gemv_q6k_fused_fits tells).
cudaError_t launch_quantize_q6k(const float *src, void *dst, int64_t n, const LaunchCtx &ctx);
cudaError_t launch_dequantize_q6k(const void *src, float *dst, int64_t n, const LaunchCtx &ctx);
cudaError_t launch_gemv_q6k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t cols,
                            int64_t batch, bool fused_f32, bool w_static, const LaunchCtx &ctx);
bool gemv_q6k_fused_fits(int64_t cols);

// Q5_K x Q8_K GEMV (gq_q5k.cu; the Q5_K codecs are in gq_codec.cu): any
// batch, one pass over W per group of up to eight vectors; sums != nullptr selects the
// int32 sums S1, S2 per 256-element block instead of y; fused_f32 and
// w_static as for launch_gemv_q6k.
cudaError_t launch_gemv_q5k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows, int64_t cols,
                            int64_t batch, bool fused_f32, bool w_static, const LaunchCtx &ctx);
bool gemv_q5k_fused_fits(int64_t cols);

// tcgen05 tensor-core family (Q4_K x Q8_K): a pack kernel writes the
// activation operand into `workspace`, then the MMA kernel runs.
cudaError_t launch_mma_q4k(const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                           int64_t cols, int64_t batch, void *workspace, const LaunchCtx &ctx);
bool mma_supported(int64_t rows, int64_t cols, int64_t batch);
size_t mma_workspace_bytes(int64_t rows, int64_t cols, int64_t batch);
// tcgen05 tensor-core family for Q4_0 / Q8_0 weights x Q8_0 activations
// (gq_mma_q0.cu): no workspace, cols a multiple of 256.
cudaError_t launch_mma_q0(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                          int64_t cols, int64_t batch, const LaunchCtx &ctx);
bool mma_q0_supported(int64_t rows, int64_t cols, int64_t batch);
// Warp-level tensor-core kernel for Q4_K / Q5_K x Q8_K at small batches
// (gq_skinny.cu): batch <= 64, cols a multiple of 256, no workspace;
// w_static as for launch_gemv (the first weight tiles are requested before
// the dependency wait).
// Q4_K or Q5_K weights (wtype); at most skinny_max_batch(wtype) vectors per
// launch (64, or 32 for Q5_K).
cudaError_t launch_skinny_q4k(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                              int64_t cols, int64_t batch, bool w_static, const LaunchCtx &ctx);
int skinny_max_batch(gq_type wtype);
bool skinny_supported(int64_t rows, int64_t cols, int64_t batch);
// The same for Q4_0 / Q8_0 weights x Q8_0 activations (gq_skinny_q0.cu):
// batch <= 64, cols a multiple of 256, no workspace, int32 sums one per
// 32-element block.
cudaError_t launch_skinny_q0(gq_type wtype, const void *W, const void *xq, float *y, int32_t *sums, int64_t rows,
                             int64_t cols, int64_t batch, bool w_static, const LaunchCtx &ctx);
bool skinny_q0_supported(int64_t rows, int64_t cols, int64_t batch);
// The library's static scratch (no allocation): its size, and its device
// address on `device` (looked up on the first call for that device, which
// must be the current device).
size_t mma_noalloc_scratch_bytes();
cudaError_t mma_noalloc_scratch(int device, void **ptr);

}  // namespace gq
