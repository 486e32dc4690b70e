// gq_api.cu -- the C ABI declared in include/gq.h: argument validation,
// per-device launch context, kernel-family dispatch and error reporting.
// Nothing here allocates device memory ("llama.cpp：一个人、一个周末…",
// 内存管理：推理时零分配: all buffers exist before the inference loop).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// Device status word (bit mask of the kernel families whose bounded waits
// ran out).  One per device: module-scope device memory, no allocation.
__device__ uint32_t g_status_word;

constexpr int MAX_DEVICES = 64;

struct DevInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t *status = nullptr;
};

DevInfo g_dev[MAX_DEVICES];
thread_local int t_last_cuda_error = 0;

gq_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return GQ_ERR_CUDA;
}

gq_status make_ctx(gq_stream_t stream, LaunchCtx *ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= MAX_DEVICES) return cuda_fail(cudaErrorInvalidDevice);
    DevInfo &d = g_dev[dev];
    std::call_once(d.once, [&d, dev]() {
        cudaError_t r = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess)
            r = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (r == cudaSuccess)
            r = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (r == cudaSuccess && d.cc_major == 10 && d.cc_minor == 3)
            r = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status_word);
        d.err = r;
    });
    if (d.err != cudaSuccess) return cuda_fail(d.err);
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return GQ_ERR_ARCH;
    ctx->stream = reinterpret_cast<cudaStream_t>(stream);
    ctx->device = dev;
    ctx->num_sms = d.num_sms;
    ctx->status = d.status;
    return GQ_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_type(int t) { return t >= GQ_Q4_0 && t <= GQ_Q5_K; }

int64_t block_elems(int t) {
    switch (t) {
    case GQ_Q4_0: case GQ_Q8_0: return 32;
    case GQ_Q4_K: case GQ_Q8_K: case GQ_Q6_K: case GQ_Q5_K: return 256;
    }
    return -1;
}

int64_t block_bytes(int t) {
    switch (t) {
    case GQ_Q4_0: return Q4_0_BYTES;
    case GQ_Q8_0: return Q8_0_BYTES;
    case GQ_Q4_K: return Q4_K_BYTES;
    case GQ_Q8_K: return Q8_K_BYTES;
    case GQ_Q6_K: return Q6_K_BYTES;
    case GQ_Q5_K: return Q5_K_BYTES;
    }
    return -1;
}

// Largest element count accepted by the codecs (keeps every byte offset
// well inside int64 and the grid-stride loops exact).
constexpr int64_t MAX_ELEMS = (int64_t)1 << 46;
// Largest reduction length of the product; bounded by the shared memory the
// GEMV kernels stage one activation vector in.
constexpr int64_t MAX_COLS = 131072;
constexpr int64_t MAX_DIM = 0x7fffffff;

gq_status check_codec(gq_type type, const void *x, const void *q, int64_t n, bool quant) {
    if (!valid_type(type)) return GQ_ERR_TYPE;
    if (n < 0 || n > MAX_ELEMS || n % block_elems(type) != 0) return GQ_ERR_SHAPE;
    if (n == 0) return GQ_OK;
    if (!x || !q) return GQ_ERR_NULL;
    if (!aligned(x, 4)) return GQ_ERR_ALIGN;
    const uintptr_t qa = (type == GQ_Q4_K || type == GQ_Q5_K || type == GQ_Q8_K) ? 4 : 2;
    if (!aligned(q, qa)) return GQ_ERR_ALIGN;
    (void)quant;
    return GQ_OK;
}

gq_status check_matmul(gq_type wtype, const void *W, const void *xq, const void *out,
                       int64_t rows, int64_t cols, int64_t batch, uintptr_t out_align) {
    if (wtype != GQ_Q4_0 && wtype != GQ_Q8_0 && wtype != GQ_Q4_K && wtype != GQ_Q6_K && wtype != GQ_Q5_K)
        return GQ_ERR_TYPE;
    if (rows < 0 || cols < 0 || batch < 0) return GQ_ERR_SHAPE;
    if (cols % block_elems(wtype) != 0) return GQ_ERR_SHAPE;
    if (rows > MAX_DIM || batch > MAX_DIM || cols > MAX_COLS) return GQ_ERR_SHAPE;
    const int64_t nblk = cols / block_elems(wtype);
    if (rows * nblk > ((int64_t)1 << 40) || batch * nblk > MAX_DIM || batch * rows > ((int64_t)1 << 40))
        return GQ_ERR_SHAPE;
    if (rows == 0 || cols == 0 || batch == 0) return GQ_OK;
    if (!W || !xq || !out) return GQ_ERR_NULL;
    if (!aligned(W, 16) || !aligned(xq, 16) || !aligned(out, out_align)) return GQ_ERR_ALIGN;
    return GQ_OK;
}

// GQ_TC_MIN_BATCH from the environment (read once), 0 when unset or invalid.
int64_t tc_min_batch_env() {
    static int64_t v = []() -> int64_t {
        const char *s = std::getenv("GQ_TC_MIN_BATCH");
        if (s && *s) {
            char *end = nullptr;
            long long x = std::strtoll(s, &end, 10);
            if (end && *end == '\0' && x > 0) return (int64_t)x;
        }
        return 0;
    }();
    return v;
}

int64_t tc_min_batch_value() { return tc_min_batch_env() ? tc_min_batch_env() : 16; }

// GQ_PATH_AUTO's choice of the tensor-core kernel for Q4_K.  Measured on
// 14336 x 4096: the tensor-core product takes about the same time at any
// batch up to 64 (its row tiles run side by side), while the GEMV grows with
// every vector, so the tensor path wins from batch 9 on matrices of 14336
// rows or more and from batch 16 on the rest.  GQ_TC_MIN_BATCH replaces the
// rule by a plain threshold.
bool tc_auto(int64_t rows, int64_t batch) {
    if (tc_min_batch_env()) return batch >= tc_min_batch_env();
    return batch >= 16 || (batch >= 9 && rows >= 14336);
}

// GQ_PATH_AUTO's choice of the warp-level tensor-core kernel for Q4_K
// (gq_skinny.cu).  Measured on 14336 x 4096 (150 CTAs of 96 rows): 12.1 us
// at batch 4 against the GEMV's 14.0 (the GEMV wins below: 11.7 us at batch
// 3), 12.5..15.7 us at 8..16 and 22 us at 32 against the tcgen05 kernel's
// 25.3..26.2, 39 us at 64 against its 30 and the GEMV's 173.  On 4096 x 4096
// (43 CTAs): 14.2 / 20.7 us at batch 16 / 32 against the GEMV's 19.6 / 38.1
// and the tcgen05 kernel's 24.4 / 24.9 (the GEMV wins at 8: 10.2 vs 11.3).
// So: from batch 4 on matrices of 8192 rows or more and from 16 on 2048 or
// more, up to 32; larger batches take the tcgen05 kernel (with or without a
// workspace, tc_auto / tc_nows_auto).  Not taken when GQ_TC_MIN_BATCH sets a
// plain threshold.
bool skinny_auto(int64_t rows, int64_t batch) {
    if (tc_min_batch_env() || rows < 2048) return false;
    return batch >= (rows >= 8192 ? 4 : 16) && batch <= 32;
}

// The warp-level kernel for Q4_0 / Q8_0 weights (gq_skinny_q0.cu).
// Measured on 14336 x 4096 (Q4_0 / Q8_0): 13.6 / 16.9 us at batch 2 against
// the GEMV's 15.5 / 18.1 (the GEMV wins at batch 1: 11.0 / 14.0), 18.8 /
// 22.1, 30.7 / 34.5, 56.4 / 59.5 us at batch 16, 32, 64 against the tcgen05
// kernel's 53-61.  On 4096 x 4096: 12.7 / 14.2 us at batch 8 against the
// GEMV's 25.8 / 17.0 (the GEMV wins at 4 for Q8_0: 10.4 vs 13.4), 55.4 /
// 57.9 at 64 against the tcgen05 kernel's 59.1 / 59.7.  So: batch 2..64 on
// matrices of 8192 rows or more, 8..64 on 2048 or more; beyond 64 (two or
// more chunks) the tcgen05 kernel.  Not taken when GQ_TC_MIN_BATCH sets a
// plain threshold.
bool skinny_auto_q0(int64_t rows, int64_t batch) {
    if (tc_min_batch_env() || rows < 2048) return false;
    return batch >= (rows >= 8192 ? 2 : 8) && batch <= 64;
}

// Q4_K without a workspace: the tcgen05 kernel's variant that packs the
// activations in the CTA (tiles of 64 columns) against the warp-level
// kernel.  Measured on 14336 x 4096: 33.5 vs 37.2 us at batch 48, 34.7 vs
// 39.5 at 64, 66.5 vs 78.2 at 128 (two chunks), 100.3 vs 156.6 at 256; the
// 28672 x 8192 x 512 prefill 0.76 vs 1.29 ms; at batch 32 (32-column
// tiles) 26.1 vs 22.1.  So: beyond batch 32 on matrices of 2048 rows or
// more, as with a workspace.
bool tc_nows_auto(int64_t rows, int64_t batch) {
    return !tc_min_batch_env() && rows >= 2048 && batch > 32;
}

// The warp-level kernel for Q5_K weights (gq_skinny.cu; Q5_K has no
// tcgen05 kernel).  Measured on 14336 x 4096: 15.4 us at batch 4 against the
// multi-vector GEMV's 16.2 (the GEMV wins below: 11.7 us at batch 2), 18.5 /
// 26.1 / 51.5 us at batch 16 / 32 / 64 against 49.3 / 96.8 / 190.9; on 4096
// x 4096: 16.8 us at batch 16 against 19.6 (the GEMV wins at 8: 10.6 vs
// 13.9).  So: from batch 4 on matrices of 8192 rows or more, from 16 on 2048
// or more, in 32-column chunks at any larger batch.
bool skinny_auto_q5k(int64_t rows, int64_t batch) {
    if (tc_min_batch_env() || rows < 2048) return false;
    return batch >= (rows >= 8192 ? 4 : 16);
}

// The same choice for Q4_0 / Q8_0 weights (gq_mma_q0.cu).
bool tc_auto_q0(int64_t rows, int64_t batch) {
    (void)rows;
    if (tc_min_batch_env()) return batch >= tc_min_batch_env();
    return batch >= 16;
}

// The family GQ_PATH_AUTO takes for a product of valid, non-empty sizes with
// quantized activations; tc_ready: a workspace large enough (and aligned)
// for the Q4_K tcgen05 kernel is passed.  Host-only arithmetic on the sizes.
gq_path auto_family(gq_type wtype, int64_t rows, int64_t cols, int64_t batch, bool tc_ready) {
    const bool q0 = wtype == GQ_Q4_0 || wtype == GQ_Q8_0;
    if (q0) {
        if (skinny_q0_supported(rows, cols, std::min<int64_t>(batch, 64)) && skinny_auto_q0(rows, batch))
            return GQ_PATH_SKINNY;
        if (tc_auto_q0(rows, batch) && mma_q0_supported(rows, cols, batch)) return GQ_PATH_MMA;
    } else if (wtype == GQ_Q4_K) {
        // without a workspace, large batches take the tcgen05 kernel that
        // packs its activations itself
        const bool tc_nows = !tc_ready && mma_supported(rows, cols, batch) && tc_nows_auto(rows, batch);
        if (tc_nows) return GQ_PATH_MMA;
        if (skinny_supported(rows, cols, std::min<int64_t>(batch, 64)) && skinny_auto(rows, batch))
            return GQ_PATH_SKINNY;
        if (tc_ready && tc_auto(rows, batch)) return GQ_PATH_MMA;
    } else if (wtype == GQ_Q5_K) {
        if (skinny_supported(rows, cols, std::min<int64_t>(batch, 32)) && skinny_auto_q5k(rows, batch))
            return GQ_PATH_SKINNY;
    }
    return GQ_PATH_GEMV;
}

// One product call.  act is xq (quantized blocks) or, with fused_f32, fp32
// activations; exactly one of y / sums is non-null.
gq_status run_matmul(gq_type wtype, const void *W, const void *act, float *y, int32_t *sums,
                     int64_t rows, int64_t cols, int64_t batch, gq_path path, unsigned flags,
                     bool fused_f32, void *ws, size_t ws_bytes, gq_stream_t stream) {
    if (path != GQ_PATH_AUTO && path != GQ_PATH_GEMV && path != GQ_PATH_MMA && path != GQ_PATH_SKINNY)
        return GQ_ERR_TYPE;
    if (flags & ~(unsigned)GQ_FLAG_W_STATIC) return GQ_ERR_TYPE;
    gq_status st = sums ? check_matmul(wtype, W, act, sums, rows, cols, batch, 4)
                        : check_matmul(wtype, W, act, y, rows, cols, batch, 4);
    if (st != GQ_OK) return st;
    const bool kstream = wtype == GQ_Q6_K || wtype == GQ_Q5_K;  // weight types with a GEMV of their own
    if (fused_f32) {
        if (path == GQ_PATH_MMA || path == GQ_PATH_SKINNY) return GQ_ERR_TYPE;
        if (cols % 256 != 0) return GQ_ERR_SHAPE;
        // Q5_K / Q6_K quantize the activations into the streaming kernel's
        // shared memory; there is no fused form of their long-vector kernel
        if (wtype == GQ_Q6_K && !gemv_q6k_fused_fits(cols)) return GQ_ERR_SHAPE;
        if (wtype == GQ_Q5_K && !gemv_q5k_fused_fits(cols)) return GQ_ERR_SHAPE;
    }
    // Q4_0 / Q8_0 weights have a tensor-core kernel of their own that needs
    // no workspace (gq_mma_q0.cu); Q4_K's packs its activations into one.
    const bool q0 = wtype == GQ_Q4_0 || wtype == GQ_Q8_0;
    if (path == GQ_PATH_MMA) {
        if (!q0 && wtype != GQ_Q4_K) return GQ_ERR_TYPE;
        if (rows == 0 || cols == 0 || batch == 0) return GQ_OK;
        if (q0) {
            if (!mma_q0_supported(rows, cols, batch)) return GQ_ERR_SHAPE;
        } else {
            if (!mma_supported(rows, cols, batch)) return GQ_ERR_SHAPE;
            // without a workspace the kernel packs the activations itself
            if (ws && ws_bytes < mma_workspace_bytes(rows, cols, batch)) return GQ_ERR_SHAPE;
            if (ws && !aligned(ws, 16)) return GQ_ERR_ALIGN;
        }
    }
    if (path == GQ_PATH_SKINNY) {
        if (!q0 && wtype != GQ_Q4_K && wtype != GQ_Q5_K) return GQ_ERR_TYPE;
        if (rows == 0 || cols == 0 || batch == 0) return GQ_OK;
        if (q0 ? !skinny_q0_supported(rows, cols, std::min<int64_t>(batch, 64))
               : !skinny_supported(rows, cols, std::min<int64_t>(batch, 64)))
            return GQ_ERR_SHAPE;
    }
    if (rows == 0 || cols == 0 || batch == 0) return GQ_OK;
    if (path == GQ_PATH_AUTO && !fused_f32) {
        const bool tc_ready = wtype == GQ_Q4_K && mma_supported(rows, cols, batch) && ws && aligned(ws, 16) &&
                              ws_bytes >= mma_workspace_bytes(rows, cols, batch);
        path = auto_family(wtype, rows, cols, batch, tc_ready);
        if (path == GQ_PATH_MMA && wtype == GQ_Q4_K && !tc_ready) ws = nullptr;  // the variant without one
    }
    const bool use_mma = path == GQ_PATH_MMA;
    const bool use_skinny = path == GQ_PATH_SKINNY;
    if (!use_mma && !use_skinny && !kstream && !gemv_fits(wtype, cols)) return GQ_ERR_SHAPE;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    if (use_skinny) {
        // chunks of up to 64 activation vectors (32 for Q5_K), one launch each
        // (y, sums and xq advance by whole vectors)
        const int64_t chunk = q0 ? 64 : skinny_max_batch(wtype);
        const bool ws_static = (flags & GQ_FLAG_W_STATIC) != 0;
        const int64_t nblk = cols / block_elems(wtype);          // weight blocks per row
        const int64_t xbytes = q0 ? cols / 32 * Q8_0_BYTES : cols / 256 * Q8_K_BYTES;  // one activation vector
        const int64_t per_row_sums = q0 ? nblk : nblk * 2;       // int32 sums per (vector, row)
        for (int64_t b0 = 0; b0 < batch; b0 += chunk) {
            const int64_t nb = std::min<int64_t>(chunk, batch - b0);
            const uint8_t *xb = static_cast<const uint8_t *>(act) + b0 * xbytes;
            float *yb = y ? y + b0 * rows : nullptr;
            int32_t *sb = sums ? sums + b0 * rows * per_row_sums : nullptr;
            cudaError_t e = q0 ? launch_skinny_q0(wtype, W, xb, yb, sb, rows, cols, nb, ws_static, ctx)
                               : launch_skinny_q4k(wtype, W, xb, yb, sb, rows, cols, nb, ws_static, ctx);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        return GQ_OK;
    }
    cudaError_t e = use_mma && q0      ? launch_mma_q0(wtype, W, act, y, sums, rows, cols, batch, ctx)
                    : use_mma          ? launch_mma_q4k(W, act, y, sums, rows, cols, batch, ws, ctx)
                    : wtype == GQ_Q6_K ? launch_gemv_q6k(W, act, y, sums, rows, cols, batch, fused_f32,
                                                         (flags & GQ_FLAG_W_STATIC) != 0, ctx)
                    : wtype == GQ_Q5_K ? launch_gemv_q5k(W, act, y, sums, rows, cols, batch, fused_f32,
                                                         (flags & GQ_FLAG_W_STATIC) != 0, ctx)
                                       : launch_gemv(wtype, W, act, y, sums, rows, cols, batch, fused_f32,
                                                     (flags & GQ_FLAG_W_STATIC) != 0, ctx);
    if (e != cudaSuccess) return cuda_fail(e);
    return GQ_OK;
}

}  // namespace
}  // namespace gq

using namespace gq;

extern "C" {

int64_t gq_block_elems(gq_type type) { return block_elems(type); }
int64_t gq_block_bytes(gq_type type) { return block_bytes(type); }

const char *gq_status_string(gq_status status) {
    switch (status) {
    case GQ_OK: return "ok";
    case GQ_ERR_NULL: return "null pointer";
    case GQ_ERR_TYPE: return "unsupported type, pairing or path";
    case GQ_ERR_SHAPE: return "invalid size (negative, not a block multiple, or too large)";
    case GQ_ERR_ALIGN: return "misaligned pointer";
    case GQ_ERR_CUDA: return "CUDA error (see gq_last_cuda_error)";
    case GQ_ERR_TIMEOUT: return "a bounded device wait timed out";
    case GQ_ERR_ARCH: return "current device is not an sm_103 GPU";
    }
    return "unknown status";
}

int gq_last_cuda_error(void) { return t_last_cuda_error; }

gq_status gq_quantize_rows_async(gq_type type, const float *src, void *dst, int64_t n,
                                 gq_stream_t stream) {
    gq_status st = check_codec(type, src, dst, n, true);
    if (st != GQ_OK || n == 0) return st;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = type == GQ_Q6_K ? launch_quantize_q6k(src, dst, n, ctx) : launch_quantize(type, src, dst, n, ctx);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

gq_status gq_quantize_rows(gq_type type, const float *src, void *dst, int64_t n) {
    return gq_quantize_rows_async(type, src, dst, n, nullptr);
}

gq_status gq_quantize_rows_ex(gq_type type, const float *src, void *dst, int64_t n, unsigned flags,
                              gq_stream_t stream) {
    if (flags & ~(unsigned)GQ_QUANT_ERRMIN) return GQ_ERR_TYPE;
    if (!(flags & GQ_QUANT_ERRMIN)) return gq_quantize_rows_async(type, src, dst, n, stream);
    if (type != GQ_Q4_K && type != GQ_Q5_K) return GQ_ERR_TYPE;
    gq_status st = check_codec(type, src, dst, n, true);
    if (st != GQ_OK || n == 0) return st;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = launch_quantize_k_errmin(type, src, dst, n, ctx);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

gq_status gq_dequantize_rows_async(gq_type type, const void *src, float *dst, int64_t n,
                                   gq_stream_t stream) {
    gq_status st = check_codec(type, dst, src, n, false);
    if (st != GQ_OK || n == 0) return st;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = type == GQ_Q6_K ? launch_dequantize_q6k(src, dst, n, ctx)
                                    : launch_dequantize(type, src, dst, n, ctx);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

gq_status gq_dequantize_rows(gq_type type, const void *src, float *dst, int64_t n) {
    return gq_dequantize_rows_async(type, src, dst, n, nullptr);
}

gq_status gq_matmul(gq_type wtype, const void *W, const void *xq, float *y, int64_t rows,
                    int64_t cols, int64_t batch, gq_stream_t stream) {
    return run_matmul(wtype, W, xq, y, nullptr, rows, cols, batch, GQ_PATH_AUTO, 0, false, nullptr, 0, stream);
}

gq_status gq_matmul_path(gq_type wtype, const void *W, const void *xq, float *y, int64_t rows,
                         int64_t cols, int64_t batch, gq_path path, gq_stream_t stream) {
    return run_matmul(wtype, W, xq, y, nullptr, rows, cols, batch, path, 0, false, nullptr, 0, stream);
}

gq_status gq_matmul_ex(gq_type wtype, const void *W, const void *xq, float *y, int64_t rows,
                       int64_t cols, int64_t batch, gq_path path, unsigned flags,
                       gq_stream_t stream) {
    return run_matmul(wtype, W, xq, y, nullptr, rows, cols, batch, path, flags, false, nullptr, 0, stream);
}

gq_status gq_matmul_f32(gq_type wtype, const void *W, const float *x, float *y, int64_t rows,
                        int64_t cols, int64_t batch, unsigned flags, gq_stream_t stream) {
    if (x && ((reinterpret_cast<uintptr_t>(x) & 15) != 0)) return GQ_ERR_ALIGN;
    return run_matmul(wtype, W, x, y, nullptr, rows, cols, batch, GQ_PATH_GEMV, flags, true, nullptr, 0, stream);
}

gq_status gq_block_sums(gq_type wtype, const void *W, const void *xq, int32_t *sums,
                        int64_t rows, int64_t cols, int64_t batch, gq_path path,
                        gq_stream_t stream) {
    if (!sums && rows > 0 && cols > 0 && batch > 0) return GQ_ERR_NULL;
    return run_matmul(wtype, W, xq, nullptr, sums, rows, cols, batch, path, 0, false, nullptr, 0, stream);
}

gq_status gq_block_sums_f32(gq_type wtype, const void *W, const float *x, int32_t *sums,
                            int64_t rows, int64_t cols, int64_t batch, gq_stream_t stream) {
    if (!sums && rows > 0 && cols > 0 && batch > 0) return GQ_ERR_NULL;
    if (x && ((reinterpret_cast<uintptr_t>(x) & 15) != 0)) return GQ_ERR_ALIGN;
    return run_matmul(wtype, W, x, nullptr, sums, rows, cols, batch, GQ_PATH_GEMV, 0, true, nullptr, 0, stream);
}

gq_status gq_matmul_ws(gq_type wtype, const void *W, const void *xq, float *y, int64_t rows,
                       int64_t cols, int64_t batch, gq_path path, unsigned flags, void *workspace,
                       size_t workspace_bytes, gq_stream_t stream) {
    return run_matmul(wtype, W, xq, y, nullptr, rows, cols, batch, path, flags, false, workspace,
                      workspace_bytes, stream);
}

gq_status gq_block_sums_ws(gq_type wtype, const void *W, const void *xq, int32_t *sums,
                           int64_t rows, int64_t cols, int64_t batch, gq_path path,
                           void *workspace, size_t workspace_bytes, gq_stream_t stream) {
    if (!sums && rows > 0 && cols > 0 && batch > 0) return GQ_ERR_NULL;
    return run_matmul(wtype, W, xq, nullptr, sums, rows, cols, batch, path, 0, false, workspace,
                      workspace_bytes, stream);
}

size_t gq_matmul_workspace_bytes(gq_type wtype, int64_t rows, int64_t cols, int64_t batch) {
    if (wtype != GQ_Q4_K || rows < 1 || batch < 1 || cols > MAX_COLS || !mma_supported(rows, cols, batch))
        return 0;
    return mma_workspace_bytes(rows, cols, batch);
}

gq_status gq_matmul_noalloc(gq_type wtype, const void *W, const void *xq, float *y, int64_t rows,
                            int64_t cols, int64_t batch, gq_stream_t stream) {
    if (wtype != GQ_Q4_K) return GQ_ERR_TYPE;
    gq_status st = check_matmul(wtype, W, xq, y, rows, cols, batch, 4);
    if (st != GQ_OK || rows == 0 || cols == 0 || batch == 0) return st;
    if (!mma_supported(rows, cols, batch)) return GQ_ERR_SHAPE;
    const size_t need = mma_workspace_bytes(rows, cols, batch);
    if (need > mma_noalloc_scratch_bytes()) return GQ_ERR_SHAPE;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    void *scratch = nullptr;
    cudaError_t e = mma_noalloc_scratch(ctx.device, &scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    return run_matmul(wtype, W, xq, y, nullptr, rows, cols, batch, GQ_PATH_MMA, 0, false, scratch,
                      mma_noalloc_scratch_bytes(), stream);
}

int64_t gq_tc_min_batch(void) { return tc_min_batch_value(); }

gq_status gq_auto_path(gq_type wtype, int64_t rows, int64_t cols, int64_t batch, int with_workspace,
                       gq_path *path) {
    if (!path) return GQ_ERR_NULL;
    if (wtype != GQ_Q4_0 && wtype != GQ_Q8_0 && wtype != GQ_Q4_K && wtype != GQ_Q5_K && wtype != GQ_Q6_K)
        return GQ_ERR_TYPE;
    if (rows < 0 || cols < 0 || batch < 0 || cols % block_elems(wtype) != 0) return GQ_ERR_SHAPE;
    if (rows == 0 || cols == 0 || batch == 0) {
        *path = GQ_PATH_GEMV;
        return GQ_OK;
    }
    const bool tc_ready = with_workspace != 0 && wtype == GQ_Q4_K && mma_supported(rows, cols, batch);
    *path = auto_family(wtype, rows, cols, batch, tc_ready);
    return GQ_OK;
}

gq_status gq_debug_kv_timeout(int on) {
    LaunchCtx ctx;
    gq_status st = make_ctx(nullptr, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = kv_debug_timeout(on);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

}  // extern "C"

namespace {
// Shape and pointer rules shared by the KV-cache calls.
gq_status check_kv(gq_type type, const void *cache, int64_t n_heads, int64_t head_dim, int64_t capacity) {
    if (type != GQ_Q8_0 && type != GQ_Q4_0) return GQ_ERR_TYPE;
    if (n_heads < 0 || n_heads > 65535 || head_dim < 32 || head_dim > 256 || head_dim % 32 != 0)
        return GQ_ERR_SHAPE;
    if (capacity < 32 || capacity % 32 != 0 || capacity > ((int64_t)1 << 30)) return GQ_ERR_SHAPE;
    if (n_heads > 0 && !cache) return GQ_ERR_NULL;
    if (!aligned(cache, 16)) return GQ_ERR_ALIGN;
    return GQ_OK;
}
}  // namespace

extern "C" {

gq_status gq_kv_append(gq_type type, const float *x, void *cache, int64_t n_heads, int64_t head_dim,
                       int64_t capacity, int64_t pos, gq_stream_t stream) {
    gq_status st = check_kv(type, cache, n_heads, head_dim, capacity);
    if (st != GQ_OK) return st;
    if (pos < 0 || pos >= capacity) return GQ_ERR_SHAPE;
    if (n_heads == 0) return GQ_OK;
    if (!x) return GQ_ERR_NULL;
    if (!aligned(x, 4)) return GQ_ERR_ALIGN;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    const int64_t nb = head_dim / 32;
    uint8_t *dst = static_cast<uint8_t *>(cache) + pos * nb * block_bytes(type);
    cudaError_t e = launch_quantize_rows_strided(type, x, dst, n_heads, nb, capacity * nb, ctx);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

gq_status gq_kv_scores(gq_type type, const void *cache, const float *q, float *scores, int64_t n_heads,
                       int64_t head_dim, int64_t capacity, int64_t n_pos, gq_stream_t stream) {
    gq_status st = check_kv(type, cache, n_heads, head_dim, capacity);
    if (st != GQ_OK) return st;
    if (n_pos < 0 || n_pos > capacity) return GQ_ERR_SHAPE;
    if (n_heads == 0 || n_pos == 0) return GQ_OK;
    if (!q || !scores) return GQ_ERR_NULL;
    if (!aligned(q, 4) || !aligned(scores, 4)) return GQ_ERR_ALIGN;
    LaunchCtx ctx;
    st = make_ctx(stream, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = launch_kv_scores(type, cache, q, scores, n_heads, head_dim, capacity, n_pos, ctx);
    return e == cudaSuccess ? GQ_OK : cuda_fail(e);
}

gq_status gq_device_status(uint32_t *word, int reset) {
    LaunchCtx ctx;
    gq_status st = make_ctx(nullptr, &ctx);
    if (st != GQ_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    uint32_t v = 0;
    e = cudaMemcpy(&v, ctx.status, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (reset && v) {
        const uint32_t zero = 0;
        e = cudaMemcpy(ctx.status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (word) *word = v;
    return v ? GQ_ERR_TIMEOUT : GQ_OK;
}

}  // extern "C"
