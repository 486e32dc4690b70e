/*
 * gq.h -- C ABI of the block-quantized GEMV/GEMM library for GB300 (sm_103a).
 *
 * The library multiplies weights stored as Q4_0 / Q8_0 / Q4_K blocks with
 * activations quantized to int8 per 32-element (Q8_0) or 256-element (Q8_K)
 * block, as per-block integer dot products scaled by the block factors and
 * summed.  The method is the one the llama.cpp pages describe:
 *   "llama.cpp 推理引擎" (runguoli.com/llm-libs/14-llama-cpp), §5.1-§5.5
 *   (symmetric / asymmetric quantization, Q4_0, Q8_0, K-quants) and §6.4
 *   (the Q4_0 vec_dot: per-block integer products scaled by the block
 *   scale); "llama.cpp：一个人、一个周末、一个改变 AI 推理格局的 C++ 文件"
 *   (tech-blog-56a.pages.dev), 第二层：量化引擎 (block quantization, the
 *   256 = 8 x 32 K-quant super-block) and 内存管理：推理时零分配 (no
 *   allocation during inference).
 *
 * Block formats (all multi-byte fields little-endian, blocks packed back to
 * back, a row of a matrix is cols / block_elems consecutive blocks and rows
 * are consecutive):
 *   Q4_0  18 B / 32 elements : fp16 d @0, 16 bytes of 4-bit codes c @2;
 *                              byte j holds element 2j (low nibble) and
 *                              2j+1 (high nibble); w = d * (c - 8).
 *   Q8_0  34 B / 32 elements : fp16 d @0, int8 q[32] @2; w = d * q.
 *   Q4_K 144 B / 256 elements: fp16 d @0, fp16 dmin @2, twelve bytes @4
 *                              holding sixteen 6-bit fields LSB-first
 *                              (fields 0..7 = sub-block scales sc_j, 8..15 =
 *                              sub-block mins m_j), 128 bytes of 4-bit codes
 *                              q @16 in the Q4_0 nibble order;
 *                              w = d * sc_j * q - dmin * m_j for element i
 *                              of sub-block j = i / 32.
 *   Q6_K 194 B / 256 elements: fp16 d @0, 128 bytes @2 holding the low
 *                              four bits of the codes c in the Q4_0 nibble
 *                              order, 64 bytes @130 holding their top two
 *                              bits (byte l: elements 4l..4l+3, element 4l+k
 *                              in bits 2k..2k+1); w = d * (c - 32).  The
 *                              6-bit K-quant of the discosf.com page ("为什么说
 *                              llama.cpp 是'裸引擎'…", §4): K blocks only, no
 *                              sub-blocks, 6-bit main quantization; the
 *                              symmetric rule and this layout are this
 *                              library's reading.
 *   Q5_K 176 B / 256 elements: bytes 0..143 as Q4_K (d, dmin, the sixteen
 *                              6-bit fields, the low four bits of the codes
 *                              q in [0, 31]), then 32 bytes @144 holding
 *                              the fifth bits: bit 2t + p of byte
 *                              144 + 4j + i is the fifth bit of element
 *                              32j + 8t + 2i + p (t, i = 0..3, p = 0..1);
 *                              w = d * sc_j * q - dmin * m_j.  The 5-bit
 *                              K-quant of the same discosf.com page (one bit
 *                              more than Q4_K); the layout is this
 *                              library's reading.
 *   Q8_K 276 B / 256 elements: fp32 d @0, int8 q[256] @4, int16 bsums[8]
 *                              @260 (bsums[j] = sum of q over sub-block j);
 *                              w = d * q.
 * Quantization rounds codes half away from zero.  Q8_0 and Q8_K use
 * d = max|x| / 127, Q4_0 uses d = max|x| / 7, Q6_K d = max|x| / 31 (fp16
 * scales rounded to nearest-even; codes clamped to [-8, 7] and [-32, 31]
 * before the offsets 8 and 32); Q4_K fits each 32-element sub-block by its min/max with fp16
 * d and dmin rounded toward +infinity (so that the ceilinged 6-bit scale and
 * min always cover the sub-block) -- see the quantize entry point below;
 * Q5_K is the same fit with 31 code steps instead of 15.
 *
 * Pairings for the product: Q4_0 and Q8_0 weights take Q8_0 activations;
 * Q4_K, Q5_K and Q6_K weights take Q8_K activations.
 *
 * General rules for every entry point:
 *   - All data pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA
 *     memory) owned by the caller.  The library never allocates or frees
 *     device memory and never copies between host and device on these calls.
 *   - Calls are asynchronous on the given stream (NULL = the legacy default
 *     stream); none of them synchronizes.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error status and launches nothing.  The
 *     library never aborts, exits or prints.
 *   - GQ_ERR_CUDA is returned when a launch fails; gq_last_cuda_error()
 *     then gives the cudaError_t value (per calling thread).
 *   - Device-side waits (on TMA transfer barriers) are bounded; a wait that
 *     runs out sets a device status word instead of hanging, and
 *     gq_device_status() reports it as GQ_ERR_TIMEOUT.
 *   - Thread safety: every entry point may be called from several host
 *     threads at once; the only shared state is a per-device attribute cache
 *     and the device status word.
 *   - The per-device cache (attributes, and the device addresses of the
 *     status word and of gq_matmul_noalloc's scratch) is filled on the first
 *     call on each device and kept for the life of the process: calling the
 *     library on a device after cudaDeviceReset() on it is unsupported.
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *gq_stream_t;

typedef enum {
    GQ_Q4_0 = 0,
    GQ_Q8_0 = 1,
    GQ_Q4_K = 2,
    GQ_Q8_K = 3,
    GQ_Q6_K = 4,
    GQ_Q5_K = 5
} gq_type;

typedef enum {
    GQ_OK = 0,
    GQ_ERR_NULL = 1,    /* a required pointer is NULL */
    GQ_ERR_TYPE = 2,    /* unknown type, or an unsupported weight/activation pairing */
    GQ_ERR_SHAPE = 3,   /* negative size, size not a block multiple, or size overflow */
    GQ_ERR_ALIGN = 4,   /* a pointer is not aligned as the call requires */
    GQ_ERR_CUDA = 5,    /* a CUDA launch or query failed (see gq_last_cuda_error) */
    GQ_ERR_TIMEOUT = 6, /* a bounded device wait ran out (reported by gq_device_status) */
    GQ_ERR_ARCH = 7     /* the current device is not an sm_103 GPU */
} gq_status;

/* Flags for gq_matmul_ex / gq_matmul_f32. */
enum {
    /* W is not written by any kernel that may still be running on the stream
     * (model weights written once at load time).  The GEMV kernels then
     * request their first weight chunks before waiting for the preceding
     * kernel in the stream to finish, overlapping the weight fetch with that
     * kernel's tail.  Without the flag every read of W happens after that
     * wait.  The Q4_0 / Q8_0 / Q4_K, Q5_K and Q6_K GEMV kernels and the
     * warp-level tensor-core kernel (GQ_PATH_SKINNY, its first two weight
     * tiles) act on it; the tcgen05 kernels read W after the wait in any
     * case. */
    GQ_FLAG_W_STATIC = 1u
};

/* Kernel family selection for gq_matmul_path / gq_block_sums. */
typedef enum {
    GQ_PATH_AUTO = 0,   /* GEMV below the tensor-core crossover batch, MMA at or above */
    GQ_PATH_GEMV = 1,   /* dp4a GEMV kernels (any batch; batch is processed in chunks) */
    GQ_PATH_MMA = 2,    /* tcgen05 tensor-core kernels (Q4_0, Q8_0, Q4_K weights) */
    GQ_PATH_SKINNY = 3  /* warp-level tensor-core kernels (mma.sync): Q4_K, Q5_K, Q4_0, Q8_0; 64 (Q5_K: 32) columns a launch */
} gq_path;

/* Elements per block: 32, 32, 256, 256, 256, 256 (Q4_0, Q8_0, Q4_K, Q8_K,
 * Q6_K, Q5_K).  -1 for an unknown type. */
int64_t gq_block_elems(gq_type type);
/* Bytes per block: 18, 34, 144, 276, 194, 176.  -1 for an unknown type. */
int64_t gq_block_bytes(gq_type type);
/* Static text for a status code (never NULL). */
const char *gq_status_string(gq_status status);
/* cudaError_t of the last GQ_ERR_CUDA returned to this host thread (0 if none). */
int gq_last_cuda_error(void);

/*
 * Quantize n fp32 values (n / block_elems(type) blocks) into packed blocks.
 *   src : device, n floats, 4-byte aligned, finite values (non-finite input
 *         gives unspecified codes; magnitudes must keep the fp16 scales in
 *         range: |x| < 65504 * 127 for Q8_0, 65504 * 7 for Q4_0, 65504 * 945
 *         for Q4_K, 65504 * 1953 for Q5_K, 65504 * 31 for Q6_K).
 *   dst : device, n / block_elems * block_bytes bytes; 4-byte aligned for
 *         Q8_K, Q4_K and Q5_K, 2-byte aligned for Q4_0 / Q8_0 / Q6_K (the product needs
 *         16-byte aligned weights, see gq_matmul).
 *   n   : element count, >= 0 and a multiple of block_elems(type).
 * Results are bit-identical to the reference definition of each format
 * ("llama.cpp 推理引擎" §5.1 symmetric rule for Q8_0 / Q4_0 / Q8_K, §5.2
 * asymmetric min/max rule per sub-block and §5.5 two-level scales for Q4_K).
 * Errors: GQ_ERR_NULL (n > 0 and a NULL pointer), GQ_ERR_TYPE, GQ_ERR_SHAPE,
 * GQ_ERR_ALIGN, GQ_ERR_CUDA.  Enqueued on the legacy default stream.
 */
gq_status gq_quantize_rows(gq_type type, const float *src, void *dst, int64_t n);
gq_status gq_quantize_rows_async(gq_type type, const float *src, void *dst, int64_t n,
                                 gq_stream_t stream);

/* Flags for gq_quantize_rows_ex. */
enum {
    /* Error-minimizing K-quant encoder (Q4_K and Q5_K only): "llama.cpp 推理
     * 引擎" §5.5 stores each sub-block's scale and min as 6-bit integers under
     * the super-block's d and dmin, and §7.1 recommends choosing them for the
     * least (importance-weighted) reconstruction error; with uniform weights
     * (no calibration data is taken) this encoder keeps the min/max fit's d
     * and dmin and, per 32-element sub-block, picks the (sc, m) within 4 of
     * the fit's pair (clipped to 0..63) whose 32 reconstructed values, codes
     * the nearest in range, have the least squared error.  The error is
     * computed in fp32 in a fixed order (each group of eight consecutive
     * elements in turn, then (g0 + g1) + (g2 + g3)); the first candidate in
     * (sc, m) ascending order strictly below the best so far wins, starting
     * from the fit's pair -- so no sub-block is reconstructed worse than by
     * the min/max fit in that measure.  Same byte format: every decoder and
     * product reads the result unchanged. */
    GQ_QUANT_ERRMIN = 1u
};

/* gq_quantize_rows_async with flags (0 = the default encoder).  Errors as
 * gq_quantize_rows, plus GQ_ERR_TYPE for an unknown flag bit or
 * GQ_QUANT_ERRMIN with a type other than Q4_K / Q5_K. */
gq_status gq_quantize_rows_ex(gq_type type, const float *src, void *dst, int64_t n, unsigned flags,
                              gq_stream_t stream);

/*
 * Reconstruct n fp32 values from packed blocks ("llama.cpp 推理引擎" §5.3
 * and §5.5 dequantization formulas, with the fp16 scale of Q8_0 and the
 * subtracted Q4_K min of this library's formats).  Each output is the exact
 * reconstruction rounded once to fp32.
 *   src : device, packed blocks (alignment as for gq_quantize_rows' dst).
 *   dst : device, n floats, 4-byte aligned.
 * Errors as for gq_quantize_rows.
 */
gq_status gq_dequantize_rows(gq_type type, const void *src, float *dst, int64_t n);
gq_status gq_dequantize_rows_async(gq_type type, const void *src, float *dst, int64_t n,
                                   gq_stream_t stream);

/*
 * y[b][r] = sum over the blocks k of row r of the scaled integer block dots
 * ("llama.cpp 推理引擎" §6.4 for the per-block dot; §5.5 for the Q4_K
 * two-level scales):
 *   Q4_0 x Q8_0 : d_w * d_x * sum_i (c_i - 8) * a_i
 *   Q8_0 x Q8_0 : d_w * d_x * sum_i w_i * a_i
 *   Q4_K x Q8_K : d_x * (d * sum_j sc_j * s_j - dmin * sum_j m_j * t_j),
 *                 s_j = sum_{i in j} q_i * a_i, t_j = bsums[j]
 *   Q5_K x Q8_K : as Q4_K x Q8_K with the 5-bit codes
 *   Q6_K x Q8_K : d_w * d_x * sum_i (c_i - 32) * a_i   (per 256-element block)
 *   wtype : GQ_Q4_0, GQ_Q8_0, GQ_Q4_K, GQ_Q5_K or GQ_Q6_K.
 *   W     : device, rows x (cols / block_elems) weight blocks, 16-byte aligned.
 *   xq    : device, batch x (cols / block_elems) activation blocks (Q8_0 for
 *           Q4_0 / Q8_0 weights, Q8_K for Q4_K / Q5_K / Q6_K), one vector after another;
 *           16-byte aligned.
 *   y     : device, float[batch][rows], 4-byte aligned; fully overwritten.
 *   rows, cols, batch : > 0 (a zero size is a no-op returning GQ_OK);
 *           cols a multiple of 256 for Q4_K / Q5_K / Q6_K and of 32 for Q4_0 / Q8_0
 *           (the fast kernels need cols % 256 == 0, and cols % 2048 == 0 up
 *           to 16384 for Q6_K; other shapes run a plain per-block kernel);
 *           Q5_K and Q6_K run one pass over W per group of up to eight
 *           activation vectors (fewer when wide vectors fill the shared
 *           memory); cols at most 131072 (and small enough for one
 *           activation vector to fit the kernels' shared memory: every cols
 *           up to that bound does).
 * The integer block sums are exact (int32); y matches the double-precision
 * sum of the same terms within 1e-4 of the sum of their magnitudes.
 * Asynchronous on `stream`; allocates nothing.
 * Dispatch (GQ_PATH_AUTO):
 *   Q4_0 / Q8_0 weights (cols % 256 == 0): the warp-level tensor-core kernel
 *     (GQ_PATH_SKINNY) at batch 2..64 on matrices of 8192 rows or more and
 *     8..64 on 2048 or more; the tcgen05 tensor-core kernel at batch >=
 *     gq_tc_min_batch() otherwise (16 unless GQ_TC_MIN_BATCH is set, which
 *     also turns the warp-level choice off); the GEMV kernels below.  Neither
 *     tensor-core kernel needs a workspace.
 *   Q4_K weights: the warp-level tensor-core kernel (GQ_PATH_SKINNY) from
 *     batch 4 on matrices of 8192 rows or more and from 16 on 2048 or more,
 *     up to batch 32; beyond 32 on such matrices the tcgen05 kernel's variant that packs
 *     its activations in the CTA (64-column tiles); the GEMV kernels
 *     otherwise.  The tcgen05 kernel with its activations repacked once into
 *     a workspace is faster still (the 28672 x 8192 x 512 prefill: 0.32 ms
 *     against 0.76): call gq_matmul_ws, or gq_matmul_noalloc to use the
 *     library's static scratch.
 *   Q5_K weights: the warp-level tensor-core kernel from batch 4 on matrices
 *     of 8192 rows or more and from 16 on 2048 or more (32-column chunks
 *     beyond 32), their GEMV kernels otherwise.
 *   Q6_K weights: their GEMV kernels.
 * The GEMV kernels take any batch, in chunks of up to eight vectors, one
 * pass over W per chunk.  gq_auto_path reports the family chosen for a shape.
 */
gq_status gq_matmul(gq_type wtype, const void *W, const void *xq, float *y,
                    int64_t rows, int64_t cols, int64_t batch, gq_stream_t stream);

/* gq_matmul with an explicit kernel family (crossover studies, tests).
 * GQ_PATH_AUTO dispatches as gq_matmul.  GQ_PATH_MMA runs the tensor-core
 * kernel of Q4_0 / Q8_0 weights (GQ_ERR_SHAPE unless cols % 256 == 0); for
 * Q4_K weights the tcgen05 kernel's variant without a workspace (tiles of at
 * most 64 columns whose idle epilogue warps pack the activation operand in
 * the CTA; the same exact sums); for Q5_K / Q6_K GQ_ERR_TYPE.  GQ_PATH_SKINNY runs the
 * warp-level tensor-core kernels of Q4_K, Q5_K, Q4_0 and Q8_0 weights
 * (mma.sync m16n8k16 on exact integer operands: sc q - 512 for Q4_K and
 * sc q - 1024 for Q5_K, whose even and odd sub-blocks accumulate apart; one
 * fresh accumulator per 32-element block for Q4_0 / Q8_0; one launch per 64
 * activation vectors, 32 for Q5_K; cols % 256 == 0, GQ_ERR_SHAPE otherwise;
 * GQ_ERR_TYPE for Q6_K and for fp32 activations). */
gq_status gq_matmul_path(gq_type wtype, const void *W, const void *xq, float *y,
                         int64_t rows, int64_t cols, int64_t batch, gq_path path,
                         gq_stream_t stream);

/*
 * gq_matmul_path with flags (GQ_FLAG_W_STATIC).  Unknown flag bits give
 * GQ_ERR_TYPE.
 */
gq_status gq_matmul_ex(gq_type wtype, const void *W, const void *xq, float *y,
                       int64_t rows, int64_t cols, int64_t batch, gq_path path,
                       unsigned flags, gq_stream_t stream);

/*
 * Bytes of workspace the tensor-core path needs for this product (0 when the
 * shape or type has no tensor-core path, and for Q4_0 / Q8_0 weights, whose
 * tensor-core kernel needs none).  The workspace holds the activation
 * operand repacked once per call as fp16 tiles (plus per-block scales, code
 * sums and the min-term operand), per column tile of tn = 32 (batch <= 32),
 * 64 (batch <= 64) or 128 columns and per super-block: ceil(batch / tn) *
 * (cols / 256) * 552 tn bytes (17664, 35328 or 70656 per unit).
 */
size_t gq_matmul_workspace_bytes(gq_type wtype, int64_t rows, int64_t cols, int64_t batch);

/*
 * The product with a caller-provided device workspace (16-byte aligned, at
 * least gq_matmul_workspace_bytes bytes, owned by the caller, contents
 * overwritten; calls that share a workspace must not overlap on the GPU).
 * GQ_PATH_AUTO for Q4_K: the warp-level kernel (GQ_PATH_SKINNY) at batch
 * 4..32 on matrices of 8192 rows or more and 16..32 on 2048 or more; else
 * the tcgen05 tensor-core kernel when batch >= gq_tc_min_batch(), or batch
 * >= 9 on matrices of 14336 rows or more (the measured crossovers), and the
 * workspace suffices; else, beyond batch 32 on matrices of 2048 rows or
 * more, the tcgen05 variant that needs no workspace; else the GEMV kernels.  Q4_0 / Q8_0
 * weights ignore the workspace and dispatch as in gq_matmul.  With
 * GQ_TC_MIN_BATCH set, batch >= that value alone decides.
 * The tensor-core path computes the same y (within the tolerance above) and
 * the same exact integer super-block sums S1 and S2 as the GEMV kernels, for
 * every input (its fp32 accumulation only ever holds integers below 2^24).
 * Errors as gq_matmul_path, plus GQ_ERR_SHAPE (workspace too small),
 * GQ_ERR_ALIGN.  A NULL workspace with GQ_PATH_MMA runs the variant without
 * one, as gq_matmul_path does.
 */
gq_status gq_matmul_ws(gq_type wtype, const void *W, const void *xq, float *y,
                       int64_t rows, int64_t cols, int64_t batch, gq_path path,
                       unsigned flags, void *workspace, size_t workspace_bytes,
                       gq_stream_t stream);

/*
 * Fused activation quantize + product: x holds fp32 activations
 * float[batch][cols] (device, 16-byte aligned); each CTA quantizes them to
 * Q8_K (Q4_K, Q5_K, Q6_K weights) or Q8_0 (Q4_0 / Q8_0 weights) in shared memory with
 * exactly the arithmetic of gq_quantize_rows, then runs the GEMV.  The result
 * equals gq_quantize_rows followed by gq_matmul_path(..., GQ_PATH_GEMV), bit
 * for bit, with one launch instead of two and no quantized activation buffer
 * ("llama.cpp：一个人、一个周末…", 第一层：GGML 张量库: operators fused over
 * the computation graph).  GEMV kernels only (any batch); cols must be a
 * multiple of 256 (GQ_ERR_SHAPE otherwise).  Q5_K and Q6_K weights: the
 * quantized vector shares shared memory with the streaming kernel's weight
 * ring, so cols is at most 18944 (Q5_K) or a multiple of 2048 up to 16384
 * (Q6_K: whole rows of 16-byte multiples), GQ_ERR_SHAPE otherwise.  Other
 * arguments as gq_matmul.
 */
gq_status gq_matmul_f32(gq_type wtype, const void *W, const float *x, float *y,
                        int64_t rows, int64_t cols, int64_t batch, unsigned flags,
                        gq_stream_t stream);

/*
 * Diagnostic: the integer block sums of the product, as computed by the
 * chosen kernel family, without the float scaling.
 *   sums : device, int32, 4-byte aligned, laid out [batch][rows][nblk][c] with
 *          nblk = cols / block_elems(wtype) and c = 1 (Q4_0, Q8_0: the block
 *          dot; Q6_K: sum_i (c_i - 32) * a_i) or c = 2 (Q4_K, Q5_K:
 *          S1 = sum_j sc_j * s_j, S2 = sum_j m_j * t_j).
 * Other arguments and errors as gq_matmul_path.
 */
gq_status gq_block_sums(gq_type wtype, const void *W, const void *xq, int32_t *sums,
                        int64_t rows, int64_t cols, int64_t batch, gq_path path,
                        gq_stream_t stream);

/* gq_block_sums with a workspace (required for GQ_PATH_MMA with Q4_K weights). */
gq_status gq_block_sums_ws(gq_type wtype, const void *W, const void *xq, int32_t *sums,
                           int64_t rows, int64_t cols, int64_t batch, gq_path path,
                           void *workspace, size_t workspace_bytes, gq_stream_t stream);

/* gq_block_sums for the fused path (fp32 activations, as gq_matmul_f32). */
gq_status gq_block_sums_f32(gq_type wtype, const void *W, const float *x, int32_t *sums,
                            int64_t rows, int64_t cols, int64_t batch, gq_stream_t stream);

/*
 * The tensor-core product for callers that cannot allocate device memory.
 * The pages describe no such call; it exists for users of this library who
 * must not call cudaMalloc themselves: hosts that own the GPU's memory pool
 * and forbid other allocators, services that plan every byte at start-up and
 * may not allocate on the request path, and callers for whom cudaMalloc's
 * implicit device synchronisation would stall a latency-sensitive pipeline.
 * The call is gq_matmul_ws(wtype, W, xq, y, rows, cols, batch, GQ_PATH_MMA,
 * 0, workspace, ...) except that the workspace is a fixed 16 MiB scratch
 * array inside the library (module-scope device memory that every GPU
 * loading the library holds until the process exits).  Nothing is
 * allocated or freed.
 *   - wtype must be GQ_Q4_K (GQ_ERR_TYPE otherwise); other arguments,
 *     alignment and errors as gq_matmul.
 *   - A product whose workspace (gq_matmul_workspace_bytes) exceeds
 *     16 MiB = 16777216 bytes is rejected with GQ_ERR_SHAPE before anything
 *     is launched; e.g. 8192 columns allow batches up to 896, 4096 columns
 *     up to 1792.
 *   - The first call on a device looks up the scratch's device address with
 *     that device current (cudaGetSymbolAddress); make that first call
 *     before any stream capture on the device.
 *   - Every call shares the one scratch array, and it keeps the previous
 *     call's contents: each call rewrites every scratch byte it reads, so no
 *     clearing is needed, but calls that overlap on the GPU (different
 *     streams, or different host threads) race on it and give wrong results.
 *     gq_matmul_path(..., GQ_PATH_MMA) runs the same tensor-core kernel
 *     with no scratch at all (its variant that packs the activations in the
 *     CTA: slower at large batches, e.g. 0.76 against 0.32 ms for the
 *     28672 x 8192 x 512 prefill) and is safe to overlap.
 */
gq_status gq_matmul_noalloc(gq_type wtype, const void *W, const void *xq, float *y,
                            int64_t rows, int64_t cols, int64_t batch, gq_stream_t stream);

/*
 * Quantized KV cache ("llama.cpp 推理引擎" §3.7.3, KV Cache 量化: keys and
 * values cached as Q8_0 or Q4_0 blocks; §6.4 for the block dot).
 *
 * Cache layout (device, owned by the caller, 16-byte aligned):
 * [n_heads][capacity][head_dim / 32] blocks of `type`, so row (h, p) -- the
 * key (or value) of head h at position p -- is head_dim / 32 consecutive
 * blocks and the rows of a head are consecutive.  Size:
 * n_heads * capacity * head_dim / 32 * gq_block_bytes(type) bytes.
 *   type     : GQ_Q8_0 or GQ_Q4_0 (GQ_ERR_TYPE otherwise).
 *   head_dim : a multiple of 32, 32 .. 256.
 *   capacity : positions per head, a multiple of 32 (the scores kernel reads
 *              whole groups of 32 rows), at most 2^30.
 *   n_heads  : 0 .. 65535 (0 is a no-op returning GQ_OK).
 * Asynchronous on `stream`; the cache bytes of other rows are never written.
 */

/* Quantizes x = float[n_heads][head_dim] (device, 4-byte aligned) into row
 * (h, pos) of every head, with exactly the arithmetic of gq_quantize_rows:
 * the bytes equal gq_quantize_rows of x[h] written at that row.  pos in
 * [0, capacity) (GQ_ERR_SHAPE otherwise). */
gq_status gq_kv_append(gq_type type, const float *x, void *cache, int64_t n_heads, int64_t head_dim,
                       int64_t capacity, int64_t pos, gq_stream_t stream);

/* Attention scores against the cached keys: for every head h and position
 * p < n_pos,
 *   scores[h][p] = sum over the blocks k of row (h, p) of d_k * d_q * s_k,
 * s_k the integer dot of the key codes (c - 8 for Q4_0) with the codes of
 * q[h] quantized to Q8_0 in the kernel (the arithmetic of gq_quantize_rows),
 * i.e. gq_matmul of head h's first n_pos rows with q[h] as one vector.  The
 * 1/sqrt(head_dim) factor and the softmax are the caller's.
 *   q      : device float[n_heads][head_dim], 4-byte aligned.
 *   scores : device float[n_heads][n_pos], 4-byte aligned.
 *   n_pos  : 0 .. capacity (0 is a no-op). */
gq_status gq_kv_scores(gq_type type, const void *cache, const float *q, float *scores, int64_t n_heads,
                       int64_t head_dim, int64_t capacity, int64_t n_pos, gq_stream_t stream);

/* Test switch for the device timeout path (not for production use).  With
 * on != 0, subsequent gq_kv_scores launches (process-wide) make one
 * warp per CTA arm its transfer barrier for its key span without issuing the
 * copy and wait on it with a short poll limit: the wait runs out with no copy
 * in flight, those scores are left unwritten and gq_device_status() reports
 * GQ_ERR_TIMEOUT.  Nothing faults or hangs, and the device stays usable.
 * on = 0 restores normal operation.  Applies to key spans of 4 KB or more
 * (Q8_0 keys at head_dim >= 128).  Returns GQ_ERR_CUDA without a usable CUDA
 * device.  (After a real timeout, as opposed to this switch, the results of
 * the call that timed out and the state of the context are suspect.) */
gq_status gq_debug_kv_timeout(int on);

/* Batch size at and above which GQ_PATH_AUTO uses the tensor-core kernels:
 * for Q4_0 / Q8_0 weights, and for Q4_K at any row count (16, the measured
 * crossover for the smaller matrices; Q4_K from batch 9 on matrices of
 * 14336 rows or more).  The
 * environment variable GQ_TC_MIN_BATCH, read once, replaces both with a
 * plain threshold, which this then returns. */
int64_t gq_tc_min_batch(void);

/*
 * The kernel family GQ_PATH_AUTO takes for a product (GQ_PATH_GEMV,
 * GQ_PATH_MMA or GQ_PATH_SKINNY) on quantized activations, as gq_matmul
 * (with_workspace == 0) or gq_matmul_ws with a sufficient workspace
 * (with_workspace != 0) would choose it: the rules of the Dispatch paragraph
 * of gq_matmul and gq_matmul_ws, including GQ_TC_MIN_BATCH.  Host-only
 * arithmetic on the sizes: no device call, no CUDA device needed.  Empty
 * products report GQ_PATH_GEMV.
 *   path : host, written on success.
 * Errors: GQ_ERR_NULL (path), GQ_ERR_TYPE (not a weight type), GQ_ERR_SHAPE
 * (negative size, cols not a block multiple).
 */
gq_status gq_auto_path(gq_type wtype, int64_t rows, int64_t cols, int64_t batch, int with_workspace,
                       gq_path *path);

/*
 * Reads (and with reset != 0 clears) the device status word of the current
 * device.  Synchronizes the device.  Returns GQ_OK when no bounded wait ran
 * out since the last reset, GQ_ERR_TIMEOUT otherwise (the raw word, a bit
 * mask of the kernels that gave up, is stored to *word when word != NULL),
 * GQ_ERR_CUDA if the query itself failed.  Not callable during stream
 * capture.
 */
gq_status gq_device_status(uint32_t *word, int reset);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H */
