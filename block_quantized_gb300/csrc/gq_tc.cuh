// gq_tc.cuh -- tcgen05 / mbarrier helpers shared by the tensor-core kernels
// (gq_mma.cu: Q4_K x Q8_K; gq_mma_q0.cu: Q4_0 / Q8_0 x Q8_0).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gq_common.cuh"

namespace gq {

// cuTensorMapEncodeTiled, looked up once through the runtime (gq_mma.cu);
// nullptr when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace tc {

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row groups
// 1024 bytes apart; K advances inside the swizzle atom by moving the start
// address (32 bytes per 16 fp16).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate, A/B fp16 (fmt 0) or
// bf16 (fmt 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, uint32_t fmt) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// One MMA with both operands in shared memory.
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far
// has completed.
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
// Generic-proxy shared-memory writes become visible to the async proxy
// (the tensor core reading an operand tile).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// K step visited at step i of a CTA's K loop: every row tile starts at its
// own step (rot), so the CTAs running at the same time read different
// activation tiles instead of all hitting the same L2 lines.
__device__ __forceinline__ int kslot(int i, int rot, int n) { return i + rot < n ? i + rot : i + rot - n; }

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

}  // namespace tc
}  // namespace gq
