// gq_mma.cu -- tensor-core (tcgen05) path for Q4_K x Q8_K at large batch.
#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {

bool mma_supported(int64_t, int64_t, int64_t) { return false; }

cudaError_t launch_mma_q4k(const void *, const void *, float *, int32_t *, int64_t, int64_t,
                           int64_t, const LaunchCtx &) {
    return cudaErrorNotSupported;
}

}  // namespace gq
