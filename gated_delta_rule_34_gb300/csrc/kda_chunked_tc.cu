// kda_chunked_tc.cu -- chunked tensor-core prefill (placeholder until the tcgen05 kernels land).
#include "kda_internal.h"

namespace kda {

size_t chunked_tc_workspace_bytes(int, int64_t, int) { return 0; }

cudaError_t run_chunked_tc(const void*, const void*, const void*, const void*, const void*,
                           const float*, void*, const float*, float*, const int32_t*, int, int64_t,
                           int64_t, int, void*, cudaStream_t, int) {
    return cudaErrorNotSupported;
}

}  // namespace kda
