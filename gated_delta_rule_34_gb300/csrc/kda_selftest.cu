// kda_selftest.cu -- failure detection, exercised without a fault.
//
// Every wait of the tensor-core kernels on an mbarrier (a TMA copy, an MMA
// commit, another warp role) is bounded: after about 2 s of GPU time it gives
// up, the kernel records a status bit in its workspace and returns, and the
// context stays usable.  A wait that runs out only happens when something
// else has already gone wrong, so the product kernels never show that path.
// This kernel does: one thread waits, through the same bounded wait, on an
// mbarrier that nothing arrives on (or, as a control, on one that its own
// arrival completes), and writes what the wait returned.
#include "../../include/kda.h"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace tc {

__global__ void selftest_wait_kernel(uint32_t* status, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (arrive) mbar_arrive(&bar);
    // phase 0 completes only through the arrival above
    *status = mbar_wait(&bar, 0) ? 0u : 1u;
}

}  // namespace tc
}  // namespace kda

extern "C" kda_status kda_selftest_bounded_wait(uint32_t* status, int arrive,
                                                cudaStream_t stream) {
    if (status == nullptr || (reinterpret_cast<uintptr_t>(status) & 3u) != 0)
        return kda::report(KDA_ERR_INVALID_ARG, "status must be a 4-byte aligned device pointer");
    kda::tc::selftest_wait_kernel<<<1, 32, 0, stream>>>(status, arrive ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return kda::report(KDA_ERR_CUDA, "kda_selftest_bounded_wait launch: %s",
                           cudaGetErrorString(e));
    return KDA_OK;
}
