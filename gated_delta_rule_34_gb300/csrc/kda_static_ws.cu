// kda_static_ws.cu -- prefill that uses a library-owned scratch area instead of a
// caller workspace, for callers that cannot allocate device memory.
//
// The chunked tensor-core prefill needs scratch memory for its per-chunk
// operand packages.  kda_chunk_prefill takes that scratch from the caller.
// Some callers cannot allocate device memory when they call the layer: a
// plugin hosted by a runtime that owns every device allocation and forbids
// its plugins from calling cudaMalloc, or a serving loop whose memory plan is
// fixed at start-up.  This entry point gives them the same computation with
// the scratch taken from a file-scope __device__ array of fixed size,
// KDA_STATIC_WORKSPACE_BYTES.  The array exists on every GPU that loads the
// library and is held until the process exits.
#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[KDA_STATIC_WORKSPACE_BYTES];

// Device address of g_static_workspace for the current device and context.  In
// host code the symbol names a host-side stand-in, so the address must come
// from cudaGetSymbolAddress with the right device current.  It is looked up on
// every call rather than cached: after cudaDeviceReset, or in a second context
// on the same device, the module is loaded again and the array may move.
cudaError_t static_workspace_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_chunk_prefill_static_workspace(
    const void* q, const void* k, const void* v, const void* z, const void* beta,
    const float* A, void* o, const float* initial_state, float* final_state,
    const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H, int d_k, int d_v, int chunk,
    kda_dtype dtype, cudaStream_t stream) {
    const size_t need =
        kda_chunk_prefill_workspace_size(n_seqs, B, T, H, d_k, d_v, chunk, dtype);
    if (need > (size_t)KDA_STATIC_WORKSPACE_BYTES)
        return kda::report(KDA_ERR_UNSUPPORTED,
                           "these sizes need %zu bytes of scratch but the static workspace holds "
                           "%zu; call kda_chunk_prefill with a caller workspace instead",
                           need, (size_t)KDA_STATIC_WORKSPACE_BYTES);
    void* ws = nullptr;
    const cudaError_t e = static_workspace_address(&ws);
    if (e != cudaSuccess)
        return kda::report(KDA_ERR_CUDA, "cudaGetSymbolAddress of the static workspace: %s",
                           cudaGetErrorString(e));
    return kda_chunk_prefill(q, k, v, z, beta, A, o, initial_state, final_state, cu_seqlens,
                             n_seqs, B, T, H, d_k, d_v, chunk, dtype, ws,
                             (size_t)KDA_STATIC_WORKSPACE_BYTES, stream);
}

extern "C" kda_status kda_static_workspace_status(uint32_t* status, cudaStream_t stream) {
    if (status == nullptr) return kda::report(KDA_ERR_INVALID_ARG, "status is NULL");
    if ((reinterpret_cast<uintptr_t>(status) & 3u) != 0)
        return kda::report(KDA_ERR_INVALID_ARG, "status is not 4-byte aligned");
    void* ws = nullptr;
    cudaError_t e = static_workspace_address(&ws);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDefault, stream);
    if (e != cudaSuccess)
        return kda::report(KDA_ERR_CUDA, "kda_static_workspace_status: %s", cudaGetErrorString(e));
    return kda::report(KDA_OK, "%s", "");
}
