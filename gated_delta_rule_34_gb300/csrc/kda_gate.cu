// kda_gate.cu -- the forget gate as a standalone elementwise kernel.
//
//   g[t, h, c] = clamp(-5 * sigmoid(exp(A[h, c]) * z[t, h, c]), -5, 0)
//
// "How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens",
// section "Sequence: three KDA to one global MLA" (g_min = -5).
// Memory-bound: 2 (bf16) or 4 (fp32) bytes in and 4 bytes out per element.
// Each thread handles one 16-byte vector of z when d_k allows it, so loads
// and stores are 128-bit and fully coalesced.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

template <typename T, int VEC>
__global__ void __launch_bounds__(256) gate_kernel(const T* __restrict__ z,
                                                   const float* __restrict__ A,
                                                   float* __restrict__ g, int64_t n_vec, int H,
                                                   int dk) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const int64_t e0 = i * VEC;                  // first element; VEC divides dk
        const int c0 = (int)(e0 % dk);
        const int h = (int)((e0 / dk) % H);
        const float* Ah = A + (int64_t)h * dk + c0;
        float zf[VEC];
        if constexpr (VEC == 8) {
            const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(z + e0));
            const __nv_bfloat16* zb = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
            for (int j = 0; j < 8; ++j) zf[j] = to_f32(zb[j]);
        } else if constexpr (VEC == 4) {
            const float4 raw = __ldcs(reinterpret_cast<const float4*>(z + e0));
            zf[0] = raw.x; zf[1] = raw.y; zf[2] = raw.z; zf[3] = raw.w;
        } else {
            zf[0] = to_f32(z[e0]);
        }
        float out[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) out[j] = gate_accurate(expf(__ldg(Ah + j)), zf[j]);
        if constexpr (VEC >= 4) {
#pragma unroll
            for (int j = 0; j < VEC; j += 4)
                __stcs(reinterpret_cast<float4*>(g + e0 + j),
                       make_float4(out[j], out[j + 1], out[j + 2], out[j + 3]));
        } else {
            g[e0] = out[0];
        }
    }
}

template <typename T, int VEC>
static cudaError_t launch_gate(const void* z, const float* A, float* g, int64_t n, int H, int dk,
                               cudaStream_t stream, int num_sms) {
    const int64_t n_vec = n / VEC;
    int64_t blocks = (n_vec + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    gate_kernel<T, VEC><<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const T*>(z), A, g,
                                                               n_vec, H, dk);
    return cudaGetLastError();
}

cudaError_t run_gate(const void* z, const float* A, float* g, int64_t n_tokens, int H, int dk,
                     bool bf16, cudaStream_t stream, int num_sms) {
    const int64_t n = n_tokens * H * dk;
    if (bf16) {
        if (dk % 8 == 0) return launch_gate<__nv_bfloat16, 8>(z, A, g, n, H, dk, stream, num_sms);
        return launch_gate<__nv_bfloat16, 1>(z, A, g, n, H, dk, stream, num_sms);
    }
    if (dk % 4 == 0) return launch_gate<float, 4>(z, A, g, n, H, dk, stream, num_sms);
    return launch_gate<float, 1>(z, A, g, n, H, dk, stream, num_sms);
}

}  // namespace kda
