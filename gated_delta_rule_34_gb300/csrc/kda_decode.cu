// kda_decode.cu -- one decode token per (sequence, head), state updated in place.
//
//   a  = exp(g),  g = -5 * sigmoid(exp(A) (.) z)        (per channel)
//   S' = Diag(a) S
//   u  = b (v - S'^T k)
//   S  <- S' + k u^T                                  (= (I - b k k^T) S' + b k v^T)
//   o  = S'^T q + u (k^T q)                           (= S_new^T q)
//
// The recurrence is the delta rule of "Kimi K3 architecture: how an open model with a million-token context competes with market leaders"
// (section "How the Kimi K3 architecture holds a million tokens of context") with
// the gate of "How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens"
// (section "Sequence: three KDA to one global MLA").  The same page notes, in
// "How to serve two different caches", that reading the large recurrent state
// is what decoding costs, so this kernel is built around one pass over S.
//
// Design (HBM-bound; > 99% of the bytes are the fp32 state):
//   one CTA of 256 threads per (b, h); warp w owns the 16-column slab
//   [16w, 16w + 16) of S for all rows; lane (rg = lane / 4, cg = lane % 4)
//   owns columns 16w + 4cg .. +3 (one float4) of rows rg, rg + 8, ..., rg + 120.
//   Every thread issues its 16 float4 loads before anything else, keeps its
//   64 state values in registers between the read and the write, and reduces
//   S'^T k and S'^T q over d_k with in-thread sums plus three xor-shuffles
//   (lane bits 2..4).  No shared-memory reduction, no second pass over S.
//   Loads and stores use the streaming cache hint: S is touched exactly once.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeRows = 16;   // rows per thread: 8 row groups x 16 = 128

template <typename T>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
              const T* __restrict__ z, const T* __restrict__ beta, const float* __restrict__ A,
              float* __restrict__ state, T* __restrict__ o, int H, int dk, int dv) {
    const int bh = blockIdx.x;
    const int h = bh % H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 2, cg = lane & 3;
    const int j0 = warp * 16 + cg * 4;
    const bool col_ok = j0 < dv;
    float* Sbh = state + (size_t)bh * dk * dv;

    // 1. Issue the whole state read first (16 independent 128-bit loads).
    float4 s[kDecodeRows];
#pragma unroll
    for (int i = 0; i < kDecodeRows; ++i) {
        const int r = rg + 8 * i;
        if (col_ok && r < dk)
            s[i] = __ldcs(reinterpret_cast<const float4*>(Sbh + (size_t)r * dv + j0));
        else
            s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // 2. Per-channel vectors (gate inline from z; g itself is never stored).
    __shared__ float s_a[128], s_k[128], s_q[128];
    if (tid < 128) {
        float kk = 0.f, qq = 0.f, aa = 1.f;
        if (tid < dk) {
            const size_t idx = (size_t)bh * dk + tid;
            kk = to_f32(k[idx]);
            qq = to_f32(q[idx]);
            aa = expf(gate_accurate(expf(A[(size_t)h * dk + tid]), to_f32(z[idx])));
        }
        s_a[tid] = aa;
        s_k[tid] = kk;
        s_q[tid] = qq;
    }
    const float b = to_f32(beta[bh]);
    float vj[4] = {0.f, 0.f, 0.f, 0.f};
    if (col_ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) vj[c] = to_f32(v[(size_t)bh * dv + j0 + c]);
    }
    __syncthreads();

    // k^T q, computed redundantly by every warp (no extra barrier).
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) kq += s_k[lane + 32 * m] * s_q[lane + 32 * m];
    kq = warp_sum(kq);

    // 3. Decay and the two reductions over d_k.
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kDecodeRows; ++i) {
        const int r = rg + 8 * i;
        const float a = s_a[r], kr = s_k[r], qr = s_q[r];
        s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
        pk[0] = fmaf(s[i].x, kr, pk[0]); pk[1] = fmaf(s[i].y, kr, pk[1]);
        pk[2] = fmaf(s[i].z, kr, pk[2]); pk[3] = fmaf(s[i].w, kr, pk[3]);
        pq[0] = fmaf(s[i].x, qr, pq[0]); pq[1] = fmaf(s[i].y, qr, pq[1]);
        pq[2] = fmaf(s[i].z, qr, pq[2]); pq[3] = fmaf(s[i].w, qr, pq[3]);
    }
#pragma unroll
    for (int m = 4; m <= 16; m <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], m);
            pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], m);
        }
    }
    float u[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = b * (vj[c] - pk[c]);

    // 4. Output (one lane per column group) and the in-place state write.
    if (col_ok && rg == 0) {
        T* ob = o + (size_t)bh * dv + j0;
#pragma unroll
        for (int c = 0; c < 4; ++c) ob[c] = from_f32<T>(fmaf(u[c], kq, pq[c]));
    }
#pragma unroll
    for (int i = 0; i < kDecodeRows; ++i) {
        const int r = rg + 8 * i;
        if (col_ok && r < dk) {
            const float kr = s_k[r];
            float4 w;
            w.x = fmaf(kr, u[0], s[i].x);
            w.y = fmaf(kr, u[1], s[i].y);
            w.z = fmaf(kr, u[2], s[i].z);
            w.w = fmaf(kr, u[3], s[i].w);
            __stcs(reinterpret_cast<float4*>(Sbh + (size_t)r * dv + j0), w);
        }
    }
}

cudaError_t run_decode(const void* q, const void* k, const void* v, const void* z,
                       const void* beta, const float* A, float* state, void* o, int B, int H,
                       int dk, int dv, bool bf16, cudaStream_t stream) {
    const unsigned grid = (unsigned)((int64_t)B * H);
    if (bf16) {
        using T = __nv_bfloat16;
        decode_kernel<T><<<grid, kDecodeThreads, 0, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
            static_cast<const T*>(z), static_cast<const T*>(beta), A, state,
            static_cast<T*>(o), H, dk, dv);
    } else {
        decode_kernel<float><<<grid, kDecodeThreads, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k),
            static_cast<const float*>(v), static_cast<const float*>(z),
            static_cast<const float*>(beta), A, state, static_cast<float*>(o), H, dk, dv);
    }
    return cudaGetLastError();
}

}  // namespace kda
