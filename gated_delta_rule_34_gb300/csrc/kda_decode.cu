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
    // The row pointer is formed here, out of the compiler's sight, so that the
    // 16 row addresses of the read are not held until the write.
    float* row = Sbh + (size_t)rg * dv + j0;
    asm volatile("mov.b64 %0, %0;" : "+l"(row));
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
            __stcs(reinterpret_cast<float4*>(row), w);
        }
        row += (size_t)8 * dv;
    }
}

// ---------------------------------------------------------------------------
// decode_stream_kernel: the same step for d_k = d_v = 128, persistent, with
// the next (b, h) state streamed in while the current one is finished.  Each
// thread copies its own 16 x 16 bytes of the next state into its own slots of
// shared memory with cp.async (so no barrier guards the buffer), issued as soon
// as the current state's values have been consumed from registers; the
// reductions, the output and the 64 KiB state write of the current pair then
// overlap the next pair's read.  Two CTAs per SM keep about 128 KiB of state
// reads in flight per SM.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16_cg(void* dst_smem, const void* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8_ca(void* dst_smem, const void* src) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst_smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// 16-byte async copy that fills the 16 - src_bytes bytes past the source with zeros.
__device__ __forceinline__ void cp_async16_zfill(void* dst_smem, const void* src, uint32_t src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst_smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all_own() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

constexpr uint32_t kStreamSmem = kDecodeRows * kDecodeThreads * 16;   // 64 KiB

template <typename T>
__global__ void __launch_bounds__(kDecodeThreads, 2)
decode_stream_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ z, const T* __restrict__ beta,
                     const float* __restrict__ A, float* __restrict__ state, T* __restrict__ o,
                     int H, int n_pairs) {
    constexpr int d = 128;
    extern __shared__ float4 s_buf[];                 // [kDecodeRows][kDecodeThreads]
    __shared__ float s_a[d], s_k[d], s_q[d];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane >> 2, cg = lane & 3;
    const int j0 = warp * 16 + cg * 4;
    auto prefetch = [&](int bh) {
        const float* Sbh = state + (size_t)bh * d * d;
#pragma unroll
        for (int i = 0; i < kDecodeRows; ++i)
            cp_async16_cg(&s_buf[i * kDecodeThreads + tid], Sbh + (size_t)(rg + 8 * i) * d + j0);
    };
    int bh = blockIdx.x;
    if (bh < n_pairs) prefetch(bh);
    for (; bh < n_pairs; bh += gridDim.x) {
        const int h = bh % H;
        float* Sbh = state + (size_t)bh * d * d;
        __syncthreads();                              // the previous pair is done with s_a, s_k, s_q
        if (tid < d) {
            const size_t idx = (size_t)bh * d + tid;
            s_k[tid] = to_f32(k[idx]);
            s_q[tid] = to_f32(q[idx]);
            s_a[tid] = expf(gate_accurate(expf(A[(size_t)h * d + tid]), to_f32(z[idx])));
        }
        const float b = to_f32(beta[bh]);
        float vj[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) vj[c] = to_f32(v[(size_t)bh * d + j0 + c]);
        __syncthreads();
        float kq = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) kq += s_k[lane + 32 * m] * s_q[lane + 32 * m];
        kq = warp_sum(kq);

        cp_async_wait_all_own();                      // this thread's slots of the state
        float4 s[kDecodeRows];
#pragma unroll
        for (int i = 0; i < kDecodeRows; ++i) s[i] = s_buf[i * kDecodeThreads + tid];
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
        // every s[i] has been consumed: the slots can take the next pair
        if (bh + (int)gridDim.x < n_pairs) prefetch(bh + gridDim.x);
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
        if (rg == 0) {
            T* ob = o + (size_t)bh * d + j0;
#pragma unroll
            for (int c = 0; c < 4; ++c) ob[c] = from_f32<T>(fmaf(u[c], kq, pq[c]));
        }
#pragma unroll
        for (int i = 0; i < kDecodeRows; ++i) {
            const int r = rg + 8 * i;
            const float kr = s_k[r];
            float4 w;
            w.x = fmaf(kr, u[0], s[i].x);
            w.y = fmaf(kr, u[1], s[i].y);
            w.z = fmaf(kr, u[2], s[i].z);
            w.w = fmaf(kr, u[3], s[i].w);
            __stcs(reinterpret_cast<float4*>(Sbh + (size_t)r * d + j0), w);
        }
    }
    cp_async_wait_all_own();
}

cudaError_t run_decode(const void* q, const void* k, const void* v, const void* z,
                       const void* beta, const float* A, float* state, void* o, int B, int H,
                       int dk, int dv, bool bf16, cudaStream_t stream) {
    const unsigned grid = (unsigned)((int64_t)B * H);
    // Other head sizes: a warp per 16 columns of S, and at least four warps (thread
    // c < 128 loads channel c of k, q, z); smaller CTAs let more pairs be resident.
    const int col_warps = (dv + 15) / 16;
    const int threads = 32 * (col_warps < 4 ? 4 : col_warps);
    if (dk == 128 && dv == 128) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int n_pairs = B * H;
        const unsigned sgrid = (unsigned)(n_pairs < 2 * sms ? n_pairs : 2 * sms);
        if (bf16) {
            using T = __nv_bfloat16;
            e = cudaFuncSetAttribute(decode_stream_kernel<T>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
            if (e != cudaSuccess) return e;
            decode_stream_kernel<T><<<sgrid, kDecodeThreads, kStreamSmem, stream>>>(
                static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
                static_cast<const T*>(z), static_cast<const T*>(beta), A, state,
                static_cast<T*>(o), H, n_pairs);
        } else {
            e = cudaFuncSetAttribute(decode_stream_kernel<float>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem);
            if (e != cudaSuccess) return e;
            decode_stream_kernel<float><<<sgrid, kDecodeThreads, kStreamSmem, stream>>>(
                static_cast<const float*>(q), static_cast<const float*>(k),
                static_cast<const float*>(v), static_cast<const float*>(z),
                static_cast<const float*>(beta), A, state, static_cast<float*>(o), H, n_pairs);
        }
        return cudaGetLastError();
    }
    if (bf16) {
        using T = __nv_bfloat16;
        decode_kernel<T><<<grid, threads, 0, stream>>>(
            static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
            static_cast<const T*>(z), static_cast<const T*>(beta), A, state,
            static_cast<T*>(o), H, dk, dv);
    } else {
        decode_kernel<float><<<grid, threads, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k),
            static_cast<const float*>(v), static_cast<const float*>(z),
            static_cast<const float*>(beta), A, state, static_cast<float*>(o), H, dk, dv);
    }
    return cudaGetLastError();
}

}  // namespace kda

// ---------------------------------------------------------------------------
// Speculative decoding: verify a span of draft tokens, then commit the
// accepted prefix.  "How Kimi K3 is built" (section "How to serve two
// different caches") describes K3 keeping the small input projections of the
// draft tokens instead of a copy of the state after each one, and recomputing
// the accepted span on chip.  Both kernels read S once into registers and
// step through up to kSpecMaxT tokens in fp32:
//   verify  o_t for every draft token; S is not written.
//   commit  S advanced by the first n_accept[b] tokens, written once in place.
//
// Decay factoring over the span: with gam_t = prod_{s <= t} a_s (per channel,
// at least e^{-5 kSpecMaxT} = e^-80, inside the fp32 range) the registers hold
// R = Diag(1 / gam) S, so that a token needs no rescaling of the state:
//   S'^T k = R^T (gam_t k),  S'^T q = R^T (gam_t q),  u = b (v - S'^T k),
//   R <- R + (k / gam_t) u^T,  o_t = S'^T q + u (k^T q),
// and commit writes S = Diag(gam_T) R.  Thread layout: warp w owns columns
// 16 w .. 16 w + 15; lane (rq = lane / 8, cq = lane % 8) holds rows
// 32 rq .. 32 rq + 31 of columns 16 w + 2 cq, + 1 (64 registers), so the d_k
// reductions are in-thread sums plus two xor-shuffles, and the per-row vectors
// are read as float4 from shared memory rows whose quarters are skewed by four
// floats (no bank conflict between the four row quarters).
// ---------------------------------------------------------------------------
namespace kda {

constexpr int kSpecMaxT = 16;
// The state staged row by row: rows of 128 floats, the four 32-row quarters 16
// floats apart, so that a warp's row-pair reads (four quarters x 64 bytes) take
// the two wavefronts 256 bytes need.
constexpr int kStageQuarter = 32 * 128 + 16;                      // floats per quarter
constexpr uint32_t kSpecStage = 4 * kStageQuarter * 4;            // 64.25 KiB
__device__ __forceinline__ int stage_at(int r, int c) { return (r >> 5) * kStageQuarter + (r & 31) * 128 + c; }
constexpr int kSpecPitch = 4 * 36;   // floats per token row: four 32-row quarters, each + 4 pad

__device__ __forceinline__ int spec_row(int c) { return (c >> 5) * 36 + (c & 31); }

// src[0 .. n) as floats, zeros past n (n <= 8): one 16-byte load (bf16) or two
// (fp32) when all eight are present and `vec` says the run is 16-byte aligned.
__device__ __forceinline__ void load_run8(const __nv_bfloat16* __restrict__ src, int n, bool vec,
                                          float (&f)[8]) {
    if (vec && n == 8) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(src));
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = __bfloat1622float2(b2[e]);
            f[2 * e] = x.x;
            f[2 * e + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = e < n ? __bfloat162float(src[e]) : 0.f;
    }
}
__device__ __forceinline__ void load_run8(const float* __restrict__ src, int n, bool vec, float (&f)[8]) {
    if (vec && n == 8) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(src));
        const float4 c = __ldg(reinterpret_cast<const float4*>(src) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = e < n ? src[e] : 0.f;
    }
}

template <typename T, bool kVerify>
__global__ void __launch_bounds__(kDecodeThreads, 2)
spec_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
            const T* __restrict__ z, const T* __restrict__ beta, const float* __restrict__ A,
            float* __restrict__ state, T* __restrict__ o, const int32_t* __restrict__ n_accept,
            int Tn, int H, int dk, int dv, int pf_dist) {
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh % H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rq = lane >> 3, cq = lane & 7;
    const int r0 = 32 * rq, j0 = warp * 16 + 2 * cq;
    const bool col_ok = j0 < dv;            // dv is a multiple of 4: both columns or neither
    float* Sbh = state + (size_t)bh * dk * dv;
    int n_steps = Tn;
    if (!kVerify) {
        const int na = n_accept[b];
        n_steps = na < 0 ? 0 : (na > Tn ? Tn : na);
        if (n_steps == 0) return;                       // nothing accepted: S unchanged
    }

    // Verify asks L2 for the draft span of pair bh + pf_dist, which starts
    // about one wave of CTAs later, so that its loads hit L2 instead of
    // queueing behind the states being streamed: thread (part, tensor, token)
    // takes one 128-byte line of one token row.  (In commit the same request
    // costs more than it saves: the kernel has no registers to spare.)
    if (kVerify && pf_dist > 0 && bh + pf_dist < (int)gridDim.x) {
        const int p2 = bh + pf_dist, b2 = p2 / H, h2 = p2 - (p2 / H) * H;
        const int t = tid & 15, which = (tid >> 4) & 3, part = tid >> 6;
        const T* src = which == 0 ? k : which == 1 ? q : which == 2 ? v : z;
        const int d = which == 2 ? dv : dk;
        if (t < Tn && part * 128 < d * (int)sizeof(T))
            prefetch_line_l2(reinterpret_cast<const char*>(src + ((size_t)(b2 * Tn + t) * H + h2) * d) + part * 128);
    }

    // The state read starts first: each thread copies its own 32 x 8 bytes into
    // its own shared-memory slots (cp.async, no registers held), so the read
    // overlaps the per-token preparation below; rows past d_k read as zeros.
    extern __shared__ __align__(16) float s_stage[];
    {
        // warp w copies rows w, w + 8, ...: 16 bytes a lane, one 512-byte row a warp
        const int c4 = 4 * lane;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = warp + 8 * i;
            const bool in = r < dk && c4 < dv;
            cp_async16_zfill(&s_stage[stage_at(r, c4)], in ? Sbh + (size_t)r * dv + c4 : Sbh, in ? 16u : 0u);
        }
    }

    // Per-token vectors: gam_t k, gam_t q, k / gam_t (rows skewed), v, beta, k^T q.
    __shared__ __align__(16) float s_kg[kSpecMaxT][kSpecPitch], s_qg[kSpecMaxT][kSpecPitch];
    __shared__ __align__(16) float s_kh[kSpecMaxT][kSpecPitch];
    __shared__ __align__(16) float s_v[kSpecMaxT][128], s_L[kSpecMaxT][128];
    __shared__ float s_b[kSpecMaxT], s_kq[kSpecMaxT], s_gam[128];
    // (a) thread (token tt = tid / 16, channels 8 c8 .. 8 c8 + 7, c8 = tid % 16)
    //     loads 16 bytes of each input row at once, so that the span takes one
    //     round of wide loads: raw k and q, v, the gate g, and k^T q summed over
    //     the token's 16 lanes.
    {
        const int tt = tid >> 4, c8 = tid & 15, cb = 8 * c8;
        const bool live = tt < n_steps;
        const size_t row = ((size_t)b * Tn + (live ? tt : 0)) * H + h;
        const int nk = live ? (dk - cb < 0 ? 0 : (dk - cb > 8 ? 8 : dk - cb)) : 0;
        const int nv = live ? (dv - cb < 0 ? 0 : (dv - cb > 8 ? 8 : dv - cb)) : 0;
        constexpr int kVec = 16 / (int)sizeof(T);          // elements per 16 bytes
        float kf[8], qf[8], zf[8], vf[8], af[8];
        load_run8(k + row * dk + cb, nk, dk % kVec == 0, kf);
        if (kVerify) load_run8(q + row * dk + cb, nk, dk % kVec == 0, qf);
        else
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[e] = 0.f;
        load_run8(z + row * dk + cb, nk, dk % kVec == 0, zf);
        load_run8(v + row * dv + cb, nv, dv % kVec == 0, vf);
        load_run8(A + (size_t)h * dk + cb, nk, dk % 4 == 0, af);
        if (live) {
            float g[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = e < nk ? gate_accurate(expf(af[e]), zf[e]) : 0.f;
            // channels cb .. cb + 7 lie in one 32-channel quarter of the skewed rows
            float4* kh4 = reinterpret_cast<float4*>(&s_kh[tt][spec_row(cb)]);
            float4* qg4 = reinterpret_cast<float4*>(&s_qg[tt][spec_row(cb)]);
            float4* l4 = reinterpret_cast<float4*>(&s_L[tt][cb]);
            float4* v4 = reinterpret_cast<float4*>(&s_v[tt][cb]);
            kh4[0] = make_float4(kf[0], kf[1], kf[2], kf[3]);
            kh4[1] = make_float4(kf[4], kf[5], kf[6], kf[7]);
            qg4[0] = make_float4(qf[0], qf[1], qf[2], qf[3]);
            qg4[1] = make_float4(qf[4], qf[5], qf[6], qf[7]);
            l4[0] = make_float4(g[0], g[1], g[2], g[3]);
            l4[1] = make_float4(g[4], g[5], g[6], g[7]);
            v4[0] = make_float4(vf[0], vf[1], vf[2], vf[3]);
            v4[1] = make_float4(vf[4], vf[5], vf[6], vf[7]);
        }
        if (kVerify) {
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) p = fmaf(kf[e], qf[e], p);
#pragma unroll
            for (int m = 1; m <= 8; m <<= 1) p += __shfl_xor_sync(0xffffffffu, p, m);
            if (live && c8 == 0) s_kq[tt] = p;
        }
    }
    if (tid < n_steps) s_b[tid] = to_f32(beta[((size_t)b * Tn + tid) * H + h]);
    __syncthreads();
    // (b) the running log-decay per channel, in place
    if (tid < 128) {
        float L = 0.f;
        for (int t = 0; t < n_steps; ++t) {
            L += s_L[t][tid];
            s_L[t][tid] = L;
        }
    }
    __syncthreads();
    // (c) the decay-scaled vectors, every (token, channel) at once
    for (int idx = tid; idx < n_steps * 128; idx += kDecodeThreads) {
        const int t = idx >> 7, c = idx & 127, r = spec_row(c);
        const float L = s_L[t][c];
        const float gam = expf(L), igam = expf(-L);
        const float kk = s_kh[t][r];
        s_kg[t][r] = gam * kk;
        s_qg[t][r] = gam * s_qg[t][r];
        s_kh[t][r] = igam * kk;
        if (t == n_steps - 1) s_gam[c] = gam;
    }
    __syncthreads();
    // R = S on entry (gam_0 = 1), held as row pairs sp[p][u] = (R[r0 + 2p][j0 + u],
    // R[r0 + 2p + 1][j0 + u]) on which packed two-lane FMAs run.  The rows were
    // copied by other warps: every thread's copies land before any is read.
    cp_async_wait_all_own();
    __syncthreads();
    uint64_t sp[16][2];
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const float2 a = *reinterpret_cast<const float2*>(&s_stage[stage_at(r0 + 2 * p, j0)]);
        const float2 c = *reinterpret_cast<const float2*>(&s_stage[stage_at(r0 + 2 * p + 1, j0)]);
        sp[p][0] = f2_pack(a.x, c.x);
        sp[p][1] = f2_pack(a.y, c.y);
    }

    for (int t = 0; t < n_steps; ++t) {
        // two accumulators per column and vector halve the dependent FMA chains
        uint64_t pk[2][2] = {{0ull, 0ull}, {0ull, 0ull}}, pq[2][2] = {{0ull, 0ull}, {0ull, 0ull}};
        const ulonglong2* kg2 = reinterpret_cast<const ulonglong2*>(&s_kg[t][36 * rq]);
        const ulonglong2* qg2 = reinterpret_cast<const ulonglong2*>(&s_qg[t][36 * rq]);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
            const ulonglong2 kg = kg2[i4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                pk[0][u] = f2_fma(sp[2 * i4][u], kg.x, pk[0][u]);
                pk[1][u] = f2_fma(sp[2 * i4 + 1][u], kg.y, pk[1][u]);
            }
            if (kVerify) {
                const ulonglong2 qg = qg2[i4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    pq[0][u] = f2_fma(sp[2 * i4][u], qg.x, pq[0][u]);
                    pq[1][u] = f2_fma(sp[2 * i4 + 1][u], qg.y, pq[1][u]);
                }
            }
        }
        float sk[2], sq[2] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float2 k0 = f2_unpack(pk[0][u]), k1 = f2_unpack(pk[1][u]);
            sk[u] = (k0.x + k0.y) + (k1.x + k1.y);
            if (kVerify) {
                const float2 q0 = f2_unpack(pq[0][u]), q1 = f2_unpack(pq[1][u]);
                sq[u] = (q0.x + q0.y) + (q1.x + q1.y);
            }
        }
#pragma unroll
        for (int m = 8; m <= 16; m <<= 1) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                sk[c] += __shfl_xor_sync(0xffffffffu, sk[c], m);
                if (kVerify) sq[c] += __shfl_xor_sync(0xffffffffu, sq[c], m);
            }
        }
        const float bt = s_b[t];
        const float2 vv = col_ok ? *reinterpret_cast<const float2*>(&s_v[t][j0]) : make_float2(0.f, 0.f);
        const float u0 = bt * (vv.x - sk[0]), u1 = bt * (vv.y - sk[1]);
        if (kVerify && col_ok && rq == 0) {
            const float kq = s_kq[t];
            T* ob = o + (((size_t)b * Tn + t) * H + h) * dv + j0;
            ob[0] = from_f32<T>(fmaf(u0, kq, sq[0]));
            ob[1] = from_f32<T>(fmaf(u1, kq, sq[1]));
        }
        if (!kVerify || t + 1 < n_steps) {
            const ulonglong2* kh2 = reinterpret_cast<const ulonglong2*>(&s_kh[t][36 * rq]);
            const uint64_t uu[2] = {f2_pack(u0, u0), f2_pack(u1, u1)};
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
                const ulonglong2 kh = kh2[i4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    sp[2 * i4][u] = f2_fma(kh.x, uu[u], sp[2 * i4][u]);
                    sp[2 * i4 + 1][u] = f2_fma(kh.y, uu[u], sp[2 * i4 + 1][u]);
                }
            }
        }
    }
    if (!kVerify) {
        // The row pointer is formed here, out of the compiler's sight, so that the
        // 32 store addresses are not computed before the token loop and held
        // through it (they would not fit in the registers left).
        float* row = Sbh + (size_t)r0 * dv + j0;
        asm volatile("mov.b64 %0, %0;" : "+l"(row));
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const int r = r0 + 2 * p;
            const uint64_t g = f2_pack(s_gam[r & 127], s_gam[(r + 1) & 127]);
            const float2 a = f2_unpack(f2_mul(sp[p][0], g)), c = f2_unpack(f2_mul(sp[p][1], g));
            if (col_ok && r < dk) __stcs(reinterpret_cast<float2*>(row), make_float2(a.x, c.x));
            row += dv;
            if (col_ok && r + 1 < dk) __stcs(reinterpret_cast<float2*>(row), make_float2(a.y, c.y));
            row += dv;
        }
    }
}

cudaError_t run_spec(const void* q, const void* k, const void* v, const void* z, const void* beta,
                     const float* A, float* state, void* o, const int32_t* n_accept, int B, int Tn,
                     int H, int dk, int dv, bool bf16, bool verify, cudaStream_t stream) {
    const unsigned grid = (unsigned)((int64_t)B * H);
    constexpr int kMaxDevices = 64;
    static bool attr_done[kMaxDevices] = {};
    static int sm_count[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (sm_count[dev] == 0) {
        e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    // two CTAs per SM are resident: the pair one wave ahead
    const int pf_dist = 2 * sm_count[dev];
    if (!attr_done[dev]) {
        const void* fns[4] = {(const void*)spec_kernel<__nv_bfloat16, true>,
                              (const void*)spec_kernel<__nv_bfloat16, false>,
                              (const void*)spec_kernel<float, true>, (const void*)spec_kernel<float, false>};
        for (const void* fn : fns) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSpecStage);
            if (e != cudaSuccess) return e;
        }
        attr_done[dev] = true;
    }
    if (bf16) {
        using Tb = __nv_bfloat16;
        auto kq = static_cast<const Tb*>(q);
        auto kk = static_cast<const Tb*>(k);
        auto kv = static_cast<const Tb*>(v);
        auto kz = static_cast<const Tb*>(z);
        auto kb = static_cast<const Tb*>(beta);
        if (verify)
            spec_kernel<Tb, true><<<grid, kDecodeThreads, kSpecStage, stream>>>(
                kq, kk, kv, kz, kb, A, state, static_cast<Tb*>(o), n_accept, Tn, H, dk, dv, pf_dist);
        else
            spec_kernel<Tb, false><<<grid, kDecodeThreads, kSpecStage, stream>>>(
                kq, kk, kv, kz, kb, A, state, static_cast<Tb*>(o), n_accept, Tn, H, dk, dv, pf_dist);
    } else {
        auto kq = static_cast<const float*>(q);
        auto kk = static_cast<const float*>(k);
        auto kv = static_cast<const float*>(v);
        auto kz = static_cast<const float*>(z);
        auto kb = static_cast<const float*>(beta);
        if (verify)
            spec_kernel<float, true><<<grid, kDecodeThreads, kSpecStage, stream>>>(
                kq, kk, kv, kz, kb, A, state, static_cast<float*>(o), n_accept, Tn, H, dk, dv, pf_dist);
        else
            spec_kernel<float, false><<<grid, kDecodeThreads, kSpecStage, stream>>>(
                kq, kk, kv, kz, kb, A, state, static_cast<float*>(o), n_accept, Tn, H, dk, dv, pf_dist);
    }
    return cudaGetLastError();
}

}  // namespace kda
