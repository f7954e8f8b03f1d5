// kda_recurrent.cu -- token-by-token prefill in fp32 SIMT arithmetic.
//
// The path for fp32 inputs (tf32 tensor cores cannot meet a 1e-4 relative
// bound) and for head sizes the tensor-core paths do not cover.  It runs the
// delta rule of "Kimi K3 architecture: how an open model with a million-token context competes with market leaders"
// (section "How the Kimi K3 architecture holds a million tokens of context") with the
// per-channel gate of "How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens"
// (section "Sequence: three KDA to one global MLA") token by token:
//
//   S' = Diag(a_t) S,  u = b_t (v_t - S'^T k_t),  S <- S' + k_t u^T,
//   o_t = S'^T q_t + u (k_t^T q_t)
//
// Decay factoring.  Inside a run of at most 8 tokens the registers hold
// R = Diag(1 / gam_t) S, with gam_t the running product of the decays since
// the run started (per channel, >= e^-40, so R stays within e^40 of S), so a
// token needs no rescaling of the state:
//   S'^T k = R^T (gam_t k),  S'^T q = R^T (gam_t q),  R <- R + (k / gam_t) u^T,
// and at the end of the run S = Diag(gam_last) R.  The scaled vectors come
// from the running log-decay L_t (gam_t = e^{L_t}), computed per channel once
// per CTA.  The result is the exact recurrence up to fp32 rounding and the
// fast exponential's error (a few units in the last place, far inside the
// 1e-4 bound for fp32 inputs).
//
// Columns of S evolve independently (column j only sees k, a, b and v[:, j]),
// so the work splits over (sequence, head, column group).  A CTA of eight
// warps owns kCols = 64 or 32 columns; warp w owns kCols / 8 of them, lane
// (rq = lane / kCq, cq = lane mod kCq, kCq = kCols / 16 column pairs) holds
// 128 / (32 / kCq) rows (16 or 8) of columns kCols / 8 w + 2 cq, + 1 (row pairs
// on which packed two-lane FMAs run), so the d_k reductions are in-thread sums
// plus xor-shuffles over the row-group lane bits.  The 32-column form doubles
// the CTAs where 64-column ones would leave most SMs idle (narrow heads, few
// sequences); each CTA repeats the per-token preparation of its tile.  Heads
// with d_k <= 64 hold only kDk = 64 rows, so their lanes own half as many.  Tiles of 16 tokens are staged
// in shared memory; the next tile's raw inputs are loaded into registers while
// the current tile's tokens run.  The per-row vectors sit in rows whose
// 16-channel groups are 20 floats apart, so the eight row groups of a warp
// read them as conflict-free 16-byte loads.
#include <type_traits>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int kRecThreads = 256;
constexpr int kRecTile = 16;     // tokens staged per shared-memory tile
constexpr int kRecRun = 8;       // tokens per factoring run (gam >= e^{-5 kRecRun})
constexpr int kRecPitch = 160;   // floats per token row of the scaled vectors: 8 groups of 16 + 4

__device__ __forceinline__ int rec_idx(int c) { return (c >> 4) * 20 + (c & 15); }

template <typename T, int kCols, int kDk>
__global__ void __launch_bounds__(kRecThreads)
recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const T* __restrict__ z, const T* __restrict__ beta,
                 const float* __restrict__ A, T* __restrict__ o,
                 const float* __restrict__ S0, float* __restrict__ S1,
                 const int32_t* __restrict__ cu, int64_t T_len, int64_t T_total, int H,
                 int dk, int dv, CheckpointSpec ck) {
    static_assert(kCols == 64 || kCols == 32, "column group");
    static_assert(kDk == 128 || kDk == 64, "rows held");
    constexpr int kCq = kCols / 16;                   // column pairs per warp (lanes along columns)
    constexpr int kRows = kDk / (32 / kCq);           // rows per lane: 16, 8 or 4
    constexpr int kPairs = kRows / 2;                 // row pairs per lane
    const int cgrp = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rq = lane / kCq, cq = lane % kCq;
    const int col0 = cgrp * kCols;                    // first column of this CTA
    const int lcol = (kCols / 8) * warp + 2 * cq;     // this lane's first column, CTA-local
    const int r0 = kRows * rq;                        // this lane's first row

    // s_kg holds g, then the running log-decay L, before gam k
    __shared__ __align__(16) float s_kg[kRecTile * kRecPitch], s_qg[kRecTile * kRecPitch];
    __shared__ __align__(16) float s_kh[kRecTile * kRecPitch];
    __shared__ __align__(16) float s_v[kRecTile][kCols], s_o[kRecTile][kCols];
    __shared__ __align__(16) float s_glast[kRecTile / kRecRun][kRecPitch];   // gam at each run's end
    __shared__ float s_b[kRecTile], s_kq[kRecTile];
    __shared__ __align__(16) float s_expA[128];

    int64_t bos, eos;
    seq_bounds(cu, n, T_len, T_total, bos, eos);

    for (int c = tid; c < 128; c += kRecThreads)
        s_expA[c] = c < dk ? expf(A[(size_t)h * dk + c]) : 0.f;

    // State registers: st[p][u] = (S[r0 + 2p][j], S[r0 + 2p + 1][j]) with
    // j = col0 + lcol + u (R inside a run).
    uint64_t st[kPairs][2];
    const size_t sbase = ((size_t)n * H + h) * dk * dv;
    const bool okc[2] = {col0 + lcol < dv, col0 + lcol + 1 < dv};
#pragma unroll
    for (int p2 = 0; p2 < kPairs; ++p2) {
        const int r = r0 + 2 * p2;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float* p = S0 ? S0 + sbase + (size_t)r * dv + col0 + lcol + u : nullptr;
            st[p2][u] = f2_pack((p && r < dk && okc[u]) ? p[0] : 0.f, (p && r + 1 < dk && okc[u]) ? p[dv] : 0.f);
        }
    }
    auto store_state = [&](float* mat) {      // mat: [d_k][d_v] of (n, h)
#pragma unroll
        for (int p2 = 0; p2 < kPairs; ++p2) {
            const int r = r0 + 2 * p2;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float2 x = f2_unpack(st[p2][u]);
                float* p = mat + (size_t)r * dv + col0 + lcol + u;
                if (okc[u] && r < dk) p[0] = x.x;
                if (okc[u] && r + 1 < dk) p[dv] = x.y;
            }
        }
    };

    // The next tile's raw inputs, loaded into registers while the current
    // tile's tokens run: warp w takes tokens w and w + 8, lane l channels
    // 4 l .. 4 l + 3 of q, k, z (one 16-byte load each for fp32, 8 bytes for
    // bf16, where the rows allow); (tt, column) pairs idx = tid + 256 i for v;
    // beta by threads < 16.
    constexpr int kVPer = kRecTile * kCols / kRecThreads;
    constexpr int kVec = 4 * (int)sizeof(T) <= 16 && (16 % (4 * (int)sizeof(T)) == 0) ? 4 : 1;
    const int c4 = 4 * lane;                          // this lane's first channel in the row passes
    float rq_[2][4], rk_[2][4], rz_[2][4], rv_[kVPer];
    float rb_ = 0.f;
    auto load4 = [&](const T* __restrict__ src, int n, float (&f)[4]) {
        // src[0 .. n) as floats, zeros past n (n <= 4); one vector load when all four are
        // present and the row is aligned for it
        if (n == 4 && (dk % 4) == 0 && kVec == 4) {
            if constexpr (sizeof(T) == 4) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(src));
                f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
            } else {
                const uint2 x = __ldg(reinterpret_cast<const uint2*>(src));
                const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
                const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
                f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = e < n ? to_f32(src[e]) : 0.f;
        }
    };
    auto fetch = [&](int64_t t0) {
        const int nt = (int)((eos - t0) < kRecTile ? (eos - t0) : kRecTile);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int tt = warp + 8 * i;
            const int n = tt < nt ? (dk - c4 < 0 ? 0 : (dk - c4 > 4 ? 4 : dk - c4)) : 0;
            const size_t e = ((size_t)(t0 + (tt < nt ? tt : 0)) * H + h) * dk + c4;
            load4(q + e, n, rq_[i]);
            load4(k + e, n, rk_[i]);
            load4(z + e, n, rz_[i]);
        }
#pragma unroll
        for (int i = 0; i < kVPer; ++i) {
            const int idx = tid + kRecThreads * i, tt = idx / kCols, j = col0 + idx % kCols;
            rv_[i] = (tt < nt && j < dv) ? to_f32(v[((size_t)(t0 + tt) * H + h) * dv + j]) : 0.f;
        }
        if (tid < kRecTile) rb_ = tid < nt ? to_f32(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    };
    if (bos < eos) fetch(bos);

    for (int64_t t0 = bos; t0 < eos; t0 += kRecTile) {
        const int nt = (int)((eos - t0) < kRecTile ? (eos - t0) : kRecTile);
        __syncthreads();   // previous tile fully consumed; s_expA visible
        // Warp w (tokens w, w + 8) keeps the raw k and q of channels 4 l .. 4 l + 3
        // in registers: g goes to s_kg, and k^T q is one warp sum per token.
        {
            const float4 ea = *reinterpret_cast<const float4*>(&s_expA[c4]);
            const float eav[4] = {ea.x, ea.y, ea.z, ea.w};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int tt = warp + 8 * i;
                float g[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) g[e] = (tt < nt && c4 + e < dk) ? gate_fast(eav[e], rz_[i][e]) : 0.f;
                *reinterpret_cast<float4*>(&s_kg[tt * kRecPitch + rec_idx(c4)]) = make_float4(g[0], g[1], g[2], g[3]);
                float p = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) p = fmaf(rk_[i][e], rq_[i][e], p);
                p = warp_sum(p);
                if (lane == 0) s_kq[tt] = p;
            }
#pragma unroll
            for (int i = 0; i < kVPer; ++i) {
                const int idx = tid + kRecThreads * i;
                s_v[idx / kCols][idx % kCols] = rv_[i];
            }
            if (tid < kRecTile) s_b[tid] = rb_;
        }
        __syncthreads();
        // The running log-decay inside each run of kRecRun tokens, per channel,
        // in place, and gam at each run's end (g = 0 past the tile's live tokens).
        if (tid < 128) {
#pragma unroll
            for (int run = 0; run < kRecTile / kRecRun; ++run) {
                float L = 0.f;
#pragma unroll
                for (int i = 0; i < kRecRun; ++i) {
                    const int ix = (run * kRecRun + i) * kRecPitch + rec_idx(tid);
                    L += s_kg[ix];
                    s_kg[ix] = L;
                }
                s_glast[run][rec_idx(tid)] = __expf(L);
            }
        }
        __syncthreads();
        // gam k (over L in place), gam q and k / gam for every (token, channel)
        {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int ix = (warp + 8 * i) * kRecPitch + rec_idx(c4);
                const float4 L = *reinterpret_cast<const float4*>(&s_kg[ix]);
                const float Lv[4] = {L.x, L.y, L.z, L.w};
                float kg[4], qg[4], kh[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float g = __expf(Lv[e]), ig = __expf(-Lv[e]);
                    kg[e] = g * rk_[i][e];
                    qg[e] = g * rq_[i][e];
                    kh[e] = ig * rk_[i][e];
                }
                *reinterpret_cast<float4*>(&s_kg[ix]) = make_float4(kg[0], kg[1], kg[2], kg[3]);
                *reinterpret_cast<float4*>(&s_qg[ix]) = make_float4(qg[0], qg[1], qg[2], qg[3]);
                *reinterpret_cast<float4*>(&s_kh[ix]) = make_float4(kh[0], kh[1], kh[2], kh[3]);
            }
        }
        __syncthreads();
        // the raw registers are free: the next tile's inputs load during the tokens
        if (t0 + kRecTile < eos) fetch(t0 + kRecTile);

        for (int tt = 0; tt < nt; ++tt) {
            const int base = tt * kRecPitch + rec_idx(r0);
            // S'^T k and S'^T q on this lane's 16 rows: row pairs on packed
            // FMAs, two accumulators per column and vector
            uint64_t pk[2][2] = {{0ull, 0ull}, {0ull, 0ull}}, pq[2][2] = {{0ull, 0ull}, {0ull, 0ull}};
#pragma unroll
            for (int x = 0; x < kPairs / 2; ++x) {
                const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&s_kg[base + 4 * x]);
                const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(&s_qg[base + 4 * x]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    pk[0][u] = f2_fma(st[2 * x][u], a.x, pk[0][u]);
                    pk[1][u] = f2_fma(st[2 * x + 1][u], a.y, pk[1][u]);
                    pq[0][u] = f2_fma(st[2 * x][u], b.x, pq[0][u]);
                    pq[1][u] = f2_fma(st[2 * x + 1][u], b.y, pq[1][u]);
                }
            }
            float sk[2], sq[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float2 k0 = f2_unpack(pk[0][u]), k1 = f2_unpack(pk[1][u]);
                const float2 q0 = f2_unpack(pq[0][u]), q1 = f2_unpack(pq[1][u]);
                sk[u] = (k0.x + k0.y) + (k1.x + k1.y);
                sq[u] = (q0.x + q0.y) + (q1.x + q1.y);
            }
#pragma unroll
            for (int m = kCq; m <= 16; m <<= 1) {
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    sk[u] += __shfl_xor_sync(0xffffffffu, sk[u], m);
                    sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], m);
                }
            }
            const float b = s_b[tt], kq = s_kq[tt];
            const float2 vv = *reinterpret_cast<const float2*>(&s_v[tt][lcol]);
            const float u0 = b * (vv.x - sk[0]), u1 = b * (vv.y - sk[1]);
            if (rq == 0)
                *reinterpret_cast<float2*>(&s_o[tt][lcol]) = make_float2(fmaf(u0, kq, sq[0]), fmaf(u1, kq, sq[1]));
            const uint64_t uu[2] = {f2_pack(u0, u0), f2_pack(u1, u1)};
#pragma unroll
            for (int x = 0; x < kPairs / 2; ++x) {
                const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&s_kh[base + 4 * x]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    st[2 * x][u] = f2_fma(a.x, uu[u], st[2 * x][u]);
                    st[2 * x + 1][u] = f2_fma(a.y, uu[u], st[2 * x + 1][u]);
                }
            }
            // end of a run: back from R to S
            if ((tt & (kRecRun - 1)) == kRecRun - 1 || tt == nt - 1) {
                const float* gl = &s_glast[tt / kRecRun][rec_idx(r0)];
#pragma unroll
                for (int x = 0; x < kPairs / 2; ++x) {
                    const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(gl + 4 * x);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        st[2 * x][u] = f2_mul(st[2 * x][u], a.x);
                        st[2 * x + 1][u] = f2_mul(st[2 * x + 1][u], a.y);
                    }
                }
            }
        }
        __syncthreads();
        for (int idx = tid; idx < nt * kCols; idx += kRecThreads) {
            const int tt = idx / kCols, jj = idx % kCols;
            const int j = col0 + jj;
            if (j < dv) o[((size_t)(t0 + tt) * H + h) * dv + j] = from_f32<T>(s_o[tt][jj]);
        }
        // Checkpoint: the state after every `ck.every` tokens of this sequence.
        const int64_t done = t0 + nt - bos;
        if (ck.out && done % ck.every == 0 && done / ck.every <= ck.max_count)
            store_state(ck.out + (((size_t)n * H + h) * ck.max_count + (done / ck.every - 1)) * dk * dv);
    }

    if (S1) store_state(S1 + sbase);
}

cudaError_t run_recurrent(const void* q, const void* k, const void* v, const void* z,
                          const void* beta, const float* A, void* o, const float* S0, float* S1,
                          const int32_t* cu, int n_seqs, int64_t T, int64_t T_total, int H,
                          int dk, int dv, bool bf16, const CheckpointSpec& ck,
                          cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // 32-column CTAs where 64-column ones would not cover the SMs
    const int64_t ctas64 = (int64_t)((dv + 63) / 64) * H * n_seqs;
    const bool narrow = ctas64 < sms;
    const int cols = narrow ? 32 : 64;
    dim3 grid((unsigned)((dv + cols - 1) / cols), (unsigned)H, (unsigned)n_seqs);
    const bool rows64 = dk <= 64;
    auto launch = [&](auto tag, auto cols_tag, auto rows_tag) {
        using TT = decltype(tag);
        constexpr int C = decltype(cols_tag)::value;
        constexpr int R = decltype(rows_tag)::value;
        recurrent_kernel<TT, C, R><<<grid, kRecThreads, 0, stream>>>(
            static_cast<const TT*>(q), static_cast<const TT*>(k), static_cast<const TT*>(v),
            static_cast<const TT*>(z), static_cast<const TT*>(beta), A, static_cast<TT*>(o), S0,
            S1, cu, T, T_total, H, dk, dv, ck);
    };
    using C32 = std::integral_constant<int, 32>;
    using C64 = std::integral_constant<int, 64>;
    using R64 = std::integral_constant<int, 64>;
    using R128 = std::integral_constant<int, 128>;
    auto by_rows = [&](auto tag, auto cols_tag) {
        if (rows64) launch(tag, cols_tag, R64{});
        else launch(tag, cols_tag, R128{});
    };
    if (bf16) {
        if (narrow) by_rows(__nv_bfloat16{}, C32{});
        else by_rows(__nv_bfloat16{}, C64{});
    } else {
        if (narrow) by_rows(float{}, C32{});
        else by_rows(float{}, C64{});
    }
    return cudaGetLastError();
}

}  // namespace kda
