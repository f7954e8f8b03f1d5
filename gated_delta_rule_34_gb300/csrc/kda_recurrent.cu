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
// so the work splits over (sequence, head, column group).  A CTA has two warp
// groups of eight warps.  The preparation group builds a tile of 16 tokens'
// per-row vectors (gates, the running log-decay, gam k, gam q, k / gam, k^T q,
// v, beta) into one of two shared-memory buffers while the token group runs
// the tokens of the previous tile from the other; two mbarriers per buffer
// hand tiles over (ready: built; freed: read), every wait bounded, and a group
// leaves its loop only on a decision all its threads share.  If a wait gives
// up, the outputs from that tile to the end of the sequence and the final
// state are NaN.
//
// Token group: kCols = 64 or 32 columns per CTA; warp w owns kCols / 8 of them,
// lane (rq = lane / kCq, cq = lane mod kCq, kCq = kCols / 16 column pairs)
// holds kDk / (32 / kCq) rows of columns kCols / 8 w + 2 cq, + 1 (row pairs on
// which packed two-lane FMAs run), so the d_k reductions are in-thread sums
// plus xor-shuffles over the row-group lane bits.  kDk = 64 when d_k <= 64.
// The 32-column form doubles the CTAs where 64-column ones would leave most
// SMs idle (narrow heads, few sequences).  The per-row vectors sit in rows
// whose 16-channel groups are 20 floats apart, so the row groups of a warp
// read them as conflict-free 16-byte loads.
#include <type_traits>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {

constexpr int kRecGroup = 256;   // threads per warp group
constexpr int kRecTile = 16;     // tokens per tile
constexpr int kRecRun = 8;       // tokens per factoring run (gam >= e^{-5 kRecRun})
constexpr int kRecPitch = 160;   // floats per token row of the scaled vectors: 8 groups of 16 + 4
constexpr uint32_t kBarRecPrep = 1, kBarRecTok = 2;   // named barriers of the two groups

__device__ __forceinline__ int rec_idx(int c) { return (c >> 4) * 20 + (c & 15); }

// Dynamic shared memory; buffer b holds one tile's vectors.
struct RecSmem {
    float kg[2][kRecTile * kRecPitch];   // g, then the running log-decay L, then gam k
    float qg[2][kRecTile * kRecPitch];
    float kh[2][kRecTile * kRecPitch];
    float glast[2][kRecTile / kRecRun][kRecPitch];   // gam at each run's end
    float v[2][kRecTile][64];
    float o[kRecTile][64];                            // token group only
    float b[2][kRecTile];
    float kq[2][kRecTile];
    float expA[128];
    unsigned long long bar[4];                        // ready[2], freed[2]
};

// Barrier over one warp group that also returns whether every thread of the
// group passed ok.
__device__ __forceinline__ bool rec_group_and(uint32_t id, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "n"(kRecGroup)
        : "memory");
    return r != 0;
}

template <typename T, int kCols, int kDk>
__global__ void __launch_bounds__(2 * kRecGroup, 1)
recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const T* __restrict__ z, const T* __restrict__ beta,
                 const float* __restrict__ A, T* __restrict__ o,
                 const float* __restrict__ S0, float* __restrict__ S1,
                 const int32_t* __restrict__ cu, int64_t T_len, int64_t T_total, int H,
                 int dk, int dv, CheckpointSpec ck) {
    static_assert(kCols == 64 || kCols == 32, "column group");
    static_assert(kDk == 128 || kDk == 64, "rows held");
    const int cgrp = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int tid = threadIdx.x;
    const bool prep = tid < kRecGroup;
    const int gtid = tid & (kRecGroup - 1), warp = gtid >> 5, lane = tid & 31;
    const int col0 = cgrp * kCols;                    // first column of this CTA
    extern __shared__ __align__(16) unsigned char rec_smem_raw[];
    RecSmem& sm = *reinterpret_cast<RecSmem*>(rec_smem_raw);
    uint64_t* ready = reinterpret_cast<uint64_t*>(sm.bar);
    uint64_t* freed = ready + 2;

    int64_t bos, eos;
    seq_bounds(cu, n, T_len, T_total, bos, eos);
    const int64_t n_tiles = (eos - bos + kRecTile - 1) / kRecTile;

    if (tid == 0) {
        for (int p = 0; p < 2; ++p) {
            tc::mbar_init(ready + p, 1);
            tc::mbar_init(freed + p, 1);
        }
        tc::fence_mbar_init();
    }
    if (tid < 128) sm.expA[tid] = tid < dk ? expf(A[(size_t)h * dk + tid]) : 0.f;
    __syncthreads();   // the one barrier over both groups: mbarriers and e^A ready

    if (prep) {
        // ============================================== preparation group
        // A tile's raw inputs, loaded into registers one tile ahead: warp w
        // takes tokens w and w + 8, lane l channels 4 l .. 4 l + 3 of q, k, z
        // (one 16-byte load each for fp32, 8 bytes for bf16, where the rows
        // allow); (tt, column) pairs idx = gtid + 256 i for v; beta by gtid < 16.
        constexpr int kVPer = kRecTile * kCols / kRecGroup;
        const int c4 = 4 * lane;
        float rq_[2][4], rk_[2][4], rz_[2][4], rv_[kVPer];
        float rb_ = 0.f;
        auto load4 = [&](const T* __restrict__ src, int cnt, float (&f)[4]) {
            // src[0 .. cnt) as floats, zeros past cnt (cnt <= 4); one vector load
            // when all four are present and the row is aligned for it
            if (cnt == 4 && (dk % 4) == 0) {
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
                for (int e = 0; e < 4; ++e) f[e] = e < cnt ? to_f32(src[e]) : 0.f;
            }
        };
        auto fetch = [&](int64_t t0) {
            const int nt = (int)((eos - t0) < kRecTile ? (eos - t0) : kRecTile);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int tt = warp + 8 * i;
                const int cnt = tt < nt ? (dk - c4 < 0 ? 0 : (dk - c4 > 4 ? 4 : dk - c4)) : 0;
                const size_t e = ((size_t)(t0 + (tt < nt ? tt : 0)) * H + h) * dk + c4;
                load4(q + e, cnt, rq_[i]);
                load4(k + e, cnt, rk_[i]);
                load4(z + e, cnt, rz_[i]);
            }
#pragma unroll
            for (int i = 0; i < kVPer; ++i) {
                const int idx = gtid + kRecGroup * i, tt = idx / kCols, j = col0 + idx % kCols;
                rv_[i] = (tt < nt && j < dv) ? to_f32(v[((size_t)(t0 + tt) * H + h) * dv + j]) : 0.f;
            }
            if (gtid < kRecTile) rb_ = gtid < nt ? to_f32(beta[(size_t)(t0 + gtid) * H + h]) : 0.f;
        };
        if (n_tiles > 0) fetch(bos);
        const float4 ea = *reinterpret_cast<const float4*>(&sm.expA[c4]);
        const float eav[4] = {ea.x, ea.y, ea.z, ea.w};

        for (int64_t i = 0; i < n_tiles; ++i) {
            const int p = (int)(i & 1);
            const int64_t t0 = bos + i * kRecTile;
            const int nt = (int)((eos - t0) < kRecTile ? (eos - t0) : kRecTile);
            // buffer p was last read by the tokens of tile i - 2
            if (i >= 2 && !rec_group_and(kBarRecPrep, tc::mbar_wait(freed + p, (uint32_t)(((i - 2) >> 1) & 1))))
                break;
            float* kg = sm.kg[p];
            float* qg = sm.qg[p];
            float* kh = sm.kh[p];
            // g into kg (0 past the live tokens and past d_k), k^T q one warp sum per token, v, beta
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int tt = warp + 8 * ii;
                float g[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) g[e] = (tt < nt && c4 + e < dk) ? gate_fast(eav[e], rz_[ii][e]) : 0.f;
                *reinterpret_cast<float4*>(&kg[tt * kRecPitch + rec_idx(c4)]) = make_float4(g[0], g[1], g[2], g[3]);
                float pp = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) pp = fmaf(rk_[ii][e], rq_[ii][e], pp);
                pp = warp_sum(pp);
                if (lane == 0) sm.kq[p][tt] = pp;
            }
#pragma unroll
            for (int ii = 0; ii < kVPer; ++ii) {
                const int idx = gtid + kRecGroup * ii;
                sm.v[p][idx / kCols][idx % kCols] = rv_[ii];
            }
            if (gtid < kRecTile) sm.b[p][gtid] = rb_;
            tc::named_bar_sync(kBarRecPrep, kRecGroup);
            // the running log-decay inside each run of kRecRun tokens, per channel,
            // in place, and gam at each run's end
            if (gtid < 128) {
#pragma unroll
                for (int run = 0; run < kRecTile / kRecRun; ++run) {
                    float L = 0.f;
#pragma unroll
                    for (int t = 0; t < kRecRun; ++t) {
                        const int ix = (run * kRecRun + t) * kRecPitch + rec_idx(gtid);
                        L += kg[ix];
                        kg[ix] = L;
                    }
                    sm.glast[p][run][rec_idx(gtid)] = __expf(L);
                }
            }
            tc::named_bar_sync(kBarRecPrep, kRecGroup);
            // gam k (over L in place), gam q and k / gam for every (token, channel)
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const int ix = (warp + 8 * ii) * kRecPitch + rec_idx(c4);
                const float4 L = *reinterpret_cast<const float4*>(&kg[ix]);
                const float Lv[4] = {L.x, L.y, L.z, L.w};
                float a[4], bq[4], c[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float gm = __expf(Lv[e]), ig = __expf(-Lv[e]);
                    a[e] = gm * rk_[ii][e];
                    bq[e] = gm * rq_[ii][e];
                    c[e] = ig * rk_[ii][e];
                }
                *reinterpret_cast<float4*>(&kg[ix]) = make_float4(a[0], a[1], a[2], a[3]);
                *reinterpret_cast<float4*>(&qg[ix]) = make_float4(bq[0], bq[1], bq[2], bq[3]);
                *reinterpret_cast<float4*>(&kh[ix]) = make_float4(c[0], c[1], c[2], c[3]);
            }
            // the raw registers are free: the next tile's inputs load now
            if (i + 1 < n_tiles) fetch(t0 + kRecTile);
            tc::named_bar_sync(kBarRecPrep, kRecGroup);
            if (gtid == 0) tc::mbar_arrive(ready + p);
        }
    } else {
        // ===================================================== token group
        constexpr int kCq = kCols / 16;               // column pairs per warp (lanes along columns)
        constexpr int kRows = kDk / (32 / kCq);       // rows per lane
        constexpr int kPairs = kRows / 2;             // row pairs per lane
        const int rq = lane / kCq, cq = lane % kCq;
        const int lcol = (kCols / 8) * warp + 2 * cq; // this lane's first column, CTA-local
        const int r0 = kRows * rq;                    // this lane's first row
        const int rb = rec_idx(r0);                   // its rows in the per-row vectors

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
                const float* sp = S0 ? S0 + sbase + (size_t)r * dv + col0 + lcol + u : nullptr;
                st[p2][u] = f2_pack((sp && r < dk && okc[u]) ? sp[0] : 0.f,
                                    (sp && r + 1 < dk && okc[u]) ? sp[dv] : 0.f);
            }
        }
        auto store_state = [&](float* mat, bool nan) {      // mat: [d_k][d_v] of (n, h)
#pragma unroll
            for (int p2 = 0; p2 < kPairs; ++p2) {
                const int r = r0 + 2 * p2;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float2 x = f2_unpack(st[p2][u]);
                    if (nan) x = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
                    float* mp = mat + (size_t)r * dv + col0 + lcol + u;
                    if (okc[u] && r < dk) mp[0] = x.x;
                    if (okc[u] && r + 1 < dk) mp[dv] = x.y;
                }
            }
        };

        bool ok = true;
        int64_t i = 0;
        for (; i < n_tiles; ++i) {
            const int p = (int)(i & 1);
            const int64_t t0 = bos + i * kRecTile;
            const int nt = (int)((eos - t0) < kRecTile ? (eos - t0) : kRecTile);
            ok = rec_group_and(kBarRecTok, tc::mbar_wait(ready + p, (uint32_t)((i >> 1) & 1)));
            if (!ok) break;
            const float* kg = sm.kg[p];
            const float* qg = sm.qg[p];
            const float* kh = sm.kh[p];
            for (int tt = 0; tt < nt; ++tt) {
                const int base = tt * kRecPitch + rb;
                // S'^T k and S'^T q on this lane's rows: row pairs on packed
                // FMAs, two accumulators per column and vector
                uint64_t pk[2][2] = {{0ull, 0ull}, {0ull, 0ull}}, pq[2][2] = {{0ull, 0ull}, {0ull, 0ull}};
#pragma unroll
                for (int x = 0; x < kPairs / 2; ++x) {
                    const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&kg[base + 4 * x]);
                    const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(&qg[base + 4 * x]);
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
                const float bt = sm.b[p][tt], kq = sm.kq[p][tt];
                const float2 vv = *reinterpret_cast<const float2*>(&sm.v[p][tt][lcol]);
                const float u0 = bt * (vv.x - sk[0]), u1 = bt * (vv.y - sk[1]);
                if (rq == 0)
                    *reinterpret_cast<float2*>(&sm.o[tt][lcol]) = make_float2(fmaf(u0, kq, sq[0]), fmaf(u1, kq, sq[1]));
                const uint64_t uu[2] = {f2_pack(u0, u0), f2_pack(u1, u1)};
#pragma unroll
                for (int x = 0; x < kPairs / 2; ++x) {
                    const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(&kh[base + 4 * x]);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        st[2 * x][u] = f2_fma(a.x, uu[u], st[2 * x][u]);
                        st[2 * x + 1][u] = f2_fma(a.y, uu[u], st[2 * x + 1][u]);
                    }
                }
                // end of a run: back from R to S
                if ((tt & (kRecRun - 1)) == kRecRun - 1 || tt == nt - 1) {
                    const float* gl = &sm.glast[p][tt / kRecRun][rb];
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
            // the tile's outputs are in o and its buffer has been read
            tc::named_bar_sync(kBarRecTok, kRecGroup);
            if (gtid == 0) tc::mbar_arrive(freed + p);
            for (int idx = gtid; idx < nt * kCols; idx += kRecGroup) {
                const int tt = idx / kCols, jj = idx % kCols;
                const int j = col0 + jj;
                if (j < dv) o[((size_t)(t0 + tt) * H + h) * dv + j] = from_f32<T>(sm.o[tt][jj]);
            }
            // Checkpoint: the state after every `ck.every` tokens of this sequence.
            const int64_t done = t0 + nt - bos;
            if (ck.out && done % ck.every == 0 && done / ck.every <= ck.max_count)
                store_state(ck.out + (((size_t)n * H + h) * ck.max_count + (done / ck.every - 1)) * dk * dv, false);
            // o has been read before the next tile's tokens write it
            tc::named_bar_sync(kBarRecTok, kRecGroup);
        }
        if (!ok) {
            // A wait gave up: NaN from this tile to the end of the sequence.
            const T nanv = from_f32<T>(__int_as_float(0x7fc00000));
            const int64_t t_first = bos + i * kRecTile;
            for (int64_t idx = gtid; idx < (eos - t_first) * kCols; idx += kRecGroup) {
                const int64_t tt = idx / kCols;
                const int j = col0 + (int)(idx % kCols);
                if (j < dv) o[((size_t)(t_first + tt) * H + h) * dv + j] = nanv;
            }
        }
        if (S1) store_state(S1 + sbase, !ok);
    }
}

template <typename TT, int C, int R>
cudaError_t launch_recurrent(dim3 grid, cudaStream_t stream, const void* q, const void* k,
                             const void* v, const void* z, const void* beta, const float* A,
                             void* o, const float* S0, float* S1, const int32_t* cu, int64_t T,
                             int64_t T_total, int H, int dk, int dv, const CheckpointSpec& ck) {
    constexpr int kMaxDevices = 64;
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(recurrent_kernel<TT, C, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(RecSmem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    recurrent_kernel<TT, C, R><<<grid, 2 * kRecGroup, sizeof(RecSmem), stream>>>(
        static_cast<const TT*>(q), static_cast<const TT*>(k), static_cast<const TT*>(v),
        static_cast<const TT*>(z), static_cast<const TT*>(beta), A, static_cast<TT*>(o), S0, S1,
        cu, T, T_total, H, dk, dv, ck);
    return cudaGetLastError();
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
    const bool rows64 = dk <= 64;
    dim3 grid((unsigned)((dv + cols - 1) / cols), (unsigned)H, (unsigned)n_seqs);
#define KDA_REC_LAUNCH(TT, C, R) \
    launch_recurrent<TT, C, R>(grid, stream, q, k, v, z, beta, A, o, S0, S1, cu, T, T_total, H, dk, dv, ck)
    if (bf16) {
        using Tb = __nv_bfloat16;
        if (narrow) return rows64 ? KDA_REC_LAUNCH(Tb, 32, 64) : KDA_REC_LAUNCH(Tb, 32, 128);
        return rows64 ? KDA_REC_LAUNCH(Tb, 64, 64) : KDA_REC_LAUNCH(Tb, 64, 128);
    }
    if (narrow) return rows64 ? KDA_REC_LAUNCH(float, 32, 64) : KDA_REC_LAUNCH(float, 32, 128);
    return rows64 ? KDA_REC_LAUNCH(float, 64, 64) : KDA_REC_LAUNCH(float, 64, 128);
#undef KDA_REC_LAUNCH
}

}  // namespace kda
