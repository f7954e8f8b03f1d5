// kda_chunk16_tc.cu -- chunked KDA prefill with 16-token chunks on the sm_103a
// tensor cores (bf16 inputs; d_k and d_v multiples of 16, at most 128).
//
// The chunked form over 16-token chunks: inside a chunk the tokens are handled
// together by tensor-core products, and the state is passed from chunk to
// chunk ("Kimi K3 architecture: how an open model with a million-token context
// competes with market leaders", section "Chip level: the specialised FlashKDA
// kernel").  With g_min = -5 ("How Kimi K3 is built: 2.8 trillion parameters,
// linear attention and agents for a million tokens", section "Sequence: three
// KDA to one global MLA") the log-decay across 16 tokens spans at most 80, so
// e^{+-L} fits in fp32 and bf16 and every causal block is one dense product:
// there is no separate path for the diagonal.
//
// Per (sequence, head) and chunk of C <= 16 tokens, with L_t = running sum of
// g from the chunk start (L_t in [-80, 0]), E_t = e^{L_t}, lam = e^{L_{C-1}},
// the start state S and beta already folded where written:
//   A_ts = b_t sum_c k_tc E_tc k_sc / E_sc  (s < t)     T = (I + A)^{-1}
//   P_ts =     sum_c q_tc E_tc k_sc / E_sc  (s <= t)
//   W = T Diag(b) (k E),  U~ = T Diag(b) V,  U = U~ - W S
//   O = (q E) S + P U,    S <- Diag(lam) S + (k lam / E)^T U
// which is the recurrence unrolled over the chunk (the same algebra as the
// 64-token path, without its cross-block factoring).
//
// One CTA of sixteen warps per (sequence, head) walks the chunks in order, in
// two warp groups: the preparation group (warps 0-7) builds, for the next
// chunk, everything that does not depend on the state (gate, scan, operands,
// A/P, the solve, W and U~), while the chain group (warps 8-15) runs the
// current chunk's state products and update.  They hand chunks over through
// double-buffered operands and two mbarriers (ready: prepared; freed: the
// chain has consumed the buffers).  All products are arranged so that TMEM
// lane = state column j (or channel c), so the fp32 state lives in registers
// as S^T[j][c] (thread = lane j, one half of the channels per warp quartet)
// and its bf16 copy is written row by row:
//   A/P    D[t][s]   = [kE ; qE] (k/E)^T           M=64  N=16  K=128
//   W^T    D[c][t]   = (b kE)^T T^T                M=128 N=16  K=16   (A MN-major)
//   U~^T   D[j][t]   = (b V)^T T^T                 M=128 N=16  K=16   (A MN-major)
//   S^T W^T, S^T (qE)^T  D[j][t] = S^T [W ; qE]^T  M=128 N=32  K=128
//   O^T   += U^T P^T                               M=128 N=16  K=16
//   D[j][c] = U^T (k lam / E)                      M=128 N=128 K=16   (B MN-major)
// and the fp32 update S^T <- S^T Diag(lam) + D on the registers.  The path
// needs no workspace beyond the status word.
#include <cuda.h>
#include <string.h>
#include <cuda_bf16.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace c16 {

using namespace tc;

constexpr int kC = 16;
constexpr int kThreads = 512;
constexpr int kGroup = 256;             // threads per warp group
constexpr uint32_t kBarPrep = 1, kBarChain = 2;   // named barriers of the two groups

// shared memory (offsets from a 1024-byte aligned base); [P] preparation group
// only, [C] chain group only, [P->C] double-buffered hand-over (buffer ci & 1)
constexpr uint32_t R_ST = 0;          // [C] S^T bf16 [128 j][128 c]: two K-blocks of 16 KB, swizzled
constexpr uint32_t R_UT = 32768;      // [C] U^T bf16 [128 j][16 t] (128-byte rows, K = 16 used)
constexpr uint32_t R_APA = 49152;     // [P] [kE ; qE ; 0] [64 rows][128 c]: two K-blocks of 8 KB
constexpr uint32_t R_APB = 65536;     // [P] k/E [16 s][128 c]: two K-blocks of 2 KB
constexpr uint32_t R_SB = 69632;      // [P->C] [W ; qE] [32 rows][128 c]: two K-blocks of 4 KB; x2
constexpr uint32_t R_BKG = 86016;     // [P] b kE token rows, two 64-channel halves of 2 KB (MN-major)
constexpr uint32_t R_BV = 90112;      // [P] b V token rows, same layout
constexpr uint32_t R_KC = 94208;      // [P->C] k lam / E token rows, same layout; x2
constexpr uint32_t R_PB = 102400;     // [P->C] P [16 t][16 s] (128-byte rows); x2
constexpr uint32_t R_TB = 106496;     // [P] T [16 t][16 s] (128-byte rows)
constexpr uint32_t R_GS = 108544;     // [P] g, then L: fp32 [16 t][128 c]
constexpr uint32_t R_AF = 116736;     // [P] A fp32 [16][17]
constexpr uint32_t R_LAM = 118016;    // [P->C] lam [128] fp32; x2
constexpr uint32_t R_EA = 119040;     // [P] e^{A_h} [128] fp32
constexpr uint32_t R_BETA = 119552;   // [P] beta [16] fp32
constexpr uint32_t R_IN = 120832;     // [P] input tiles z, k, q, v of a chunk, 4 KB each (256-byte
                                      //     token rows, as the tensor maps land them); two stages
constexpr uint32_t IN_STAGE = 16384;
constexpr uint32_t R_BAR = R_IN + 2 * IN_STAGE;   // mbarriers (prep MMA, chain MMA, ready x2,
                                                  // freed x2, inputs x2), TMEM slot
constexpr uint32_t SMEM = R_BAR + 128 + 1024;   // + slack for aligning the base
static_assert(SMEM <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t T_AP = 0;      // [P] A/P (M=64 layout: row r in lane 32 (r / 16) + r mod 16)
constexpr uint32_t T_WT = 16;     // [P] W^T
constexpr uint32_t T_UT = 32;     // [P->C] U~^T, two buffers of 16
constexpr uint32_t T_ST = 64;     // [C] [(W S)^T | O^T]
constexpr uint32_t T_SU = 128;    // [C] U^T (k lam / E)
constexpr uint32_t kTmemCols = 256;

constexpr uint32_t kErrWait = 8u;   // status bit: a bounded wait gave up

__device__ __forceinline__ uint32_t idesc_bmn(uint32_t M, uint32_t N) {
    return idesc_bf16(M, N) | (1u << 16);   // B MN-major
}

// Barrier over one warp group (named barrier `id`, kGroup threads) that also
// returns whether every thread of the group passed ok.
__device__ __forceinline__ bool group_and(uint32_t id, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "n"(kGroup)
        : "memory");
    return r != 0;
}

// Bounded wait for the phase of `bar` with the given parity, agreed on by the
// whole warp group.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, uint32_t id) {
    const bool ok = mbar_wait(bar, parity);
    tc_fence_after();
    return group_and(id, ok);
}

// Stores 8 bf16 values (channels 8 c8 .. 8 c8 + 7) as token row t of a [rows][128]
// K-major operand split in two 64-channel K-blocks `kb_bytes` apart.
__device__ __forceinline__ void store_row8(uint8_t* base, uint32_t kb_bytes, int row, int c8,
                                           const float (&f)[8]) {
    uint4 r;
    r.x = pack_bf16x2(f[0], f[1]);
    r.y = pack_bf16x2(f[2], f[3]);
    r.z = pack_bf16x2(f[4], f[5]);
    r.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(base + (c8 >> 3) * kb_bytes + sw128(row, c8 & 7)) = r;
}

__device__ __forceinline__ void unpack8(uint4 raw, float (&f)[8]) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(b[e]);
}

// 8 consecutive floats from 16-byte aligned shared memory.
__device__ __forceinline__ void load8f(const float* p, float (&f)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Tensor maps of the inputs [T_total][H][d] with boxes of 16 tokens x 1 head x
// 128 channels (4 KB): a chunk's tile of each input is one TMA load.
struct InputMaps16 {
    CUtensorMap q, k, v, z;
};

__global__ void __launch_bounds__(kThreads, 1)
chunk16_kernel(const __grid_constant__ InputMaps16 maps, const __nv_bfloat16* __restrict__ beta,
               const float* __restrict__ A,
               __nv_bfloat16* __restrict__ o, const float* __restrict__ S0, float* __restrict__ S1,
               const int32_t* __restrict__ cu, int64_t T_len, int64_t T_total, int H, int dk, int dv,
               uint32_t* __restrict__ status, CheckpointSpec ck) {
    const int n = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* gs = reinterpret_cast<float*>(sm + R_GS);
    float* af = reinterpret_cast<float*>(sm + R_AF);
    float* ea = reinterpret_cast<float*>(sm + R_EA);
    float* bs = reinterpret_cast<float*>(sm + R_BETA);
    uint64_t* bar_p = reinterpret_cast<uint64_t*>(sm + R_BAR);
    uint64_t* bar_c = bar_p + 1;
    uint64_t* ready = bar_p + 2;     // [2]
    uint64_t* freed = bar_p + 4;     // [2]
    uint64_t* inb = bar_p + 6;       // [2] input tiles of chunk ci in stage ci & 1 landed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + R_BAR + 64);

    int64_t bos, eos;
    seq_bounds(cu, n, T_len, T_total, bos, eos);
    const int64_t len_seq = eos - bos;
    const int nchunks = (int)((len_seq + kC - 1) / kC);
    const bool prep = tid < kGroup;
    const uint32_t tl = (uint32_t)(32 * (warp & 3)) << 16;   // TMEM lane field of this warp

    if (warp == 0) tmem_alloc<kTmemCols>(tslot);
    if (tid == 32) {
        mbar_init(bar_p, 1);
        mbar_init(bar_c, 1);
        for (int p = 0; p < 2; ++p) {
            mbar_init(ready + p, 1);
            mbar_init(freed + p, 1);
            mbar_init(inb + p, 1);
        }
        fence_mbar_init();
    }
    // Rows 32..63 of the A/P operand stay zero; e^A of the head.
    for (int i = tid; i < 4096; i += kThreads)
        reinterpret_cast<uint32_t*>(sm + R_APA)[i] = 0u;
    if (tid < 128) ea[tid] = tid < dk ? __expf(A[(size_t)h * dk + tid]) : 0.f;

    // Chain group: lane j = 32 (warp mod 4) + lane, channel half ch; it holds
    // S^T[j][64 ch .. 64 ch + 63] in fp32 registers.
    const int cw = warp - 8;
    const int j = 32 * (warp & 3) + lane, ch = (cw >> 2) & 1;
    const size_t smat = ((size_t)n * H + h) * dk * dv;
    float st[64];
    auto write_st = [&]() {
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            uint4 r;
            r.x = pack_bf16x2(st[8 * q8 + 0], st[8 * q8 + 1]);
            r.y = pack_bf16x2(st[8 * q8 + 2], st[8 * q8 + 3]);
            r.z = pack_bf16x2(st[8 * q8 + 4], st[8 * q8 + 5]);
            r.w = pack_bf16x2(st[8 * q8 + 6], st[8 * q8 + 7]);
            *reinterpret_cast<uint4*>(sm + R_ST + ch * 16384 + sw128(j, q8)) = r;
        }
    };
    auto store_state = [&](float* mat) {      // mat: [d_k][d_v] of (n, h)
        if (j < dv) {
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const int c = 64 * ch + e;
                if (c < dk) mat[(size_t)c * dv + j] = st[e];
            }
        }
    };
    if (!prep) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            const int c = 64 * ch + e;
            st[e] = (S0 && c < dk && j < dv) ? __ldg(S0 + smat + (size_t)c * dv + j) : 0.f;
        }
        write_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (prep) {
        // ============================================ preparation group
        const int tt = tid >> 4, c8 = tid & 15;   // token tt, channels 8 c8 .. + 7
        uint32_t phase = 0;
        // The input tiles of chunk ci land in stage ci & 1 by TMA, requested two
        // chunks ahead by thread 0 (tokens past the sequence belong to the next
        // one or read as zeros; `live` masks them).  beta is loaded one chunk
        // ahead as raw bits and converted where it is used.
        auto issue_inputs = [&](int ci) {
            const int64_t t0 = bos + (int64_t)ci * kC;
            uint8_t* in = sm + R_IN + (ci & 1) * IN_STAGE;
            uint64_t* bar = inb + (ci & 1);
            mbar_expect_tx(bar, IN_STAGE);
            tma_load_3d(in, &maps.z, 0, h, (int)t0, bar);
            tma_load_3d(in + 4096, &maps.k, 0, h, (int)t0, bar);
            tma_load_3d(in + 8192, &maps.q, 0, h, (int)t0, bar);
            tma_load_3d(in + 12288, &maps.v, 0, h, (int)t0, bar);
        };
        auto load_beta_bits = [&](int ci) -> uint32_t {
            const int64_t t0 = bos + (int64_t)ci * kC;
            return (tid < kC && ci < nchunks && t0 + tid < eos)
                       ? reinterpret_cast<const unsigned short*>(beta)[(size_t)(t0 + tid) * H + h]
                       : 0u;
        };
        int issued = 0, landed = 0;               // input requests (thread 0) and completed waits
        if (tid == 0)
            for (; issued < 2 && issued < nchunks; ++issued) issue_inputs(issued);
        uint32_t braw = load_beta_bits(0);
        for (int ci = 0; ci < nchunks; ++ci) {
            const int p = ci & 1;
            const int64_t t0 = bos + (int64_t)ci * kC;
            const int len = (int)((eos - t0) < kC ? (eos - t0) : kC);
            const bool live = tt < len;
            uint8_t* sb = sm + R_SB + p * 8192;
            uint8_t* kc = sm + R_KC + p * 4096;
            uint8_t* pb = sm + R_PB + p * 2048;
            float* lam = reinterpret_cast<float*>(sm + R_LAM + p * 512);
            const uint8_t* in = sm + R_IN + p * IN_STAGE;
            // buffers p were last used for chunk ci - 2
            if (ci >= 2 && !(ok = group_wait(freed + p, ((ci - 2) >> 1) & 1, kBarPrep))) break;
            if (!(ok = group_wait(inb + p, (ci >> 1) & 1, kBarPrep))) break;
            ++landed;
            const uint4 zr = live ? *reinterpret_cast<const uint4*>(in + tt * 256 + c8 * 16) : make_uint4(0, 0, 0, 0);
            const float bnext = __uint_as_float(braw << 16);
            braw = load_beta_bits(ci + 1);

            // ---- gate -> gs (zeros past the chunk and past d_k)
            {
                float zf[8], g[8], eav[8];
                unpack8(zr, zf);
                load8f(ea + 8 * c8, eav);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = 8 * c8 + e;
                    g[e] = (live && c < dk) ? gate_fast(eav[e], zf[e]) : 0.f;
                }
                float4* gp = reinterpret_cast<float4*>(gs + tt * 128 + 8 * c8);
                gp[0] = make_float4(g[0], g[1], g[2], g[3]);
                gp[1] = make_float4(g[4], g[5], g[6], g[7]);
                if (tid < kC) bs[tid] = bnext;
            }
            named_bar_sync(kBarPrep, kGroup);
            // ---- L = running sum over the chunk, per channel; lam = e^{L_last}
            if (tid < 128) {
                float run = 0.f;
#pragma unroll
                for (int t = 0; t < kC; ++t) {
                    run += gs[t * 128 + tid];
                    gs[t * 128 + tid] = run;
                }
                lam[tid] = __expf(run);
            }
            named_bar_sync(kBarPrep, kGroup);

            // ---- decay-scaled operands of token tt (bf16)
            {
                float kf[8], qf[8], vf[8], E[8], R[8], o8[8];
                const uint4 zero = make_uint4(0, 0, 0, 0);
                unpack8(live ? *reinterpret_cast<const uint4*>(in + 4096 + tt * 256 + c8 * 16) : zero, kf);
                unpack8(live ? *reinterpret_cast<const uint4*>(in + 8192 + tt * 256 + c8 * 16) : zero, qf);
                unpack8(live ? *reinterpret_cast<const uint4*>(in + 12288 + tt * 256 + c8 * 16) : zero, vf);
                const float4* lp = reinterpret_cast<const float4*>(gs + tt * 128 + 8 * c8);
                const float4 l0 = lp[0], l1 = lp[1];
                const float L[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    E[e] = __expf(L[e]);
                    R[e] = __fdividef(1.0f, E[e]);
                }
                const float bt = bs[tt];
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = kf[e] * E[e];
                store_row8(sm + R_APA, 8192, tt, c8, o8);                           // k E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = bt * o8[e];
                store_row8(sm + R_BKG, 2048, tt, c8, o8);                           // b k E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[e];
                store_row8(sm + R_APA, 8192, 16 + tt, c8, o8);                      // q E
                store_row8(sb, 4096, 16 + tt, c8, o8);
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = kf[e] * R[e];
                store_row8(sm + R_APB, 2048, tt, c8, o8);                           // k / E
                float lv[8];
                load8f(lam + 8 * c8, lv);
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = o8[e] * lv[e];
                store_row8(kc, 2048, tt, c8, o8);                                   // k lam / E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = bt * vf[e];
                store_row8(sm + R_BV, 2048, tt, c8, o8);                            // b V
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(kBarPrep, kGroup);
            tc_fence_after();
            // Stage p has been read: it takes chunk ci + 2's inputs.
            if (tid == 0 && issued < nchunks) issue_inputs(issued++);

            // ---- A and P: D[t][s] = [kE ; qE] (k/E)^T, M=64 N=16 K=128
            if (tid == 0) {
                const uint32_t idesc = idesc_bf16(64, 16);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + T_AP, desc_sw128(smem_u32(sm + R_APA + kb * 8192 + off)),
                             desc_sw128(smem_u32(sm + R_APB + kb * 2048 + off)), idesc, ks > 0);
                }
                mma_commit(bar_p);
            }
            ok = group_wait(bar_p, phase, kBarPrep);
            phase ^= 1u;
            if (!ok) break;
            // rows 0..15 (A, lanes 0..15 of warp 0), rows 16..31 (P, lanes 32..47 of warp 1)
            if (warp < 2) {
                float d[16];
                tmem_ld16(tbase + tl + T_AP, d);
                tmem_wait_ld();
                if (lane < kC) {
                    const int t = lane;
                    if (warp == 0) {
                        const float bt = bs[t];
#pragma unroll
                        for (int s2 = 0; s2 < kC; ++s2) af[t * 17 + s2] = s2 < t ? bt * d[s2] : 0.f;
                    } else {
                        float p8[8];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) p8[e] = (8 * hh + e <= t) ? d[8 * hh + e] : 0.f;
                            uint4 r;
                            r.x = pack_bf16x2(p8[0], p8[1]);
                            r.y = pack_bf16x2(p8[2], p8[3]);
                            r.z = pack_bf16x2(p8[4], p8[5]);
                            r.w = pack_bf16x2(p8[6], p8[7]);
                            *reinterpret_cast<uint4*>(pb + sw128(t, hh)) = r;
                        }
                    }
                }
            }
            tc_fence_before();
            named_bar_sync(kBarPrep, kGroup);

            // ---- T = (I + A)^{-1}: column jc by forward substitution (16 threads)
            if (tid < kC) {
                const int jc = tid;
                float x[kC];
#pragma unroll
                for (int r = 0; r < kC; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) acc = fmaf(af[r * 17 + m], x[m], acc);
                    x[r] = (r < jc) ? 0.f : (r == jc ? 1.f : -acc);
                }
#pragma unroll
                for (int r = 0; r < kC; ++r)
                    *reinterpret_cast<__nv_bfloat16*>(sm + R_TB + sw128(r, jc >> 3) + (jc & 7) * 2) =
                        __float2bfloat16_rn(x[r]);
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(kBarPrep, kGroup);
            tc_fence_after();

            // ---- W^T = (b kE)^T T^T and U~^T = (b V)^T T^T (M=128 N=16 K=16, A MN-major)
            if (tid == 0) {
                const uint32_t idesc = idesc_bf16_amn(128, 16);
                const uint64_t tb = desc_sw128(smem_u32(sm + R_TB));
                mma_bf16(tbase + T_WT, desc_sw128_mn(smem_u32(sm + R_BKG), 2048, 1024), tb, idesc, false);
                mma_bf16(tbase + T_UT + 16 * p, desc_sw128_mn(smem_u32(sm + R_BV), 2048, 1024), tb, idesc,
                         false);
                mma_commit(bar_p);
            }
            ok = group_wait(bar_p, phase, kBarPrep);
            phase ^= 1u;
            if (!ok) break;
            // W rows t of the [W ; qE] operand: lane c of warps 0..3 writes column c
            if (warp < 4) {
                float w[16];
                tmem_ld16(tbase + tl + T_WT, w);
                tmem_wait_ld();
                const int c = 32 * warp + lane;
#pragma unroll
                for (int t = 0; t < kC; ++t)
                    *reinterpret_cast<__nv_bfloat16*>(sb + (c >> 6) * 4096 + sw128(t, (c & 63) >> 3) +
                                                       (c & 7) * 2) = __float2bfloat16_rn(w[t]);
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(kBarPrep, kGroup);
            if (tid == 0) mbar_arrive(ready + p);
        }
        // After a wait gave up, let the input copies still in flight land
        // (bounded) before the CTA exits.
        if (tid == 0)
            for (int c = landed; c < issued; ++c) mbar_wait(inb + (c & 1), (c >> 1) & 1);
    } else {
        // ================================================== chain group
        uint32_t phase = 0;
        const bool lead = tid == kGroup;          // issues the chain's products
        for (int ci = 0; ci < nchunks; ++ci) {
            const int p = ci & 1;
            const int64_t t0 = bos + (int64_t)ci * kC;
            const int len = (int)((eos - t0) < kC ? (eos - t0) : kC);
            const uint8_t* sb = sm + R_SB + p * 8192;
            const uint8_t* kc = sm + R_KC + p * 4096;
            const uint8_t* pb = sm + R_PB + p * 2048;
            const float* lam = reinterpret_cast<const float*>(sm + R_LAM + p * 512);
            if (!(ok = group_wait(ready + p, (ci >> 1) & 1, kBarChain))) break;

            // ---- [(W S)^T | (qE S)^T] = S^T [W ; qE]^T, M=128 N=32 K=128
            if (lead) {
                const uint32_t idesc = idesc_bf16(128, 32);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + T_ST, desc_sw128(smem_u32(sm + R_ST + kb * 16384 + off)),
                             desc_sw128(smem_u32(sb + kb * 4096 + off)), idesc, ks > 0);
                }
                mma_commit(bar_c);
            }
            ok = group_wait(bar_c, phase, kBarChain);
            phase ^= 1u;
            if (!ok) break;
            // U^T[j][s] = U~^T[j][s] - (W S)^T[j][s] -> bf16 row j (warps 8..11)
            if (cw < 4) {
                float ws_[16], ut[16];
                tmem_ld16(tbase + tl + T_ST, ws_);
                tmem_ld16(tbase + tl + T_UT + 16 * p, ut);
                tmem_wait_ld();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint4 r;
                    r.x = pack_bf16x2(ut[8 * hh + 0] - ws_[8 * hh + 0], ut[8 * hh + 1] - ws_[8 * hh + 1]);
                    r.y = pack_bf16x2(ut[8 * hh + 2] - ws_[8 * hh + 2], ut[8 * hh + 3] - ws_[8 * hh + 3]);
                    r.z = pack_bf16x2(ut[8 * hh + 4] - ws_[8 * hh + 4], ut[8 * hh + 5] - ws_[8 * hh + 5]);
                    r.w = pack_bf16x2(ut[8 * hh + 6] - ws_[8 * hh + 6], ut[8 * hh + 7] - ws_[8 * hh + 7]);
                    *reinterpret_cast<uint4*>(sm + R_UT + sw128(j, hh)) = r;
                }
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(kBarChain, kGroup);
            tc_fence_after();

            // ---- O^T += U^T P^T (M=128 N=16 K=16); D = U^T (k lam / E) (M=128 N=128 K=16, B MN-major)
            if (lead) {
                const uint64_t ua = desc_sw128(smem_u32(sm + R_UT));
                mma_bf16(tbase + T_ST + 16, ua, desc_sw128(smem_u32(pb)), idesc_bf16(128, 16), true);
                mma_bf16(tbase + T_SU, ua, desc_sw128_mn(smem_u32(kc), 2048, 1024), idesc_bmn(128, 128), false);
                mma_commit(bar_c);
            }
            ok = group_wait(bar_c, phase, kBarChain);
            phase ^= 1u;
            if (!ok) break;

            // ---- outputs o[t0 + t][h][j] = O^T[j][t] (warps 8..11; the TMEM load is
            //      warp-collective, so every lane takes it and only the stores are masked)
            if (cw < 4) {
                float ov[16];
                tmem_ld16(tbase + tl + T_ST + 16, ov);
                tmem_wait_ld();
                if (j < dv) {
#pragma unroll
                    for (int t = 0; t < kC; ++t)
                        if (t < len) o[((size_t)(t0 + t) * H + h) * dv + j] = __float2bfloat16_rn(ov[t]);
                }
            }
            // ---- S^T <- S^T Diag(lam) + D, then its bf16 copy
#pragma unroll
            for (int q16 = 0; q16 < 4; ++q16) {
                float d[16];
                tmem_ld16(tbase + tl + T_SU + 64 * ch + 16 * q16, d);
                tmem_wait_ld();
                // lam of this slice's 16 channels as four 16-byte broadcasts
                float lv[16];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(lam + 64 * ch + 16 * q16 + 4 * e4);
                    lv[4 * e4] = l4.x; lv[4 * e4 + 1] = l4.y; lv[4 * e4 + 2] = l4.z; lv[4 * e4 + 3] = l4.w;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int idx = 16 * q16 + e;
                    st[idx] = fmaf(lv[e], st[idx], d[e]);
                }
            }
            write_st();
            if (ck.out) {
                const int64_t done = (int64_t)(ci + 1) * kC;
                if (done <= len_seq && done % ck.every == 0 && done / ck.every <= ck.max_count)
                    store_state(ck.out + (((size_t)n * H + h) * ck.max_count + (done / ck.every - 1)) * dk * dv);
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(kBarChain, kGroup);
            // the chunk's hand-over buffers are consumed
            if (lead) mbar_arrive(freed + p);
        }
    }
    if (!ok) atomicOr(status, kErrWait);
    tc_fence_before();
    __syncthreads();
    if (!prep && S1) store_state(S1 + smat);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmemCols>(tbase);
    }
}

// ---------------------------------------------------------------------------
// Speculative verify on the tensor cores (bf16 inputs).  The T <= 16 draft
// tokens of one (b, h) are one chunk of the 16-token form above, taken from
// the state S read once ("How Kimi K3 is built", section "How to serve two
// different caches": the draft tokens' projections are kept and recomputed on
// chip instead of a state copy per token).  With L_t, E, P, T, W and U~ as
// above and S the state before the span:
//   U = U~ - W S,   O = (q E) S + P U
// Persistent: CTAs of eight warps, two per SM, each walking the (b, h) pairs
// blockIdx.x, blockIdx.x + gridDim.x, ...  Per pair: the gate and its running
// sum, the operands, A/P, the solve and W^T, U~^T, then S^T (bf16) [W ; qE]^T,
// U^T and O^T += U^T P^T.  The next pair's loads are issued as soon as their
// buffers are free, so that they land while this pair computes: its draft
// inputs (cp.async, each thread its own 16-byte slots) once the operands are
// built, its state (64 values per thread, in registers) once S^T is copied.
// The state is only read.  A bounded wait that gives up leaves NaN in the
// outputs of that pair and of the CTA's remaining pairs.
// ---------------------------------------------------------------------------
constexpr int kVThreads = 256;
constexpr uint32_t V_ST = 0;          // S^T bf16 [128 j][128 c]: two K-blocks of 16 KB, swizzled
constexpr uint32_t V_UT = 32768;      // U^T bf16 [128 j][16 t]
constexpr uint32_t V_APA = 49152;     // [kE ; qE ; *] [64 rows][128 c]
constexpr uint32_t V_APB = 65536;     // k/E [16 s][128 c]
constexpr uint32_t V_SB = 69632;      // [W ; qE] [32 rows][128 c]
constexpr uint32_t V_BKG = 77824;     // b kE token rows (MN-major)
constexpr uint32_t V_BV = 81920;      // b V token rows (MN-major)
constexpr uint32_t V_PB = 86016;      // P [16 t][16 s]
constexpr uint32_t V_TB = 88064;      // T [16 t][16 s]
constexpr uint32_t V_IN2 = 90112;     // next pair's v and z: 256 threads x 16 B each
constexpr uint32_t V_AF = 98304;      // A fp32 [16][17]
constexpr uint32_t V_EA = 99584;      // e^{A_h} [128]
constexpr uint32_t V_BETA = 100096;   // beta [16]
constexpr uint32_t V_BAR = 100160;    // mbarrier, TMEM slot
constexpr uint32_t V_SMEM = V_BAR + 64 + 1024;
static_assert(2 * (V_SMEM + 1024) <= 233472, "two verify CTAs per SM");
constexpr uint32_t kVTmemCols = 128;
// The next pair's k and q sit in rows 32..63 of the A/P operand (4 KB in each
// K-block).  Those rows only feed accumulator rows 32..63 (TMEM lanes 64..79
// and 96..111 of columns T_AP..T_AP + 15), which are never read, so whatever
// they hold while the A/P product runs leaves A and P unchanged.
constexpr uint32_t V_IN_K = V_APA + 4096;
constexpr uint32_t V_IN_Q = V_APA + 8192 + 4096;
constexpr uint32_t V_IN_V = V_IN2;
constexpr uint32_t V_IN_Z = V_IN2 + 4096;

// 32 lanes x 32-bit, 8 consecutive columns: thread i of the warp receives TMEM
// lane (lane field of taddr) + i, columns col .. col + 7.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t& phase) {
    const bool ok = mbar_wait(bar, phase);
    phase ^= 1u;
    tc_fence_after();
    return __syncthreads_and(ok) != 0;
}

// Copies this thread's 16 bytes of token row `row`, channels 8 c8 .. + 7, of
// one [rows][H][d] input into its own slot; zeros where the row or the
// channels are absent.
__device__ __forceinline__ void fetch8(uint8_t* slot, const __nv_bfloat16* __restrict__ x, int64_t row,
                                       bool live, int H, int h, int d, int c8) {
    const bool in = live && 8 * c8 < d;
    const __nv_bfloat16* src = in ? x + ((size_t)row * H + h) * d + 8 * c8 : x;
    cp_async16(slot, src, in ? 16u : 0u);
}

__global__ void __launch_bounds__(kVThreads, 2)
spec_verify_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ z,
                   const __nv_bfloat16* __restrict__ beta, const float* __restrict__ A,
                   const float* __restrict__ state, __nv_bfloat16* __restrict__ o, int n_pairs,
                   int Tn, int H, int dk, int dv) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* af = reinterpret_cast<float*>(sm + V_AF);
    float* ea = reinterpret_cast<float*>(sm + V_EA);
    float* bs = reinterpret_cast<float*>(sm + V_BETA);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + V_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + V_BAR + 8);
    // token tt, channels 8 c8 .. + 7: a warp holds all 16 tokens of two channel
    // groups, so the running sum over the span is a 16-lane shuffle scan
    const int tt = lane & 15, c8 = 2 * warp + (lane >> 4);
    const int j = 32 * (warp & 3) + lane, ch = warp >> 2;  // state column j, channel half ch
    const uint32_t tl = (uint32_t)(32 * (warp & 3)) << 16;
    const bool live = tt < Tn;
    uint8_t* const slot_k = sm + V_IN_K + 16 * tid;
    uint8_t* const slot_q = sm + V_IN_Q + 16 * tid;
    uint8_t* const slot_v = sm + V_IN_V + 16 * tid;
    uint8_t* const slot_z = sm + V_IN_Z + 16 * tid;

    if (warp == 0) tmem_alloc<kVTmemCols>(tslot);
    if (tid == 32) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }

    // The first pair's loads: its draft inputs first, so that they do not queue
    // behind the state, then the state S[64 ch + e][j].
    int pair = blockIdx.x;
    float a_h = 0.f, b_t = 0.f;                 // the pair's e^{A} exponent and beta, per thread
    float st[64];
    auto fetch_inputs = [&](int p) {
        const int pb = p / H, ph = p - pb * H;
        const int64_t row = (int64_t)pb * Tn + tt;        // token row of [B, Tn, H, d]
        fetch8(slot_k, k, row, live, H, ph, dk, c8);
        fetch8(slot_q, q, row, live, H, ph, dk, c8);
        fetch8(slot_v, v, row, live, H, ph, dv, c8);
        fetch8(slot_z, z, row, live, H, ph, dk, c8);
        a_h = (tid < 128 && tid < dk) ? A[(size_t)ph * dk + tid] : 0.f;
        b_t = (tid < kC && tid < Tn) ? __bfloat162float(beta[((size_t)pb * Tn + tid) * H + ph]) : 0.f;
    };
    auto fetch_state = [&](int p) {
        const float* Sp = state + (size_t)p * dk * dv;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            const int c = 64 * ch + e;
            st[e] = (c < dk && j < dv) ? __ldcs(Sp + (size_t)c * dv + j) : 0.f;
        }
    };
    if (pair < n_pairs) {
        fetch_inputs(pair);
        fetch_state(pair);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    uint32_t phase = 0;
    bool ok = true;

    for (; pair < n_pairs; pair += gridDim.x) {
        const int b = pair / H, h = pair - b * H;
        const int next = pair + gridDim.x;
        if (ok) do {
            if (tid < 128) ea[tid] = tid < dk ? __expf(a_h) : 0.f;
            if (tid < kC) bs[tid] = b_t;
            cp_async_wait_all();                    // this thread's own slots have landed
            __syncthreads();
            // ---- gate, and its running sum L over the span (inclusive shuffle scan)
            {
                const uint4 zr = *reinterpret_cast<const uint4*>(slot_z);
                float zf[8], L[8];
                unpack8(zr, zf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = 8 * c8 + e;
                    L[e] = (live && c < dk) ? gate_fast(ea[c], zf[e]) : 0.f;
                }
#pragma unroll
                for (int off = 1; off < kC; off <<= 1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float y = __shfl_up_sync(0xffffffffu, L[e], off, kC);
                        if (tt >= off) L[e] += y;
                    }
                }
                // ---- decay-scaled operands of token tt
                const uint4 kr = *reinterpret_cast<const uint4*>(slot_k);
                const uint4 qr = *reinterpret_cast<const uint4*>(slot_q);
                const uint4 vr = *reinterpret_cast<const uint4*>(slot_v);
                float kf[8], qf[8], vf[8], E[8], o8[8];
                unpack8(kr, kf);
                unpack8(qr, qf);
                unpack8(vr, vf);
#pragma unroll
                for (int e = 0; e < 8; ++e) E[e] = __expf(L[e]);
                const float bt = bs[tt];
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = kf[e] * E[e];
                store_row8(sm + V_APA, 8192, tt, c8, o8);                           // k E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = bt * o8[e];
                store_row8(sm + V_BKG, 2048, tt, c8, o8);                           // b k E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[e];
                store_row8(sm + V_APA, 8192, 16 + tt, c8, o8);                      // q E
                store_row8(sm + V_SB, 4096, 16 + tt, c8, o8);
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = kf[e] * __fdividef(1.0f, E[e]);
                store_row8(sm + V_APB, 2048, tt, c8, o8);                           // k / E
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = bt * vf[e];
                store_row8(sm + V_BV, 2048, tt, c8, o8);                            // b V
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // every slot has been read: the next pair's inputs start now
            if (next < n_pairs) fetch_inputs(next);
            // ---- A and P (M=64 N=16 K=128)
            if (tid == 0) {
                const uint32_t idesc = idesc_bf16(64, 16);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + T_AP, desc_sw128(smem_u32(sm + V_APA + kb * 8192 + off)),
                             desc_sw128(smem_u32(sm + V_APB + kb * 2048 + off)), idesc, ks > 0);
                }
                mma_commit(bar);
            }
            if (!(ok = cta_wait(bar, phase))) break;
            if (warp < 2) {
                float d[16];
                tmem_ld16(tbase + tl + T_AP, d);
                tmem_wait_ld();
                if (lane < kC) {
                    const int t = lane;
                    if (warp == 0) {
                        const float bt = bs[t];
#pragma unroll
                        for (int s2 = 0; s2 < kC; ++s2) af[t * 17 + s2] = s2 < t ? bt * d[s2] : 0.f;
                    } else {
                        float p8[8];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) p8[e] = (8 * hh + e <= t) ? d[8 * hh + e] : 0.f;
                            uint4 r;
                            r.x = pack_bf16x2(p8[0], p8[1]);
                            r.y = pack_bf16x2(p8[2], p8[3]);
                            r.z = pack_bf16x2(p8[4], p8[5]);
                            r.w = pack_bf16x2(p8[6], p8[7]);
                            *reinterpret_cast<uint4*>(sm + V_PB + sw128(t, hh)) = r;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncthreads();
            // ---- T = (I + A)^{-1}
            if (tid < kC) {
                const int jc = tid;
                float x[kC];
#pragma unroll
                for (int r = 0; r < kC; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) acc = fmaf(af[r * 17 + m], x[m], acc);
                    x[r] = (r < jc) ? 0.f : (r == jc ? 1.f : -acc);
                }
#pragma unroll
                for (int r = 0; r < kC; ++r)
                    *reinterpret_cast<__nv_bfloat16*>(sm + V_TB + sw128(r, jc >> 3) + (jc & 7) * 2) =
                        __float2bfloat16_rn(x[r]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ---- W^T and U~^T (M=128 N=16 K=16, A MN-major)
            if (tid == 0) {
                const uint32_t idesc = idesc_bf16_amn(128, 16);
                const uint64_t tb = desc_sw128(smem_u32(sm + V_TB));
                mma_bf16(tbase + T_WT, desc_sw128_mn(smem_u32(sm + V_BKG), 2048, 1024), tb, idesc, false);
                mma_bf16(tbase + T_UT, desc_sw128_mn(smem_u32(sm + V_BV), 2048, 1024), tb, idesc, false);
                mma_commit(bar);
            }
            if (!(ok = cta_wait(bar, phase))) break;
            {
                // W rows: channel c = lane j of the warp's quadrant, tokens 8 th .. 8 th + 7
                const int th = warp >> 2, c = j;
                float w[8];
                tmem_ld8(tbase + tl + T_WT + 8 * th, w);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    *reinterpret_cast<__nv_bfloat16*>(sm + V_SB + (c >> 6) * 4096 + sw128(8 * th + t, (c & 63) >> 3) +
                                                       (c & 7) * 2) = __float2bfloat16_rn(w[t]);
            }
            // ---- the state's bf16 copy S^T, row j (its loads have landed by now)
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint4 r;
                r.x = pack_bf16x2(st[8 * q8 + 0], st[8 * q8 + 1]);
                r.y = pack_bf16x2(st[8 * q8 + 2], st[8 * q8 + 3]);
                r.z = pack_bf16x2(st[8 * q8 + 4], st[8 * q8 + 5]);
                r.w = pack_bf16x2(st[8 * q8 + 6], st[8 * q8 + 7]);
                *reinterpret_cast<uint4*>(sm + V_ST + ch * 16384 + sw128(j, q8)) = r;
            }
            // the registers are free: the next pair's state starts now
            if (next < n_pairs) fetch_state(next);
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ---- [(W S)^T | (qE S)^T] = S^T [W ; qE]^T (M=128 N=32 K=128)
            if (tid == 0) {
                const uint32_t idesc = idesc_bf16(128, 32);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + T_ST, desc_sw128(smem_u32(sm + V_ST + kb * 16384 + off)),
                             desc_sw128(smem_u32(sm + V_SB + kb * 4096 + off)), idesc, ks > 0);
                }
                mma_commit(bar);
            }
            if (!(ok = cta_wait(bar, phase))) break;
            {
                // U^T row j, tokens 8 hh .. 8 hh + 7 (hh = warp half)
                const int hh = warp >> 2;
                float ws_[8], ut[8];
                tmem_ld8(tbase + tl + T_ST + 8 * hh, ws_);
                tmem_ld8(tbase + tl + T_UT + 8 * hh, ut);
                tmem_wait_ld();
                uint4 r;
                r.x = pack_bf16x2(ut[0] - ws_[0], ut[1] - ws_[1]);
                r.y = pack_bf16x2(ut[2] - ws_[2], ut[3] - ws_[3]);
                r.z = pack_bf16x2(ut[4] - ws_[4], ut[5] - ws_[5]);
                r.w = pack_bf16x2(ut[6] - ws_[6], ut[7] - ws_[7]);
                *reinterpret_cast<uint4*>(sm + V_UT + sw128(j, hh)) = r;
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            // ---- O^T += U^T P^T (M=128 N=16 K=16)
            if (tid == 0) {
                mma_bf16(tbase + T_ST + 16, desc_sw128(smem_u32(sm + V_UT)), desc_sw128(smem_u32(sm + V_PB)),
                         idesc_bf16(128, 16), true);
                mma_commit(bar);
            }
            ok = cta_wait(bar, phase);
        } while (false);

        // ---- outputs o[b][t][h][j], tokens 8 th .. 8 th + 7 (th = warp half); NaN
        //      once a wait has given up
        {
            const int th = warp >> 2;
            float ov[8];
            if (ok) {
                tmem_ld8(tbase + tl + T_ST + 16 + 8 * th, ov);
                tmem_wait_ld();
            }
            if (j < dv) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 8 * th + e;
                    if (t < Tn)
                        o[(((size_t)b * Tn + t) * H + h) * dv + j] =
                            __float2bfloat16_rn(ok ? ov[e] : __int_as_float(0x7fc00000));
                }
            }
        }
        // this pair's TMEM reads are done before the next pair's products
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    cp_async_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kVTmemCols>(tbase);
    }
}

}  // namespace c16

cudaError_t run_chunk16_tc(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, void* o, const float* S0, float* S1,
                           const int32_t* cu, int n_seqs, int64_t T, int64_t T_total, int H,
                           int dk, int dv, void* workspace, const CheckpointSpec& ck,
                           cudaStream_t stream) {
    constexpr int kMaxDevices = 64;
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(c16::chunk16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)c16::SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    uint32_t* status = static_cast<uint32_t*>(workspace);
    e = cudaMemsetAsync(status, 0, CHUNK16_WORKSPACE_BYTES, stream);
    if (e != cudaSuccess) return e;
    // TMA token coordinates are 32-bit.  Without tokens no input is read (the
    // kernel only passes the states through), so no map is built.
    if (T_total > 0x7fffffffLL) return cudaErrorInvalidValue;
    c16::InputMaps16 maps;
    memset(&maps, 0, sizeof(maps));
    if (T_total > 0 && (!make_rows_tensor_map(&maps.q, q, T_total, H, dk, c16::kC) ||
                        !make_rows_tensor_map(&maps.k, k, T_total, H, dk, c16::kC) ||
                        !make_rows_tensor_map(&maps.v, v, T_total, H, dv, c16::kC) ||
                        !make_rows_tensor_map(&maps.z, z, T_total, H, dk, c16::kC)))
        return cudaErrorInvalidValue;
    using bf = __nv_bfloat16;
    profile_event(0, stream);
    dim3 grid((unsigned)n_seqs, (unsigned)H);
    c16::chunk16_kernel<<<grid, c16::kThreads, c16::SMEM, stream>>>(
        maps, static_cast<const bf*>(beta), A, static_cast<bf*>(o), S0, S1, cu, T, T_total, H, dk, dv,
        status, ck);
    e = cudaGetLastError();
    profile_event(1, stream);
    return e;
}

cudaError_t run_spec_verify_tc(const void* q, const void* k, const void* v, const void* z,
                               const void* beta, const float* A, const float* state, void* o, int B,
                               int Tn, int H, int dk, int dv, cudaStream_t stream) {
    constexpr int kMaxDevices = 64;
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(c16::spec_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)c16::V_SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    static int sm_count[kMaxDevices] = {};
    if (sm_count[dev] == 0) {
        e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int64_t n_pairs = (int64_t)B * H;
    if (n_pairs > INT32_MAX) return cudaErrorInvalidValue;
    if (n_pairs == 0) return cudaSuccess;
    // two persistent CTAs per SM walk the (b, h) pairs
    const int64_t grid = n_pairs < 2LL * sm_count[dev] ? n_pairs : 2LL * sm_count[dev];
    using bf = __nv_bfloat16;
    c16::spec_verify_kernel<<<(unsigned)grid, c16::kVThreads, c16::V_SMEM, stream>>>(
        static_cast<const bf*>(q), static_cast<const bf*>(k), static_cast<const bf*>(v),
        static_cast<const bf*>(z), static_cast<const bf*>(beta), A, state, static_cast<bf*>(o),
        (int)n_pairs, Tn, H, dk, dv);
    return cudaGetLastError();
}

}  // namespace kda
