// kda_chunked_tc.cu -- chunked KDA prefill on the sm_103a tensor cores
// (bf16 inputs, d_k = d_v = 128, chunk C = 64).
//
// The pages describe the kernel only in outline: tokens inside a chunk are
// processed in parallel and the state is then passed on across all heads
// ("Kimi K3 architecture review", chip-level FlashKDA section), and bounding
// the log-decay below by g_min = -5 keeps every causal block a dense matmul
// with no separate diagonal path ("How Kimi K3 is built", gate section).  The
// algebra below is derived from the recurrence.  Per (sequence, head) and
// chunk, with start state S0 and G_t = running sum of g inside the chunk:
//
//   A_ts = b_t sum_c k_tc k_sc e^{G_tc - G_sc}   (s < t)     T = (I + A)^{-1}
//   P_ts =     sum_c q_tc k_sc e^{G_tc - G_sc}   (s <= t)
//   W = T Diag(b) K^g,  U~ = T Diag(b) V,        K^g_t = k_t e^{G_t}
//   U = U~ - W S0,  O = Q^g S0 + P U,            Q^g_t = q_t e^{G_t}
//   S_C = Diag(e^{G_C}) S0 + (K^C)^T U,          K^C_s = k_s e^{G_C - G_s}
//
// Two kernels:
//   chunk_prep   one CTA per (chunk, head), fully parallel.  Gate, cumulative
//                log-decay, decay-scaled operands, A and P as tcgen05 MMAs into
//                TMEM, the unit-lower solve for T, then W and U~ as MMAs.  It
//                writes a 73 KB "package" per (chunk, head) to the workspace,
//                laid out exactly as the shared-memory operand images the
//                state pass consumes (128-byte-swizzled K-major tiles).
//   state_pass   one CTA per (sequence, head), sequential over chunks.  Holds
//                S in fp32 registers, streams packages with one bulk copy per
//                chunk (double-buffered), and runs the three state products
//                (W S, Q^g S + P U, (K^C)^T U) on tcgen05 with S^T and U^T as
//                bf16 shared-memory operands.
//
// Decay factoring.  Over a 64-token chunk G spans down to -320, so e^{+-G}
// does not fit fp32/bf16.  With g >= -5 a 16-token block spans at most e^80,
// which does.  Row t (in 16-row block i) of the causal products is scaled
// to the reference r_i = G at the token before block i: the row operand
// k_t e^{G_t - r_i} <= 1 and the column operand k_s e^{r_i - G_s} <= e^80
// (>= 1 only inside block i).  The column operand therefore has one variant
// per row block (K^(i), rows s < 16(i+1)); the four products are dense
// M=128 MMAs whose A operand stacks the 64 key rows over the 64 query rows.
#include <cuda_bf16.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace tc {

constexpr int kC = 64;        // chunk length
constexpr int kD = 128;       // d_k = d_v
constexpr int kThreads = 256;

// ---- package: one per (chunk, head), byte offsets -------------------------
constexpr uint32_t PKG_W = 0;        // W    [t][c]  two swizzled K-blocks (c<64, c>=64), 8 KB each
constexpr uint32_t PKG_Q = 16384;    // Q^g  [t][c]  same layout
constexpr uint32_t PKG_KC = 32768;   // K^C  [c][s]  one swizzled K-block, 128 rows
constexpr uint32_t PKG_P = 49152;    // P    [t][s]  one swizzled K-block, 64 rows
constexpr uint32_t PKG_U = 57344;    // U~   [t][j]  plain row-major bf16
constexpr uint32_t PKG_LAM = 73728;  // e^{G_C} [c] fp32
constexpr uint32_t PKG_BYTES = 74752;
constexpr uint32_t WS_HEADER = 1024;  // word 0: device status (0 = ok)

// Status bits written to workspace word 0 when a bounded wait gives up.
constexpr uint32_t kErrPrepWait = 1u;
constexpr uint32_t kErrStateWait = 2u;

// ---- chunk_prep shared memory (offsets from a 1024-byte aligned base) -----
constexpr uint32_t P_K = 0;            // raw k [64][128] bf16        -> later W staging
constexpr uint32_t P_V = 16384;        // raw v [64][128] bf16        -> later U~ staging
constexpr uint32_t P_G = 32768;        // G fp32 [64][132]            -> later P staging
constexpr uint32_t G_LD = 132;
constexpr uint32_t P_AST = 67584;      // A-stack [128][128] swizzled -> later A fp32, T fp32
constexpr uint32_t P_KV = 100352;      // K^(i) variants (40 KB)      -> later T bf16, scratch
constexpr uint32_t P_BKT = 141312;     // (b K^g)^T [128][64] swizzled
constexpr uint32_t P_BVT = 157696;     // (b V)^T   [128][64] swizzled
constexpr uint32_t P_KC = 174080;      // K^C staging [128][64] swizzled
constexpr uint32_t P_SMALL = 190464;   // per-channel constants, beta
constexpr uint32_t P_AF = P_AST;       // A fp32 [64][65]
constexpr uint32_t P_TF = P_AST + 16896;  // T fp32 [64][65]
constexpr uint32_t P_TB = P_KV + 1024; // T bf16 [64][64] swizzled (T fp32 ends at P_KV + 768)
constexpr uint32_t P_XS = P_TB + 8192; // solve scratch [3][16][16] fp32
constexpr uint32_t F_LD = 65;
// small region, in floats: R[5][128] refs, X[6][128] cross factors,
// ER[4][128] = e^{r_b}, EC[4][128] = e^{G_C - r_b}, beta[64]
constexpr uint32_t SM_R = 0, SM_X = 640, SM_ER = 1408, SM_EC = 1920, SM_B = 2432;
constexpr uint32_t P_SMALL_BYTES = (2432 + 64) * 4;
constexpr uint32_t P_BAR = P_SMALL + P_SMALL_BYTES;  // mbarrier + TMEM slot
constexpr uint32_t P_SMEM = P_BAR + 64 + 1024;       // + alignment slack

// K^(i): variant i covers rows s < 16 (i + 1); two K-blocks of N_i * 128 bytes.
__host__ __device__ constexpr uint32_t kv_base(int i) {
    return i == 0 ? 0u : i == 1 ? 4096u : i == 2 ? 12288u : 24576u;
}
__host__ __device__ constexpr uint32_t kv_rows(int i) { return 16u * (uint32_t)(i + 1); }
// TMEM columns of the row-block products D_i (width 16 (i + 1)).
__host__ __device__ constexpr uint32_t d_col(int i) {
    return i == 0 ? 0u : i == 1 ? 16u : i == 2 ? 48u : 96u;
}
// Index of the cross factor e^{r_i - r_b} for i > b.
__host__ __device__ constexpr int xidx(int i, int b) {
    return b == 0 ? i - 1 : (b == 1 ? i + 1 : 5);   // (1,0)0 (2,0)1 (3,0)2 (2,1)3 (3,1)4 (3,2)5
}

// ---- state_pass shared memory ---------------------------------------------
constexpr uint32_t S_STAGE0 = 0;
constexpr uint32_t S_STAGE1 = PKG_BYTES;           // 73 * 1024
constexpr uint32_t S_ST = 2 * PKG_BYTES;           // S^T [128 j][128 c] swizzled, 2 K-blocks
constexpr uint32_t S_UT = S_ST + 32768;            // U^T [128 j][64 t] swizzled
constexpr uint32_t S_BAR = S_UT + 16384;
constexpr uint32_t S_SMEM = S_BAR + 64 + 1024;

struct SeqMap {
    const int32_t* cu;  // nullable
    int64_t T;          // per-sequence length when cu == nullptr
    int64_t T_total;
    int n_seqs;
};

// First package slot of sequence n: floor(bos / 64) + n.  Slots of different
// sequences never overlap, and every slot is below floor(T_total / 64) + n_seqs.
__device__ __forceinline__ int64_t seq_slot_base(const SeqMap& m, int n, int64_t& bos,
                                                 int64_t& eos) {
    seq_bounds(m.cu, n, m.T, m.T_total, bos, eos);
    return bos / kC + n;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
    atomicOr(status, bit);
}

__device__ __forceinline__ void unpack8(uint4 raw, float (&f)[8]) {
    const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __bfloat162float(b[e]);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 r;
    r.x = pack_bf16x2(f[0], f[1]);
    r.y = pack_bf16x2(f[2], f[3]);
    r.z = pack_bf16x2(f[4], f[5]);
    r.w = pack_bf16x2(f[6], f[7]);
    return r;
}

// Row-block product readback: thread owns row t of block I; copies D_I's
// 16 (I + 1) columns into row[] (columns beyond stay as they are).
template <int I>
__device__ __forceinline__ void load_block_row(uint32_t taddr_lane, bool mine, float (&row)[64]) {
#pragma unroll
    for (int q = 0; q <= I; ++q) {
        float v[16];
        tmem_ld16(taddr_lane + d_col(I) + 16u * q, v);
        tmem_wait_ld();
        if (mine) {
#pragma unroll
            for (int e = 0; e < 16; ++e) row[16 * q + e] = v[e];
        }
    }
}

// One step of the blocked unit-lower inverse: for every block pair (i, j) with
// i - j = d, X = sum_{m=j}^{i-1} A_im T_mj, then T_ij = -T_ii X.
template <int d>
__device__ __forceinline__ void solve_offdiag(const float* Af, float* Tf, float* Xs, int tid) {
    const int r = tid >> 4, col = tid & 15;
#pragma unroll
    for (int p = 0; p < 4 - d; ++p) {
        const int jb = p, ib = p + d;
        float acc = 0.f;
        for (int m = jb; m < ib; ++m) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
                acc = fmaf(Af[(16 * ib + r) * F_LD + 16 * m + e], Tf[(16 * m + e) * F_LD + 16 * jb + col],
                           acc);
        }
        Xs[(p * 16 + r) * 16 + col] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < 4 - d; ++p) {
        const int jb = p, ib = p + d;
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            acc = fmaf(Tf[(16 * ib + r) * F_LD + 16 * ib + e], Xs[(p * 16 + e) * 16 + col], acc);
        Tf[(16 * ib + r) * F_LD + 16 * jb + col] = -acc;
    }
    __syncthreads();
}

// ============================================================================
// chunk_prep: one CTA per (package slot, head).
// ============================================================================
__global__ void __launch_bounds__(kThreads, 1)
chunk_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ z,
                  const __nv_bfloat16* __restrict__ beta, const float* __restrict__ A,
                  uint8_t* __restrict__ ws, SeqMap map, int H) {
    const int slot = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Which sequence and chunk this slot holds (binary search on slot bases).
    int lo = 0, hi = map.n_seqs - 1;
    int64_t bos, eos;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seq_slot_base(map, mid, bos, eos) <= slot) lo = mid; else hi = mid - 1;
    }
    const int64_t chunk = slot - seq_slot_base(map, lo, bos, eos);
    const int64_t n_chunks = (eos - bos + kC - 1) / kC;
    if (chunk < 0 || chunk >= n_chunks) return;   // empty slot: nothing allocated yet
    const int64_t t0 = bos + chunk * kC;
    const int len = (int)((eos - t0) < kC ? (eos - t0) : kC);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* G = reinterpret_cast<float*>(sm + P_G);
    float* small = reinterpret_cast<float*>(sm + P_SMALL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + P_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + P_BAR + 8);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    uint8_t* pkg = ws + WS_HEADER + ((size_t)slot * H + h) * PKG_BYTES;

    if (warp == 0) tmem_alloc<256>(tslot);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }

    // ---- phase 0: raw k and v rows into shared memory (zero rows past len)
    const size_t row0 = ((size_t)t0 * H + h) * kD;
    const size_t rstride = (size_t)H * kD;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int i = it * kThreads + tid;           // 0..2047
        const int which = i >> 10, t = (i >> 4) & 63, ch = i & 15;
        const __nv_bfloat16* src = (which ? v : k) + row0 + (size_t)(t < len ? t : 0) * rstride + ch * 8;
        cp_async16(sm + (which ? P_V : P_K) + t * 256 + ch * 16, src, t < len ? 16u : 0u);
    }
    if (tid < kC)
        small[SM_B + tid] = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;

    // ---- phase A: gate g = -5 sigmoid(e^A z) into G (0 on padded rows)
    {
        const int c8 = tid & 15;
        float eA[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) eA[e] = __expf(A[(size_t)h * kD + c8 * 8 + e]);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int t = it * 16 + (tid >> 4);
            float g[8];
            if (t < len) {
                float zf[8];
                unpack8(__ldg(reinterpret_cast<const uint4*>(z + row0 + (size_t)t * rstride + c8 * 8)), zf);
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = gate_fast(eA[e], zf[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = 0.f;
            }
            float4* dst = reinterpret_cast<float4*>(G + t * G_LD + c8 * 8);
            dst[0] = make_float4(g[0], g[1], g[2], g[3]);
            dst[1] = make_float4(g[4], g[5], g[6], g[7]);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- phase B: G = running sum over the chunk, per channel
    {
        const int c = tid & 127, half = tid >> 7;
        float run = 0.f;
        for (int t = 32 * half; t < 32 * half + 32; ++t) {
            run += G[t * G_LD + c];
            G[t * G_LD + c] = run;
        }
        __syncthreads();
        if (half) {
            const float carry = G[31 * G_LD + c];
            for (int t = 32; t < 64; ++t) G[t * G_LD + c] += carry;
        }
        __syncthreads();
        const float r1 = G[15 * G_LD + c], r2 = G[31 * G_LD + c], r3 = G[47 * G_LD + c];
        const float rc = G[63 * G_LD + c];
        if (half == 0) {
            small[SM_R + 0 * 128 + c] = 0.f;
            small[SM_R + 1 * 128 + c] = r1;
            small[SM_R + 2 * 128 + c] = r2;
            small[SM_R + 3 * 128 + c] = r3;
            small[SM_R + 4 * 128 + c] = rc;
            small[SM_ER + 0 * 128 + c] = 1.f;
            small[SM_ER + 1 * 128 + c] = __expf(r1);
            small[SM_ER + 2 * 128 + c] = __expf(r2);
            small[SM_ER + 3 * 128 + c] = __expf(r3);
            reinterpret_cast<float*>(pkg + PKG_LAM)[c] = __expf(rc);
        } else {
            small[SM_EC + 0 * 128 + c] = __expf(rc);
            small[SM_EC + 1 * 128 + c] = __expf(rc - r1);
            small[SM_EC + 2 * 128 + c] = __expf(rc - r2);
            small[SM_EC + 3 * 128 + c] = __expf(rc - r3);
            small[SM_X + xidx(1, 0) * 128 + c] = __expf(r1);
            small[SM_X + xidx(2, 0) * 128 + c] = __expf(r2);
            small[SM_X + xidx(3, 0) * 128 + c] = __expf(r3);
            small[SM_X + xidx(2, 1) * 128 + c] = __expf(r2 - r1);
            small[SM_X + xidx(3, 1) * 128 + c] = __expf(r3 - r1);
            small[SM_X + xidx(3, 2) * 128 + c] = __expf(r3 - r2);
        }
        __syncthreads();
    }

    // ---- phase C1: row-side operands (thread = token t, 8 channels)
    {
        const int c8 = tid & 15, kb = c8 >> 3, chk = c8 & 7;
#pragma unroll 1
        for (int it = 0; it < 4; ++it) {
            const int t = it * 16 + (tid >> 4);
            const int b = t >> 4;
            const float4* gp = reinterpret_cast<const float4*>(G + t * G_LD + c8 * 8);
            const float4 g0 = gp[0], g1 = gp[1];
            const float gt[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            float kf[8], qf[8], E[8], Rr[8];
            unpack8(*reinterpret_cast<const uint4*>(sm + P_K + t * 256 + c8 * 16), kf);
            if (t < len)
                unpack8(__ldg(reinterpret_cast<const uint4*>(q + row0 + (size_t)t * rstride + c8 * 8)), qf);
            else
#pragma unroll
                for (int e = 0; e < 8; ++e) qf[e] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                E[e] = __expf(gt[e] - small[SM_R + b * 128 + c8 * 8 + e]);   // e^{G_t - r_b} <= 1
                Rr[e] = __fdividef(1.0f, E[e]);                              // e^{r_b - G_t} <= e^80
            }
            float o8[8];
            // A-stack: key rows 0..63, query rows 64..127, both scaled to r_b.
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = kf[e] * E[e];
            *reinterpret_cast<uint4*>(sm + P_AST + kb * 16384 + sw128(t, chk)) = pack8(o8);
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[e];
            *reinterpret_cast<uint4*>(sm + P_AST + kb * 16384 + sw128(64 + t, chk)) = pack8(o8);
            // Q^g for the state pass: q e^{G_t} = q E e^{r_b}.
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[e] * small[SM_ER + b * 128 + c8 * 8 + e];
            *reinterpret_cast<uint4*>(pkg + PKG_Q + kb * 8192 + sw128(t, chk)) = pack8(o8);
            // Column variants K^(i) for i >= b: k e^{r_i - G_t} = k R e^{r_i - r_b}.
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (i < b) continue;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = (i == b) ? 1.f : small[SM_X + xidx(i, b) * 128 + c8 * 8 + e];
                    o8[e] = kf[e] * Rr[e] * x;
                }
                *reinterpret_cast<uint4*>(sm + P_KV + kv_base(i) + kb * kv_rows(i) * 128 +
                                          sw128(t, chk)) = pack8(o8);
            }
        }
    }

    // ---- phase C2: column-side operands, transposed (thread = channel c, 8 tokens)
    {
        const int c = tid & 127, sg = tid >> 7;
        const __nv_bfloat16* kraw = reinterpret_cast<const __nv_bfloat16*>(sm + P_K);
        const __nv_bfloat16* vraw = reinterpret_cast<const __nv_bfloat16*>(sm + P_V);
#pragma unroll 1
        for (int it = 0; it < 4; ++it) {
            const int s8 = sg * 4 + it, b = s8 >> 1;
            const float rb = small[SM_R + b * 128 + c], er = small[SM_ER + b * 128 + c];
            const float ec = small[SM_EC + b * 128 + c];
            float bk[8], kc[8], bv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = s8 * 8 + e;
                const float bs = small[SM_B + s];
                const float kf = __bfloat162float(kraw[s * kD + c]);
                const float E = __expf(G[s * G_LD + c] - rb);
                bk[e] = bs * kf * E * er;                    // b_s k_s e^{G_s}
                kc[e] = kf * ec * __fdividef(1.0f, E);       // k_s e^{G_C - G_s}
                bv[e] = bs * __bfloat162float(vraw[s * kD + c]);
            }
            *reinterpret_cast<uint4*>(sm + P_BKT + sw128(c, s8)) = pack8(bk);
            *reinterpret_cast<uint4*>(sm + P_KC + sw128(c, s8)) = pack8(kc);
            *reinterpret_cast<uint4*>(sm + P_BVT + sw128(c, s8)) = pack8(bv);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    // ---- A and P: four row-block products D_i = Astack * K^(i)^T into TMEM
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t idesc = idesc_bf16(128, kv_rows(i));
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                const uint64_t ad = desc_sw128(smem_u32(sm + P_AST + kb * 16384 + off));
                const uint64_t bd =
                    desc_sw128(smem_u32(sm + P_KV + kv_base(i) + kb * kv_rows(i) * 128 + off));
                mma_bf16(tbase + d_col(i), ad, bd, idesc, ks > 0);
            }
        }
        mma_commit(bar);
        bulk_s2g(pkg + PKG_KC, sm + P_KC, 16384);
        bulk_commit();
    }
    bool ok = mbar_wait(bar, 0);
    if (!ok) set_status(status, kErrPrepWait);
    tc_fence_after();

    // Readback: warps 0/1 hold key rows (-> A), warps 2/3 query rows (-> P).
    if (warp < 4) {
        const int lane_base = 32 * warp;
        const int t = (lane_base + lane) & 63;
        const int blk = t >> 4;
        const uint32_t taddr = tbase + ((uint32_t)lane_base << 16);
        float row[64];
#pragma unroll
        for (int s = 0; s < 64; ++s) row[s] = 0.f;
        if ((warp & 1) == 0) {
            load_block_row<0>(taddr, blk == 0, row);
            load_block_row<1>(taddr, blk == 1, row);
        } else {
            load_block_row<2>(taddr, blk == 2, row);
            load_block_row<3>(taddr, blk == 3, row);
        }
        if (warp < 2) {
            float* Af = reinterpret_cast<float*>(sm + P_AF);
            const float bt = small[SM_B + t];
#pragma unroll
            for (int s = 0; s < 64; ++s) Af[t * F_LD + s] = (s < t) ? bt * row[s] : 0.f;
        } else {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = (ch * 8 + e <= t) ? row[ch * 8 + e] : 0.f;
                *reinterpret_cast<uint4*>(sm + P_G + sw128(t, ch)) = pack8(o8);   // P staging
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(pkg + PKG_P, sm + P_G, 8192);
        bulk_commit();
    }

    // ---- T = (I + A)^{-1}: diagonal 16x16 blocks by forward substitution,
    //      then off-diagonal blocks by distance.
    {
        const float* Af = reinterpret_cast<const float*>(sm + P_AF);
        float* Tf = reinterpret_cast<float*>(sm + P_TF);
        float* Xs = reinterpret_cast<float*>(sm + P_XS);
        if (tid < 64) {
            const int blk = tid >> 4, j = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(Af[(16 * blk + r) * F_LD + 16 * blk + m], x[m], acc);
                x[r] = (r < j) ? 0.f : (r == j ? 1.f : -acc);
                Tf[(16 * blk + r) * F_LD + 16 * blk + j] = x[r];
            }
        }
        __syncthreads();
        solve_offdiag<1>(Af, Tf, Xs, tid);
        solve_offdiag<2>(Af, Tf, Xs, tid);
        solve_offdiag<3>(Af, Tf, Xs, tid);
        // T as a bf16 K-major operand [t][s]
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int i = it * kThreads + tid, t = i >> 3, ch = i & 7;
            float o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = ch * 8 + e;
                o8[e] = (s <= t) ? Tf[t * F_LD + s] : 0.f;
            }
            *reinterpret_cast<uint4*>(sm + P_TB + sw128(t, ch)) = pack8(o8);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- W^T = (b K^g)^T T^T and U~^T = (b V)^T T^T  (M = 128, N = 64, K = 64)
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, 64);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = desc_sw128(smem_u32(sm + P_TB + ks * 32));
            mma_bf16(tbase + 0, desc_sw128(smem_u32(sm + P_BKT + ks * 32)), bd, idesc, ks > 0);
            mma_bf16(tbase + 64, desc_sw128(smem_u32(sm + P_BVT + ks * 32)), bd, idesc, ks > 0);
        }
        mma_commit(bar);
    }
    ok = mbar_wait(bar, 1);
    if (!ok) set_status(status, kErrPrepWait);
    tc_fence_after();
    {
        const int lane_base = 32 * (warp & 3);
        const int cidx = lane_base + lane;           // channel c (W) or column j (U~)
        const uint32_t taddr = tbase + ((uint32_t)lane_base << 16) + (warp < 4 ? 0u : 64u);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float vals[16];
            tmem_ld16(taddr + 16 * q4, vals);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int t = 16 * q4 + e;
                const __nv_bfloat16 bv = __float2bfloat16_rn(vals[e]);
                if (warp < 4) {
                    const uint32_t kb = cidx >> 6, cc = cidx & 63;
                    *reinterpret_cast<__nv_bfloat16*>(sm + P_K + kb * 8192 + sw128(t, cc >> 3) +
                                                      (cc & 7) * 2) = bv;
                } else {
                    *reinterpret_cast<__nv_bfloat16*>(sm + P_V + t * 256 + cidx * 2) = bv;
                }
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(pkg + PKG_W, sm + P_K, 16384);
        bulk_s2g(pkg + PKG_U, sm + P_V, 16384);
        bulk_commit();
        bulk_wait_all();
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<256>(tbase);
    }
}

// ============================================================================
// state_pass: one CTA per (sequence, head), sequential over its chunks.
// Thread (warp w, lane l) owns state column j = 32 (w mod 4) + l and the
// channel half c in [64 g, 64 g + 64), g = w / 4.
// ============================================================================
__global__ void __launch_bounds__(kThreads, 1)
state_pass_kernel(const uint8_t* __restrict__ ws, __nv_bfloat16* __restrict__ o,
                  const float* __restrict__ S0, float* __restrict__ S1, SeqMap map, int H) {
    const int n = blockIdx.x, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lane_base = 32 * (warp & 3);
    const int j = lane_base + lane, g = warp >> 2;

    int64_t bos, eos;
    const int64_t slot0 = seq_slot_base(map, n, bos, eos);
    const int nc = (int)((eos - bos + kC - 1) / kC);
    uint32_t* status = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(ws));
    const uint8_t* pkgs = ws + WS_HEADER;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S_BAR);        // [2]
    uint64_t* mma1 = full + 2;
    uint64_t* mma2 = full + 3;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 4);
    __shared__ int s_abort;

    const size_t sbase = ((size_t)n * H + h) * kD * kD;
    float st[64];
#pragma unroll
    for (int e = 0; e < 64; ++e)
        st[e] = S0 ? S0[sbase + (size_t)(64 * g + e) * kD + j] : 0.f;

    if (nc == 0) {      // empty sequence: the final state is the initial one
        if (S1) {
#pragma unroll
            for (int e = 0; e < 64; ++e) S1[sbase + (size_t)(64 * g + e) * kD + j] = st[e];
        }
        return;
    }

    if (warp == 0) tmem_alloc<256>(tslot);
    if (tid == 0) {
        mbar_init(full + 0, 1);
        mbar_init(full + 1, 1);
        mbar_init(mma1, 1);
        mbar_init(mma2, 1);
        fence_mbar_init();
        s_abort = 0;
        for (int p = 0; p < 2 && p < nc; ++p) {
            const uint8_t* src = pkgs + ((size_t)(slot0 + p) * H + h) * PKG_BYTES;
            mbar_expect_tx(full + p, PKG_BYTES);
            uint8_t* dst = sm + (p ? S_STAGE1 : S_STAGE0);
            bulk_g2s(dst, src, 32768, full + p);
            bulk_g2s(dst + 32768, src + 32768, 32768, full + p);
            bulk_g2s(dst + 65536, src + 65536, PKG_BYTES - 65536, full + p);
        }
    }
    // S^T as bf16 operand: row j, K-block g.
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        float o8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o8[e] = st[8 * ch + e];
        *reinterpret_cast<uint4*>(sm + S_ST + g * 16384 + sw128(j, ch)) = pack8(o8);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t tl = tbase + ((uint32_t)lane_base << 16);

    for (int c = 0; c < nc; ++c) {
        const int stage = c & 1;
        uint8_t* stg = sm + (stage ? S_STAGE1 : S_STAGE0);
        const int64_t t0 = bos + (int64_t)c * kC;
        const int len = (int)((eos - t0) < kC ? (eos - t0) : kC);
        bool ok = mbar_wait(full + stage, (c >> 1) & 1);

        // (W S)^T = S^T W^T -> cols [0,64);  (Q^g S)^T -> cols [64,128)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, 64);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                const uint64_t ad = desc_sw128(smem_u32(sm + S_ST + kb * 16384 + off));
                mma_bf16(tbase + 0, ad, desc_sw128(smem_u32(stg + PKG_W + kb * 8192 + off)), idesc,
                         ks > 0);
                mma_bf16(tbase + 64, ad, desc_sw128(smem_u32(stg + PKG_Q + kb * 8192 + off)),
                         idesc, ks > 0);
            }
            mma_commit(mma1);
        }
        ok = mbar_wait(mma1, c & 1) && ok;
        tc_fence_after();

        // U^T = U~^T - (W S)^T for t in [32 g, 32 g + 32)
        {
            float ws32[32];
            tmem_ld16(tl + 32 * g, *reinterpret_cast<float(*)[16]>(ws32));
            tmem_ld16(tl + 32 * g + 16, *reinterpret_cast<float(*)[16]>(ws32 + 16));
            tmem_wait_ld();
            const __nv_bfloat16* ut = reinterpret_cast<const __nv_bfloat16*>(stg + PKG_U);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = 32 * g + 8 * q4 + e;
                    o8[e] = __bfloat162float(ut[t * kD + j]) - ws32[8 * q4 + e];
                }
                *reinterpret_cast<uint4*>(sm + S_UT + sw128(j, 4 * g + q4)) = pack8(o8);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // dS^T = U^T K^C -> cols [128,256);  O^T += U^T P^T -> cols [64,128)
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = desc_sw128(smem_u32(sm + S_UT + ks * 32));
                mma_bf16(tbase + 128, ad, desc_sw128(smem_u32(stg + PKG_KC + ks * 32)),
                         idesc_bf16(128, 128), ks > 0);
                mma_bf16(tbase + 64, ad, desc_sw128(smem_u32(stg + PKG_P + ks * 32)),
                         idesc_bf16(128, 64), true);
            }
            mma_commit(mma2);
        }
        ok = mbar_wait(mma2, c & 1) && ok;
        tc_fence_after();

        // S <- Diag(e^{G_C}) S + dS; refresh the bf16 operand copy of S^T.
        {
            const float* lam = reinterpret_cast<const float*>(stg + PKG_LAM) + 64 * g;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float d16[16];
                tmem_ld16(tl + 128 + 64 * g + 16 * q4, d16);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    st[16 * q4 + e] = fmaf(lam[16 * q4 + e], st[16 * q4 + e], d16[e]);
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float o8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = st[8 * ch + e];
                *reinterpret_cast<uint4*>(sm + S_ST + g * 16384 + sw128(j, ch)) = pack8(o8);
            }
            // o[t, h, j] for t in [32 g, 32 g + 32)
            float o32[32];
            tmem_ld16(tl + 64 + 32 * g, *reinterpret_cast<float(*)[16]>(o32));
            tmem_ld16(tl + 64 + 32 * g + 16, *reinterpret_cast<float(*)[16]>(o32 + 16));
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int t = 32 * g + e;
                if (t < len) o[((size_t)(t0 + t) * H + h) * kD + j] = __float2bfloat16_rn(o32[e]);
            }
        }
        if (!ok) {
            set_status(status, kErrStateWait);
            s_abort = 1;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (s_abort) break;
        if (tid == 0 && c + 2 < nc) {
            const uint8_t* src = pkgs + ((size_t)(slot0 + c + 2) * H + h) * PKG_BYTES;
            mbar_expect_tx(full + stage, PKG_BYTES);
            bulk_g2s(stg, src, 32768, full + stage);
            bulk_g2s(stg + 32768, src + 32768, 32768, full + stage);
            bulk_g2s(stg + 65536, src + 65536, PKG_BYTES - 65536, full + stage);
        }
    }

    if (S1) {
#pragma unroll
        for (int e = 0; e < 64; ++e) S1[sbase + (size_t)(64 * g + e) * kD + j] = st[e];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<256>(tbase);
    }
}

}  // namespace tc

size_t chunked_tc_workspace_bytes(int n_seqs, int64_t T_total, int H) {
    const int64_t slots = T_total / tc::kC + n_seqs + 1;
    return tc::WS_HEADER + (size_t)slots * H * tc::PKG_BYTES;
}

cudaError_t run_chunked_tc(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, void* o, const float* S0, float* S1,
                           const int32_t* cu, int n_seqs, int64_t T, int64_t T_total, int H,
                           void* workspace, cudaStream_t stream, int /*num_sms*/) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(tc::chunk_prep_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)tc::P_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::state_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::S_SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemsetAsync(ws, 0, tc::WS_HEADER, stream);
    if (e != cudaSuccess) return e;
    tc::SeqMap map{cu, T, T_total, n_seqs};
    using bf = __nv_bfloat16;
    profile_event(0, stream);
    const int64_t slots = T_total / tc::kC + n_seqs + 1;
    if (T_total > 0) {
        dim3 grid_p((unsigned)slots, (unsigned)H);
        tc::chunk_prep_kernel<<<grid_p, tc::kThreads, tc::P_SMEM, stream>>>(
            static_cast<const bf*>(q), static_cast<const bf*>(k), static_cast<const bf*>(v),
            static_cast<const bf*>(z), static_cast<const bf*>(beta), A, ws, map, H);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    profile_event(1, stream);
    dim3 grid_s((unsigned)n_seqs, (unsigned)H);
    tc::state_pass_kernel<<<grid_s, tc::kThreads, tc::S_SMEM, stream>>>(
        ws, static_cast<bf*>(o), S0, S1, map, H);
    e = cudaGetLastError();
    profile_event(2, stream);
    return e;
}

}  // namespace kda
