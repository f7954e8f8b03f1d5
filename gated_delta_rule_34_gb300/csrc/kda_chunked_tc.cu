// kda_chunked_tc.cu -- chunked KDA prefill on the sm_103a tensor cores
// (bf16 inputs, chunk C = 64, d_k = d_v = 128; narrower heads -- d_k a
// multiple of 16, d_v a multiple of 32 -- run on the same 128-wide tiles, the
// extra channels arriving as zeros from the input tensor maps).
//
// The pages describe the kernel in outline only: the tokens of a chunk are
// processed in parallel and the state is then passed on across all heads
// ("Kimi K3 architecture: how an open model with a million-token context
// competes with market leaders", section "Chip level: the specialised FlashKDA
// kernel"), and bounding the log-decay below by g_min = -5 keeps every causal
// block a dense matmul with no separate diagonal path ("How Kimi K3 is built:
// 2.8 trillion parameters, linear attention and agents for a million tokens",
// section "Sequence: three KDA to one global MLA").  The algebra is derived
// from the recurrence.  Per (sequence, head) and chunk, with start state S0 and
// G_t = running sum of g from the chunk start:
//
//   A_ts = b_t sum_c k_tc k_sc e^{G_tc - G_sc}  (s < t)    T = (I + A)^{-1}
//   P_ts =     sum_c q_tc k_sc e^{G_tc - G_sc}  (s <= t)
//   W = T Diag(b) K^g,  U~ = T Diag(b) V,       K^g_t = k_t e^{G_t}
//   K^C_s = k_s e^{G_C - G_s},  Q^g_t = q_t e^{G_t}
// and, since U = U~ - W S0, O = Q^g S0 + P U, S_C = Diag(e^{G_C}) S0 + (K^C)^T U:
//   S_C = Diag(lam) S0 - N S0 + X,   N = (K^C)^T W,  X = (K^C)^T U~,  lam = e^{G_C}
//   O   = Q' S0 + O',               Q' = Q^g - P W,  O' = P U~
// Everything but the two products with S0 is independent of the state.
//
// Two kernels:
//   chunk_prep   one CTA (16 warps) per (chunk, head), fully parallel.  Gate,
//                block-local cumulative log-decay, decay-scaled operands, A and
//                P (tcgen05, TMEM), the unit-lower solve for T, W and U~, then N,
//                X, O' and P W (tcgen05).  Writes one 97 KB "package" per
//                (chunk, head): the operand images the state pass feeds to the
//                tensor cores unchanged.
//   state_pass   one CTA per (sequence, head, 32-column tile of S), sequential
//                over its chunks.  The tile lives in fp32 registers; per chunk
//                one tcgen05 product N S (M=128, N=32, K=128) from the bf16
//                copy of the tile's S^T feeds S <- lam (.) S - N S + X, and a
//                second one, Q' S (M=64), runs beside the chain; its result is
//                finished with O' and stored as o.
//
// Decay factoring.  Over 64 tokens G reaches -320, outside fp32/bf16; across
// a 16-token block it spans at most e^80, which fits.  Row t of 16-row block i
// is scaled by e^{G_t - r_i} (<= 1) and column s by e^{r_i - G_s} (<= e^80),
// with r_i = G at the token before block i.  The column operand therefore has
// one variant per row block (K^(i), rows s < 16 (i + 1)); the four products are
// dense M=128 MMAs whose A operand stacks the 64 key rows over the 64 query
// rows.  All exponents are block-local: L_t = G_t - r_{b(t)} comes from a
// 16-token scan, and the block references only enter through per-channel
// factors e^{r_i - r_b}, e^{r_b}, e^{G_C - r_b}.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace tc {

constexpr int kC = 64;        // chunk length
constexpr int kD = 128;       // d_k = d_v

// ---- package: one per (chunk, head), byte offsets -------------------------
// B operand of the state-pass products, per K-block kb (channels 64 kb ..
// 64 kb + 63 of the contraction): rows 0..127 = N[c][c'], rows 128..191 =
// Q'[t][c'].  X and O' are split into four 32-column tiles, one per state
// column tile, each [rows][32] bf16 with 16-byte chunks XOR-permuted by
// (row / 2) mod 4 (see jtile_off).
constexpr uint32_t PKG_B0 = 0;
constexpr uint32_t PKG_BK = 24576;   // bytes per K-block (192 rows x 128 B)
constexpr uint32_t PKG_X = 49152;    // X[c][j]: tile r at PKG_X + 8192 r, [128 c][32 j]
constexpr uint32_t PKG_OP = 81920;   // O'[t][j]: tile r at PKG_OP + 4096 r, [64 t][32 j]
constexpr uint32_t PKG_LAM = 98304;  // lam [c] fp32
constexpr uint32_t PKG_BYTES = 99328;
constexpr uint32_t WS_HEADER = 1024;  // word 0: device status (0 = ok)

// Status bits written to workspace word 0 when a bounded wait gives up.
constexpr uint32_t kErrPrepWait = 1u;
constexpr uint32_t kErrStateWait = 2u;
constexpr uint32_t kErrSmemAlign = 4u;

// ---- chunk_prep ------------------------------------------------------------
constexpr int kPrepThreads = 512;
constexpr int kLoadThread = 480;       // lane 0 of the last warp issues the input copies
// shared memory (offsets from a 1024-byte aligned base).  The package image of
// one item is staged in [0, PKG_BYTES) and stored asynchronously while the next
// item starts: that range only holds buffers the next item first writes after
// its scan (A-stack, K^(i), b K^g, (b V)^T), so the store has time to drain.
constexpr uint32_t R_AST = 0;          // A-stack [128][128] swizzled (k rows, then q rows)
constexpr uint32_t R_KV = 32768;       // K^(i) variants, 40 KB
constexpr uint32_t R_BKT = 73728;      // b K^g [64 s][128 c]: two 64-channel halves, swizzled
constexpr uint32_t R_BVT = 90112;      // (b V)^T  [128 j][64 s] swizzled
constexpr uint32_t R_G = 106496;       // L = block-local cumulative gate, fp32 [64][132];
                                       // also raw z and q of the next item (prefetched)
constexpr uint32_t G_LD = 132;
constexpr uint32_t R_K = 141312;       // raw k [64][128] bf16
constexpr uint32_t R_V = 157696;       // raw v [64][128] bf16
constexpr uint32_t R_KC = 174080;      // K^C [64 s][128 c]: two 64-channel halves, swizzled
constexpr uint32_t R_P = 190464;       // P        [64 t][64 s] swizzled (follows K^C)
constexpr uint32_t R_QG = 198656;      // Q^g      [64 t][128 c] swizzled, two K-blocks
constexpr uint32_t R_SMALL = 215040;   // per-channel constants, beta
constexpr uint32_t R_ZQ = R_G;         // raw z [64][128] bf16, then raw q, of the next item
// reuse after the A/P products
constexpr uint32_t R_AF = 0;           // A fp32 [64][68]
constexpr uint32_t R_TF = 17408;       // T fp32 [64][68]
constexpr uint32_t R_TB = 34816;       // T bf16 [64][64] swizzled
constexpr uint32_t R_XS = 43008;       // solve scratch, 1024 fp32
constexpr uint32_t F_LD = 68;           // fp32 row stride: 16-byte aligned rows, 4-bank skew
// reuse after W / U~ (the solve's buffers and the A/P operands are dead)
constexpr uint32_t R_WT = 0;           // W^T  [128 c][64 s] swizzled
constexpr uint32_t R_UT = 16384;       // U~^T [128 j][64 s] swizzled
constexpr uint32_t R_PKG = 0;          // package image, after the last products
// small region, in floats
constexpr uint32_t SM_TOT = 0;         // [4][128] block totals of g
constexpr uint32_t SM_ER = 512;        // [4][128] e^{r_b}
constexpr uint32_t SM_EC = 1024;       // [4][128] e^{G_C - r_b}
constexpr uint32_t SM_X = 1536;        // [6][128] e^{r_i - r_b}, i > b
constexpr uint32_t SM_LAM = 2304;      // [128] e^{G_C}
constexpr uint32_t SM_B = 2432;        // [64] beta
constexpr uint32_t SM_A = 2496;        // [128] A row of the next item (prefetched)
constexpr uint32_t R_SMALL_BYTES = (2496 + 128) * 4;
constexpr uint32_t kInputBytesZQ = 2 * 16384;        // z, q tiles (the A row adds 4 d_k)
constexpr uint32_t kInputBytesKV = 2 * 16384;        // k, v tiles
constexpr uint32_t R_BAR = R_SMALL + R_SMALL_BYTES;
constexpr uint32_t P_SMEM = R_BAR + 64 + 1024;   // + slack for aligning the base

// K^(i): variant i covers rows s < 16 (i + 1).  The four variants are stacked
// into one 160-row operand (variant i from row d_col(i)), two K-blocks of
// 160 x 128 bytes, so that the four row-block products are one N=160 product.
constexpr uint32_t KV_ROWS = 160;
constexpr uint32_t KV_KB = KV_ROWS * 128;
// TMEM columns of the row-block products D_i (width 16 (i + 1)), which are
// also the first row of variant i in the stacked operand.
__host__ __device__ constexpr uint32_t d_col(int i) {
    return i == 0 ? 0u : i == 1 ? 16u : i == 2 ? 48u : 96u;
}
// Index of the cross factor e^{r_i - r_b} for i > b.
__host__ __device__ constexpr int xidx(int i, int b) {
    return b == 0 ? i - 1 : (b == 1 ? i + 1 : 5);   // (1,0)0 (2,0)1 (3,0)2 (2,1)3 (3,1)4 (3,2)5
}

// ---- state_pass ------------------------------------------------------------
// One CTA per (sequence, head, 32-column tile of S): columns of S evolve
// independently, so four CTAs share a head and each streams only its tiles of
// X and O' plus the shared [N ; Q'] operand.  Warp roles (a warp reaches the
// TMEM lanes 32 (warp mod 4) .. + 31):
//   warps 0-7            update the state: row c = 32 (w mod 4) + lane, columns
//                        16 (w / 4) .. + 15 of the tile;
//   warps 8-11           write the outputs: the O product is M=64, whose row t
//                        sits in TMEM lane 32 (t / 16) + t mod 16, so lanes
//                        0..15 of warp 8 + t / 16 hold token t;
//   warp 12              issues the S product (on the chain from one chunk's
//                        update to the next);
//   warp 13              issues the O product once the S product is done, so
//                        that it never delays the chain;
//   warp 14              issues the package copies.
// The tensor pipe accepts a small-N tcgen05.mma only every ~50 cycles, so the
// chain's floor is about eight of those plus the update.
constexpr int kStateThreads = 32 * 15;
constexpr int kUpdWarps = 8, kOutWarps = 4;
constexpr int kJ = 32;                             // state columns per tile
constexpr int kStages = 4;
constexpr uint32_t ST_BYTES = 49152;               // per stage: [N ; Q'], both K-blocks
constexpr uint32_t S_ST = kStages * ST_BYTES;      // 2 x S^T tile [32 j][128 c] bf16 (2 K-blocks of 4 KB)
constexpr uint32_t S_BAR = S_ST + 2 * 8192;
constexpr uint32_t S_SMEM = S_BAR + 256;           // the dynamic base is 1024-aligned
constexpr uint32_t kDBuf = 64;                     // per accumulator buffer: D_S, then D_O at +32
constexpr uint32_t kTmemCols = 2 * kDBuf;
constexpr int kL2Ahead = 6;                        // packages prefetched into L2 this far ahead

static_assert(S_SMEM <= 232448, "state_pass shared memory");
static_assert(P_SMEM <= 232448, "chunk_prep shared memory");
static_assert(R_TF + 64 * F_LD * 4 <= R_TB && R_XS + 1024 * 4 <= R_BKT, "solve scratch");
static_assert(R_UT + 16384 <= R_BKT && R_PKG + PKG_BYTES <= R_G, "reuse regions");
static_assert(R_G + 64 * G_LD * 4 <= R_K && R_P == R_KC + 16384, "layout");

// Sequences of one launch.  A launch covers a window of tokens: for a
// fixed-length batch, positions [w0, w1) of every sequence (window edges are
// multiples of 64); for a packed one, the chunks of each sequence whose first
// row lies in rows [w0, w1) of the packed tensor, chunks being counted from the
// sequence's own start (so a sequence's last chunk in a window may reach up to
// 63 rows past w1, and checkpoints keep falling on chunk ends).  The state
// carries over between windows.
struct SeqMap {
    const int32_t* cu;  // nullable
    int64_t T;          // per-sequence length when cu == nullptr
    int64_t T_total;    // token rows of the input tensors
    int n_seqs;
    int64_t w0, w1;     // the window
};

// The rows of sequence n inside the window, [bos, eos), and its first row
// bos_seq.  Returns the sequence's first package slot, floor(p / 64) + n with p
// = bos counted from the window's start (packed; at least 0) or n (w1 - w0)
// (fixed length): slots of different sequences never overlap, and every slot
// is below floor(window tokens / 64) + n_seqs + 1 (for a packed window of
// 64-multiple length the overhang of the last chunks fits: the last slot is at
// most floor((w1 - w0 + 126) / 64) - 1 + (n_seqs - 1)).
__device__ __forceinline__ int64_t seq_slot_base(const SeqMap& m, int n, int64_t& bos,
                                                 int64_t& eos, int64_t& bos_seq) {
    if (m.cu) {
        int64_t b, e;
        seq_bounds(m.cu, n, m.T, m.T_total, b, e);
        bos_seq = b;
        // first chunk start of the sequence at or after row w (chunks from b)
        auto align = [&](int64_t w) { return w <= b ? b : b + (w - b + kC - 1) / kC * kC; };
        const int64_t lo = align(m.w0), hi = align(m.w1);
        bos = lo < e ? lo : e;
        eos = hi < e ? hi : e;
        if (eos < bos) eos = bos;
        return ((bos > m.w0 ? bos : m.w0) - m.w0) / kC + n;
    }
    bos_seq = (int64_t)n * m.T;
    bos = bos_seq + m.w0;
    eos = bos_seq + m.w1;
    return (int64_t)n * (m.w1 - m.w0) / kC + n;
}
__device__ __forceinline__ int64_t seq_slot_base(const SeqMap& m, int n, int64_t& bos,
                                                 int64_t& eos) {
    int64_t bos_seq;
    return seq_slot_base(m, n, bos, eos, bos_seq);
}

// Byte offset of 16-byte chunk q (0..3) of row `row` in a [rows][32] bf16 tile.
__host__ __device__ __forceinline__ uint32_t jtile_off(uint32_t row, uint32_t q) {
    return row * 64u + (((q ^ (row >> 1)) & 3u) << 4);
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

__device__ __forceinline__ void load8f(const float* p, float (&f)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// The same 8 floats, for rows where the 8 lanes of a quarter-warp read
// consecutive 32-byte pieces: lanes with `swap` take their upper half first,
// so that each of the two 16-byte loads touches 8 distinct bank groups.
__device__ __forceinline__ void load8f_sw(const float* p, float (&f)[8], bool swap) {
    const float4 a = reinterpret_cast<const float4*>(p)[swap ? 1 : 0];
    const float4 b = reinterpret_cast<const float4*>(p)[swap ? 0 : 1];
    const float4 lo = swap ? b : a, hi = swap ? a : b;
    f[0] = lo.x; f[1] = lo.y; f[2] = lo.z; f[3] = lo.w;
    f[4] = hi.x; f[5] = hi.y; f[6] = hi.z; f[7] = hi.w;
}
__device__ __forceinline__ void store8f_sw(float* p, const float (&f)[8], bool swap) {
    const float4 lo = make_float4(f[0], f[1], f[2], f[3]), hi = make_float4(f[4], f[5], f[6], f[7]);
    reinterpret_cast<float4*>(p)[swap ? 1 : 0] = swap ? hi : lo;
    reinterpret_cast<float4*>(p)[swap ? 0 : 1] = swap ? lo : hi;
}

// Copies TMEM columns [col0, col0 + 16 N16) of this thread's lane, as bf16,
// into row `row` of a swizzled K-major tile (atoms 1024-aligned): column
// col0 + x becomes element x of the row; elements 64 kb .. 64 kb + 63 sit in
// K-block kb, `kb_stride` bytes after the first.
template <int N16>
__device__ __forceinline__ void tmem_row_to_tile(uint32_t taddr, uint8_t* tile_kb0,
                                                 uint32_t kb_stride, uint32_t row) {
#pragma unroll
    for (int q = 0; q < N16; ++q) {
        float v[16];
        tmem_ld16(taddr + 16u * q, v);
        tmem_wait_ld();
        uint4 lo, hi;
        lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[2], v[3]);
        lo.z = pack_bf16x2(v[4], v[5]);   lo.w = pack_bf16x2(v[6], v[7]);
        hi.x = pack_bf16x2(v[8], v[9]);   hi.y = pack_bf16x2(v[10], v[11]);
        hi.z = pack_bf16x2(v[12], v[13]); hi.w = pack_bf16x2(v[14], v[15]);
        const uint32_t chunk = 2u * q;                     // element 16 q = chunk 2 q
        uint8_t* base = tile_kb0 + (chunk >> 3) * kb_stride;
        *reinterpret_cast<uint4*>(base + sw128(row, chunk & 7)) = lo;
        *reinterpret_cast<uint4*>(base + sw128(row, (chunk & 7) + 1)) = hi;
    }
}

// T = (I + A)^{-1} for the strictly lower 64 x 64 A (fp32, row stride F_LD):
// the four 16 x 16 diagonal blocks by forward substitution (one thread per
// block column), then for n = 16, 32 each 2n x 2n diagonal block
// [T11 0; T21 T22] from its halves by T21 = -T22 (A21 T11), with the n x n
// scratch X = A21 T11.  Every fp32 T entry that a later level reads is
// written first, zeros above the diagonal included.  The last level writes its
// T21 straight into the bf16 image of T; the other warps image the two
// diagonal 32 x 32 blocks (and the zero block above T21) once named barrier 4
// says they are final.  Run by the first kSolveThreads threads, which
// synchronise among themselves on named barrier 1.
constexpr int kSolveThreads = 256;

// acc[0..3] += sum_{m < n} row[m] * M[m][0..3], with M's rows `ld` floats
// apart; the row's values are loaded first and M's rows in batches of eight,
// so that each batch's loads are in flight together.
template <int n>
__device__ __forceinline__ float4 row_times_block(const float* __restrict__ row,
                                                  const float* __restrict__ M, int ld) {
    float r[n];
#pragma unroll
    for (int m4 = 0; m4 < n; m4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(row + m4);
        r[m4] = a.x; r[m4 + 1] = a.y; r[m4 + 2] = a.z; r[m4 + 3] = a.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kB = n < 8 ? n : 8;
#pragma unroll
    for (int m0 = 0; m0 < n; m0 += kB) {
        float4 t[kB];
#pragma unroll
        for (int e = 0; e < kB; ++e) t[e] = *reinterpret_cast<const float4*>(M + (m0 + e) * ld);
#pragma unroll
        for (int e = 0; e < kB; ++e) {
            const float a = r[m0 + e];
            acc.x = fmaf(a, t[e].x, acc.x); acc.y = fmaf(a, t[e].y, acc.y);
            acc.z = fmaf(a, t[e].z, acc.z); acc.w = fmaf(a, t[e].w, acc.w);
        }
    }
    return acc;
}

template <int n>
__device__ __forceinline__ void solve_level(const float* __restrict__ Af, float* Tf, float* Xs,
                                            int tid) {
    // A thread computes four adjacent entries (row i, columns j .. j + 3):
    // lane = (pair p, row i), warp = column group, so the T (or X) row that a
    // warp reads at step m is the same for all lanes of a pair (a broadcast)
    // and the rows of A (or T22) are spread over the lanes.
    constexpr int kThreads = 8 * n;                      // n / 4 warps
    static_assert(kThreads <= kSolveThreads, "solve threads");
    const int lane = tid & 31;
    const int p = lane / n, i = lane % n, j = 4 * (tid >> 5);
    const int e0 = (p * n + i) * n + j;
    const int base = 2 * n * p;
    if (tid < kThreads) {
        // X[i][j..j+3] = sum_m A21[i][m] T11[m][j..j+3]
        const float4 acc = row_times_block<n>(Af + (base + n + i) * F_LD + base,
                                              Tf + base * F_LD + base + j, F_LD);
        *reinterpret_cast<float4*>(Xs + e0) = acc;
    }
    named_bar_sync(1, kSolveThreads);
    if (tid < kThreads) {
        // T21[i][j..j+3] = -sum_m T22[i][m] X[m][j..j+3]; T12 = 0
        const float4 acc = row_times_block<n>(Tf + (base + n + i) * F_LD + base + n,
                                              Xs + p * n * n + j, n);
        *reinterpret_cast<float4*>(Tf + (base + n + i) * F_LD + base + j) =
            make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        *reinterpret_cast<float4*>(Tf + (base + i) * F_LD + base + n + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    named_bar_sync(1, kSolveThreads);
}

// The last level (n = 32, one pair) with 4 x 4 register tiles and the
// 32-term sums split four ways inside a warp: warp w takes rows 4w .. 4w + 3,
// lane (kg, jt) columns 4 jt .. 4 jt + 3 and terms 8 kg .. 8 kg + 7, so that
// each pair of 16-byte loads feeds sixteen FMAs.  The four partial tiles are
// added with shuffles across kg, and lane kg stores row kg of the tile.  The
// eight lanes of a quarter warp share kg: they read one A (or T22) row
// segment (a broadcast) and 128 contiguous bytes of T11 (or X).
__device__ __forceinline__ void tile4x4_part(float (&acc)[4][4], const float* __restrict__ a, int lda,
                                             const float* __restrict__ b, int ldb) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll
    for (int m4 = 0; m4 < 8; m4 += 4) {
        float ar[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float4 v = *reinterpret_cast<const float4*>(a + r * lda + m4);
            ar[r][0] = v.x; ar[r][1] = v.y; ar[r][2] = v.z; ar[r][3] = v.w;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 bv = *reinterpret_cast<const float4*>(b + (m4 + e) * ldb);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[r][0] = fmaf(ar[r][e], bv.x, acc[r][0]);
                acc[r][1] = fmaf(ar[r][e], bv.y, acc[r][1]);
                acc[r][2] = fmaf(ar[r][e], bv.z, acc[r][2]);
                acc[r][3] = fmaf(ar[r][e], bv.w, acc[r][3]);
            }
        }
    }
}

// Sums the tile over the four kg lanes (lane bits 3 and 4) and returns row kg.
__device__ __forceinline__ float4 tile4x4_reduce_row(float (&acc)[4][4], int kg) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            acc[r][c] += __shfl_xor_sync(0xffffffffu, acc[r][c], 8);
            acc[r][c] += __shfl_xor_sync(0xffffffffu, acc[r][c], 16);
        }
    float4 out = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
#pragma unroll
    for (int r = 1; r < 4; ++r)
        if (kg == r) out = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    return out;
}

__device__ __forceinline__ void solve_level32(const float* __restrict__ Af, float* Tf, float* Xs,
                                              uint8_t* Tb, int tid) {
    constexpr int n = 32;
    const int lane = tid & 31, kg = lane >> 3;
    const int i0 = 4 * (tid >> 5), j0 = 4 * (lane & 7), m0 = 8 * kg;
    float acc[4][4];
    // X = A21 T11
    tile4x4_part(acc, Af + (n + i0) * F_LD + m0, F_LD, Tf + m0 * F_LD + j0, F_LD);
    *reinterpret_cast<float4*>(Xs + (i0 + kg) * n + j0) = tile4x4_reduce_row(acc, kg);
    named_bar_sync(1, kSolveThreads);
    // T21 = -T22 X, straight into the bf16 image Tb (the other blocks of the
    // image are written by the other warps)
    tile4x4_part(acc, Tf + (n + i0) * F_LD + n + m0, F_LD, Xs + m0 * n + j0, n);
    const float4 x = tile4x4_reduce_row(acc, kg);
    const int r = n + i0 + kg;
    *reinterpret_cast<uint2*>(Tb + sw128(r, j0 >> 3) + (j0 & 7) * 2) =
        make_uint2(pack_bf16x2(-x.x, -x.y), pack_bf16x2(-x.z, -x.w));
}

__device__ __forceinline__ void solve_unit_lower(const float* __restrict__ Af, float* Tf,
                                                 float* Xs, uint8_t* Tb, int tid) {
    if (tid < 64) {
        // column j of the 16 x 16 diagonal block k: x_r = -sum_{m<r} A_rm x_m
        // below the unit entry, 0 above it.  The lanes of a block read the same
        // A row (a broadcast).
        const int k = tid >> 4, j = tid & 15;
        const float* ab = Af + 16 * k * F_LD + 16 * k;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a[16];
#pragma unroll
            for (int m4 = 0; m4 < r; m4 += 4) {
                const float4 v = *reinterpret_cast<const float4*>(ab + r * F_LD + m4);
                a[m4] = v.x; a[m4 + 1] = v.y; a[m4 + 2] = v.z; a[m4 + 3] = v.w;
            }
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc = fmaf(a[m], x[m], acc);
            x[r] = (r < j) ? 0.f : (r == j ? 1.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(16 * k + r) * F_LD + 16 * k + j] = x[r];
    }
    named_bar_sync(1, kSolveThreads);
    solve_level<16>(Af, Tf, Xs, tid);
    // The diagonal 32 x 32 blocks are final: the other warps image them.
    named_bar_arrive(4, kPrepThreads);
    solve_level32(Af, Tf, Xs, Tb, tid);
}

// Which chunk package slot `slot` holds: its first token t0 and length.
// False for slots that hold no chunk (the slot space has a few spares).
__device__ __forceinline__ bool slot_chunk(const SeqMap& map, int64_t slot, int64_t& t0, int& len) {
    int lo = 0, hi = map.n_seqs - 1;
    int64_t bos, eos;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seq_slot_base(map, mid, bos, eos) <= slot) lo = mid; else hi = mid - 1;
    }
    const int64_t chunk = slot - seq_slot_base(map, lo, bos, eos);
    const int64_t n_chunks = (eos - bos + kC - 1) / kC;
    if (chunk < 0 || chunk >= n_chunks) return false;
    t0 = bos + chunk * kC;
    len = (int)((eos - t0) < kC ? (eos - t0) : kC);
    return true;
}

// Copies TMEM columns [col, col + 32) of this thread's lane, as bf16, into
// 16-byte chunks chunk0 .. chunk0 + 3 of row `row` of a 128-byte-swizzled
// K-major tile.
__device__ __forceinline__ void tmem32_to_swizzled(uint32_t taddr, uint8_t* tile, uint32_t row,
                                                   uint32_t chunk0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float v[16];
        tmem_ld16(taddr + 16u * q, v);
        tmem_wait_ld();
        uint4 lo, hi;
        lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[2], v[3]);
        lo.z = pack_bf16x2(v[4], v[5]);   lo.w = pack_bf16x2(v[6], v[7]);
        hi.x = pack_bf16x2(v[8], v[9]);   hi.y = pack_bf16x2(v[10], v[11]);
        hi.z = pack_bf16x2(v[12], v[13]); hi.w = pack_bf16x2(v[14], v[15]);
        *reinterpret_cast<uint4*>(tile + sw128(row, chunk0 + 2 * q)) = lo;
        *reinterpret_cast<uint4*>(tile + sw128(row, chunk0 + 2 * q + 1)) = hi;
    }
}

// Copies TMEM columns [col, col + 32) of this thread's lane, as bf16, into
// row `row` of one [rows][32] tile.
__device__ __forceinline__ void tmem32_to_jtile(uint32_t taddr, uint8_t* tile, uint32_t row) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float v[16];
        tmem_ld16(taddr + 16u * q, v);
        tmem_wait_ld();
        uint4 lo, hi;
        lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[2], v[3]);
        lo.z = pack_bf16x2(v[4], v[5]);   lo.w = pack_bf16x2(v[6], v[7]);
        hi.x = pack_bf16x2(v[8], v[9]);   hi.y = pack_bf16x2(v[10], v[11]);
        hi.z = pack_bf16x2(v[12], v[13]); hi.w = pack_bf16x2(v[14], v[15]);
        *reinterpret_cast<uint4*>(tile + jtile_off(row, 2 * q)) = lo;
        *reinterpret_cast<uint4*>(tile + jtile_off(row, 2 * q + 1)) = hi;
    }
}

// As tmem32_to_jtile, with the columns of each 16-column group stored in the
// order 0 1 8 9 2 3 10 11 | 4 5 12 13 6 7 14 15, so that a reader holding
// columns 2w, 2w + 1, 8 + 2w, 9 + 2w (the 16x256b fragment layout) finds them
// in 8 contiguous bytes.  Used for the X tiles.
__device__ __forceinline__ void tmem32_to_jtile_pairs(uint32_t taddr, uint8_t* tile, uint32_t row) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float v[16];
        tmem_ld16(taddr + 16u * q, v);
        tmem_wait_ld();
        uint4 lo, hi;
        lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[8], v[9]);
        lo.z = pack_bf16x2(v[2], v[3]);   lo.w = pack_bf16x2(v[10], v[11]);
        hi.x = pack_bf16x2(v[4], v[5]);   hi.y = pack_bf16x2(v[12], v[13]);
        hi.z = pack_bf16x2(v[6], v[7]);   hi.w = pack_bf16x2(v[14], v[15]);
        *reinterpret_cast<uint4*>(tile + jtile_off(row, 2 * q)) = lo;
        *reinterpret_cast<uint4*>(tile + jtile_off(row, 2 * q + 1)) = hi;
    }
}

// Copies TMEM columns [col0, col0 + 128) of this thread's lane, as bf16, into
// row `row` of four [rows][32] tiles `tile_bytes` apart (columns 32 r .. 32 r
// + 31 go to tile r).
__device__ __forceinline__ void tmem_row_to_jtiles(uint32_t taddr, uint8_t* tile0,
                                                   uint32_t tile_bytes, uint32_t row) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float v[16];
        tmem_ld16(taddr + 16u * q, v);
        tmem_wait_ld();
        uint4 lo, hi;
        lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[2], v[3]);
        lo.z = pack_bf16x2(v[4], v[5]);   lo.w = pack_bf16x2(v[6], v[7]);
        hi.x = pack_bf16x2(v[8], v[9]);   hi.y = pack_bf16x2(v[10], v[11]);
        hi.z = pack_bf16x2(v[12], v[13]); hi.w = pack_bf16x2(v[14], v[15]);
        uint8_t* t = tile0 + (q >> 1) * tile_bytes;            // 16 q .. 16 q + 15 in tile q / 2
        const uint32_t c0 = (q & 1) * 2;
        *reinterpret_cast<uint4*>(t + jtile_off(row, c0)) = lo;
        *reinterpret_cast<uint4*>(t + jtile_off(row, c0 + 1)) = hi;
    }
}

// Input tensor maps: q, k, v, z as 3-D tensors [T_total][H][128] bf16 with
// boxes of 64 tokens x 1 head x 128 channels (16 KB, rows at 256-byte pitch
// in shared memory); boxes past the last token read zeros.
struct InputMaps {
    CUtensorMap q, k, v, z;
};

// One thread issues the loads of an item's inputs, q, k, v, z tiles by TMA
// and the A row by a bulk copy, in two groups: z, q and A (read first)
// complete on `inbar`, k and v on `kvbar`.  Rows past the item's `len` belong
// to the next sequence (or are zero); the consumers mask them.
__device__ __forceinline__ void issue_item_zq(uint8_t* sm, const InputMaps& maps,
                                              const float* __restrict__ A, int64_t t0, int h,
                                              int dk, uint64_t* inbar) {
    mbar_expect_tx(inbar, kInputBytesZQ + 4u * (uint32_t)dk);
    tma_load_3d(sm + R_ZQ, &maps.z, 0, h, (int)t0, inbar);
    tma_load_3d(sm + R_ZQ + 16384, &maps.q, 0, h, (int)t0, inbar);
    bulk_g2s(sm + R_SMALL + SM_A * 4, A + (size_t)h * dk, 4u * (uint32_t)dk, inbar);
}
__device__ __forceinline__ void issue_item_kv(uint8_t* sm, const InputMaps& maps, int64_t t0, int h,
                                              uint64_t* kvbar) {
    mbar_expect_tx(kvbar, kInputBytesKV);
    tma_load_3d(sm + R_K, &maps.k, 0, h, (int)t0, kvbar);
    tma_load_3d(sm + R_V, &maps.v, 0, h, (int)t0, kvbar);
}

// beta's raw bits for threads < 64, converted only when the item starts so
// that the load stays in flight meanwhile.
__device__ __forceinline__ uint32_t load_beta_raw(const __nv_bfloat16* __restrict__ beta,
                                                  int64_t t0, int len, int h, int H, int tid) {
    uint32_t r = 0u;
    if (tid < kC && tid < len) r = reinterpret_cast<const unsigned short*>(beta)[(size_t)(t0 + tid) * H + h];
    return r;
}

// ============================================================================
// chunk_prep: persistent.  Each CTA walks the (package slot, head) items
// blockIdx.x, blockIdx.x + gridDim.x, ... with item = slot * H + head.
// ============================================================================
__global__ void __launch_bounds__(kPrepThreads, 1)
chunk_prep_kernel(const __grid_constant__ InputMaps maps, const __nv_bfloat16* __restrict__ beta,
                  const float* __restrict__ A, uint8_t* __restrict__ ws, SeqMap map, int H, int dk,
                  int64_t n_items) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Offset from the array (not an integer cast) so that the compiler keeps
    // every access below in the shared window.
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* G = reinterpret_cast<float*>(sm + R_G);
    float* small = reinterpret_cast<float*>(sm + R_SMALL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + R_BAR);
    uint64_t* inbar = bar + 1;
    uint64_t* bar2 = bar + 2;               // second half of the last products
    uint64_t* kvbar = bar + 3;              // k, v tiles of the item
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + R_BAR + 32);
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);

    if (warp == 0) tmem_alloc<512>(tslot);
    // Channels d_k .. 127 of a narrower head: the input tiles arrive
    // zero-filled there (the tensor maps are d_k wide), and the A row entries,
    // which the copies never write, are set to 0 once so that those channels
    // stay finite; with k = q = 0 they contribute nothing.
    if (tid >= dk && tid < kD) small[SM_A + tid] = 0.f;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(inbar, 1);
        mbar_init(bar2, 1);
        mbar_init(kvbar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    uint32_t phase = 0;                      // parity of the next completion of `bar`
    uint32_t in_phase = 0;                   // parity of the next completion of `inbar`
    uint32_t phase2 = 0;                     // parity of the next completion of `bar2`
    uint32_t kv_phase = 0;                   // parity of the next completion of `kvbar`
    bool ok = true;
    const int c8 = tid & 15;                 // channels 8 c8 .. 8 c8 + 7 in the row-side passes

    // The first item's inputs; later items' inputs are issued one item ahead.
    // item = slot * H + head, walked as (slot, head) so that no 64-bit
    // division is left in the loop.
    const int step_slot = (int)(gridDim.x / (unsigned)H), step_head = (int)(gridDim.x % (unsigned)H);
    auto advance = [&](int64_t& it, int64_t& sl, int& hd) {
        it += gridDim.x;
        sl += step_slot;
        hd += step_head;
        if (hd >= H) { hd -= H; ++sl; }
    };
    int64_t item = blockIdx.x, slot = blockIdx.x / (unsigned)H;
    int head = (int)(blockIdx.x % (unsigned)H);
    int64_t t0 = 0;
    int len = 0;
    uint32_t bt_raw = 0u;
    while (item < n_items && !slot_chunk(map, slot, t0, len)) advance(item, slot, head);
    if (item < n_items) {
        if (tid == kLoadThread) {
            issue_item_zq(sm, maps, A, t0, head, dk, inbar);
            issue_item_kv(sm, maps, t0, head, kvbar);
        }
        bt_raw = load_beta_raw(beta, t0, len, head, H, tid);
    }

    while (item < n_items) {
        uint8_t* pkg = ws + WS_HEADER + (size_t)item * PKG_BYTES;
        // The next item this CTA processes (skipping slots that hold no chunk).
        int64_t nitem = item, nslot = slot, nt0 = 0;
        int nhead = head, nlen = 0;
        advance(nitem, nslot, nhead);
        while (nitem < n_items && !slot_chunk(map, nslot, nt0, nlen)) advance(nitem, nslot, nhead);

        // ---- inputs of this item (issued during the previous one) -> registers
        ok = mbar_wait(inbar, in_phase) && ok;
        in_phase ^= 1u;
        __syncthreads();
        int tt[2];
        uint4 qraw[2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            // tokens r and 63 - r: blocks b and 3 - b, so that every thread
            // writes the same number of K^(i) variants (4 - b of them) below
            tt[it] = it == 0 ? (tid >> 4) : 63 - (tid >> 4);
            qraw[it] = tt[it] < len
                           ? *reinterpret_cast<const uint4*>(sm + R_ZQ + 16384 + tt[it] * 256 + c8 * 16)
                           : make_uint4(0, 0, 0, 0);
        }
        // Gate and scan are fused, thread = (channel pair gc, gc + 1; tokens
        // 16 gb + 8 hb .. + 7): z of those tokens and channels is read before G
        // (which overlays the raw z and q tiles) is written.
        const int hb = tid & 1, gc = 2 * ((tid >> 1) & 63), gb = tid >> 7;
        uint32_t zc[8];
        {
            const uint32_t* zr = reinterpret_cast<const uint32_t*>(sm + R_ZQ);
#pragma unroll
            for (int i = 0; i < 8; ++i) zc[i] = zr[(16 * gb + 8 * hb + i) * (kD / 2) + (gc >> 1)];
        }
        const float eA0 = __expf(small[SM_A + gc]), eA1 = __expf(small[SM_A + gc + 1]);
        if (tid < kC) small[SM_B + tid] = __uint_as_float(bt_raw << 16);   // bf16 -> fp32
        __syncthreads();                         // raw z, q are read before G is written

        // ---- gate g = -5 sigmoid(e^A z) (0 on padded rows) and the block-local
        //      cumulative log-decay L_t = G_t - r_b (16-token scans), then the
        //      per-channel block factors from the block totals.
        {
            // Each half-block scans its 8 tokens; the second half then adds the
            // first half's total (from the neighbouring lane).
            float s0[8], s1[8], run0 = 0.f, run1 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const bool in = 16 * gb + 8 * hb + i < len;
                const float2 zz = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&zc[i]));
                run0 += in ? gate_fast(eA0, zz.x) : 0.f;
                run1 += in ? gate_fast(eA1, zz.y) : 0.f;
                s0[i] = run0;
                s1[i] = run1;
            }
            const float p0 = __shfl_xor_sync(0xffffffffu, run0, 1);
            const float p1 = __shfl_xor_sync(0xffffffffu, run1, 1);
            const float a0 = hb ? p0 : 0.f, a1 = hb ? p1 : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float2*>(G + (16 * gb + 8 * hb + i) * G_LD + gc) =
                    make_float2(s0[i] + a0, s1[i] + a1);
            if (hb) {
                small[SM_TOT + gb * 128 + gc] = run0 + a0;
                small[SM_TOT + gb * 128 + gc + 1] = run1 + a1;
            }
            __syncthreads();
            const int c = tid & 127, b = tid >> 7;
            const float t0v = small[SM_TOT + c], t1v = small[SM_TOT + 128 + c];
            const float t2v = small[SM_TOT + 256 + c], t3v = small[SM_TOT + 384 + c];
            const float r1 = t0v, r2 = t0v + t1v, r3 = r2 + t2v, rc = r3 + t3v;
            if (b == 0) {
                small[SM_ER + 0 * 128 + c] = 1.f;
                small[SM_ER + 1 * 128 + c] = __expf(r1);
                small[SM_ER + 2 * 128 + c] = __expf(r2);
                small[SM_ER + 3 * 128 + c] = __expf(r3);
            } else if (b == 1) {
                small[SM_EC + 0 * 128 + c] = __expf(rc);
                small[SM_EC + 1 * 128 + c] = __expf(rc - r1);
                small[SM_EC + 2 * 128 + c] = __expf(rc - r2);
                small[SM_EC + 3 * 128 + c] = __expf(rc - r3);
            } else if (b == 2) {
                small[SM_X + xidx(1, 0) * 128 + c] = __expf(r1);
                small[SM_X + xidx(2, 0) * 128 + c] = __expf(r2);
                small[SM_X + xidx(3, 0) * 128 + c] = __expf(r3);
                small[SM_LAM + c] = __expf(rc);
            } else {
                small[SM_X + xidx(2, 1) * 128 + c] = __expf(r2 - r1);
                small[SM_X + xidx(3, 1) * 128 + c] = __expf(r3 - r1);
                small[SM_X + xidx(3, 2) * 128 + c] = __expf(r3 - r2);
            }
            // The previous item's package store must have read the staging area
            // before the row-side pass overwrites it.
            if (tid == 0) bulk_wait_read_all();
            ok = mbar_wait(kvbar, kv_phase) && ok;          // k, v of this item
            kv_phase ^= 1u;
            __syncthreads();
        }

        // ---- operands from the token rows (thread = token t, 8 channels): first
        //      the two of the A/P product, then (below, while it runs) Q^g and
        //      the key-side operands of the later products, K^C and b K^g, also
        //      as token rows: their MMAs read them MN-major, so no transposed
        //      copy is built.
        const int kb = c8 >> 3, chk = c8 & 7;
        const bool sw = (c8 >> 2) & 1;
        float E[2][8], Rr[2][8];                 // e^{G_t - r_b} in [e^-80, 1], its inverse
        uint4 kraw[2];
        {
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                const int t = tt[it], b = t >> 4;
                float Lt[8], kf[8], qf[8], o8[8];
                load8f_sw(G + t * G_LD + c8 * 8, Lt, sw);
                kraw[it] = t < len ? *reinterpret_cast<const uint4*>(sm + R_K + t * 256 + c8 * 16)
                                   : make_uint4(0, 0, 0, 0);
                unpack8(kraw[it], kf);
                unpack8(qraw[it], qf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    E[it][e] = __expf(Lt[e]);
                    Rr[it][e] = __fdividef(1.0f, E[it][e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = kf[e] * E[it][e];
                *reinterpret_cast<uint4*>(sm + R_AST + kb * 16384 + sw128(t, chk)) = pack8(o8);
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[it][e];
                *reinterpret_cast<uint4*>(sm + R_AST + kb * 16384 + sw128(64 + t, chk)) = pack8(o8);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < b) continue;
                    float x[8];
                    if (i == b) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = 1.f;
                    } else {
                        load8f_sw(small + SM_X + xidx(i, b) * 128 + c8 * 8, x, sw);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) o8[e] = kf[e] * Rr[it][e] * x[e];  // k e^{r_i - G_t}
                    *reinterpret_cast<uint4*>(sm + R_KV + kb * KV_KB + sw128(d_col(i) + t, chk)) =
                        pack8(o8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- A and P: the row-block products D_i = Astack * K^(i)^T, as one
        //      N=160 product into TMEM columns [0, 160).  G and the raw z, q
        //      are dead: the next item's z, q and A row start loading now.
        if (tid == kLoadThread && nitem < n_items) issue_item_zq(sm, maps, A, nt0, nhead, dk, inbar);
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16(128, KV_ROWS);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                const uint64_t ad = desc_sw128(smem_u32(sm + R_AST + kb * 16384 + off));
                const uint64_t bd = desc_sw128(smem_u32(sm + R_KV + kb * KV_KB + off));
                mma_bf16(tbase, ad, bd, idesc, ks > 0);
            }
            mma_commit(bar);
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int t = tt[it], b = t >> 4;
            float kf[8], qf[8], er[8], ec[8], o8[8];
            load8f_sw(small + SM_ER + b * 128 + c8 * 8, er, sw);
            load8f_sw(small + SM_EC + b * 128 + c8 * 8, ec, sw);
            unpack8(kraw[it], kf);
            unpack8(qraw[it], qf);
            const float bt = small[SM_B + t];
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = qf[e] * E[it][e] * er[e];          // q e^{G_t}
            *reinterpret_cast<uint4*>(sm + R_QG + kb * 8192 + sw128(t, chk)) = pack8(o8);
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = kf[e] * Rr[it][e] * ec[e];         // k e^{G_C - G_t}
            *reinterpret_cast<uint4*>(sm + R_KC + kb * 8192 + sw128(t, chk)) = pack8(o8);
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = bt * kf[e] * E[it][e] * er[e];     // b k e^{G_t}
            *reinterpret_cast<uint4*>(sm + R_BKT + kb * 8192 + sw128(t, chk)) = pack8(o8);
        }

        ok = mbar_wait(bar, phase) && ok;
        phase ^= 1u;
        tc_fence_after();

        // Readback of A (key rows, TMEM lanes 0..63) and P (query rows, lanes
        // 64..127): warp w covers the lanes of quadrant w mod 4 and output
        // columns 16 (w / 4) .. + 15.  Lanes 0..15 and 16..31 of a warp hold
        // rows of two different 16-row blocks, so the warp loads both blocks'
        // column slices and each lane keeps its own.
        {
            const int q = warp & 3, s0 = 16 * (warp >> 2);
            const int t = (32 * q + lane) & 63, blk = t >> 4;
            const int b0 = 2 * (q & 1), b1 = b0 + 1;
            const uint32_t taddr = tbase + ((uint32_t)(32 * q) << 16);
            float v0[16], v1[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) { v0[e] = 0.f; v1[e] = 0.f; }
            if (s0 < 16 * (b0 + 1)) tmem_ld16(taddr + d_col(b0) + s0, v0);   // D_b has 16 (b+1) columns
            if (s0 < 16 * (b1 + 1)) tmem_ld16(taddr + d_col(b1) + s0, v1);
            tmem_wait_ld();
            const bool lo = blk == b0;
            const bool valid = s0 < 16 * (blk + 1);
            if (q < 2) {
                const float bt = small[SM_B + t];
                float* Af = reinterpret_cast<float*>(sm + R_AF);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    float o4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = s0 + 4 * s4 + e;
                        const float val = lo ? v0[4 * s4 + e] : v1[4 * s4 + e];
                        o4[e] = (valid && s < t) ? bt * val : 0.f;
                    }
                    *reinterpret_cast<float4*>(Af + t * F_LD + s0 + 4 * s4) =
                        make_float4(o4[0], o4[1], o4[2], o4[3]);
                }
            } else {
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    float o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = s0 + 8 * h8 + e;
                        const float val = lo ? v0[8 * h8 + e] : v1[8 * h8 + e];
                        o8[e] = (valid && s <= t) ? val : 0.f;
                    }
                    *reinterpret_cast<uint4*>(sm + R_P + sw128(t, (s0 >> 3) + h8)) = pack8(o8);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (nitem < n_items) bt_raw = load_beta_raw(beta, nt0, nlen, nhead, H, tid);

        // ---- T = (I + A)^{-1}
        {
            const float* Af = reinterpret_cast<const float*>(sm + R_AF);
            float* Tf = reinterpret_cast<float*>(sm + R_TF);
            float* Xs = reinterpret_cast<float*>(sm + R_XS);
            if (tid < kSolveThreads) {
                solve_unit_lower(Af, Tf, Xs, sm + R_TB, tid);
            } else {
                // Meanwhile the other warps build (b V)^T, thread = (channel c,
                // tokens 32 half .. 32 half + 31).
                const int u = tid - kSolveThreads, c = u & 127, half = u >> 7;
                const __nv_bfloat16* vraw = reinterpret_cast<const __nv_bfloat16*>(sm + R_V);
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int s8 = 4 * half + it;
                    float bv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = s8 * 8 + e;
                        bv[e] = s < len ? small[SM_B + s] * __bfloat162float(vraw[s * kD + c]) : 0.f;
                    }
                    *reinterpret_cast<uint4*>(sm + R_BVT + sw128(c, s8)) = pack8(bv);
                }
                // Raw k and v are dead once all of these warps are here.
                named_bar_sync(3, kPrepThreads - kSolveThreads);
                if (tid == kLoadThread && nitem < n_items)
                    issue_item_kv(sm, maps, nt0, nhead, kvbar);
                // T as a bf16 K-major operand [t][s], 16-byte chunk (t, ch):
                // once the diagonal 32 x 32 blocks are final, these warps write
                // them and the zero block above them; the solve writes T21.
                named_bar_sync(4, kPrepThreads);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    if (pass == 1 && u >= 128) break;
                    const int t = pass == 0 ? (u >> 3) : 32 + (u >> 2);
                    const int ch = pass == 0 ? (u & 7) : 4 + (u & 3);
                    float o8[8];
                    load8f_sw(Tf + t * F_LD + ch * 8, o8, (ch >> 2) & 1);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (ch * 8 + e > t) o8[e] = 0.f;
                    *reinterpret_cast<uint4*>(sm + R_TB + sw128(t, ch)) = pack8(o8);
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- W^T = (b K^g)^T T^T -> cols [0,64) on bar, U~^T = (b V)^T T^T ->
        //      cols [64,128) on bar2, so that W^T's readback overlaps U~^T.
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16(128, 64), idesc_mn = idesc_bf16_amn(128, 64);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)      // (b K^g)^T MN-major: 16 tokens = 2 KB
                mma_bf16(tbase + 0, desc_sw128_mn(smem_u32(sm + R_BKT + ks * 2048), 8192, 1024),
                         desc_sw128(smem_u32(sm + R_TB + ks * 32)), idesc_mn, ks > 0);
            mma_commit(bar);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tbase + 64, desc_sw128(smem_u32(sm + R_BVT + ks * 32)),
                         desc_sw128(smem_u32(sm + R_TB + ks * 32)), idesc, ks > 0);
            mma_commit(bar2);
        }
        // W^T and U~^T as bf16 K-major operands, thread = row (channel / column):
        // warps 0-7 take W^T, warps 8-15 U~^T, 32 columns each.
        {
            const bool wpart = warp < 8;
            const uint32_t half = (uint32_t)(warp >> 2) & 1u;
            ok = mbar_wait(wpart ? bar : bar2, wpart ? phase : phase2) && ok;
            tc_fence_after();
            const uint32_t taddr = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + (wpart ? 0u : 64u) + 32 * half;
            tmem32_to_swizzled(taddr, sm + (wpart ? R_WT : R_UT), 32 * (warp & 3) + lane, 4 * half);
            phase ^= 1u;
            phase2 ^= 1u;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();

        // ---- [N | X] = (K^C)^T [W | U~] -> cols [0,256), with W^T and U~^T
        //      stacked as one 256-row operand; then P W -> [256,384) and
        //      O' = P U~ -> [384,512) on bar2, so that the readback of X
        //      overlaps them.  Both are M=128 products with P as 64 of the A
        //      rows: P W reads A from 64 rows before P, so that its rows land
        //      in TMEM lanes 64..127, and O' from P itself (lanes 0..63); the
        //      other 64 A rows read neighbouring tiles and land in unused
        //      accumulator rows.  That splits the readback evenly over the
        //      four lane quadrants.
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16_amn(128, 256), idesc_h = idesc_bf16(128, 128);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)      // (K^C)^T MN-major: 16 tokens = 2 KB
                mma_bf16(tbase + 0, desc_sw128_mn(smem_u32(sm + R_KC + ks * 2048), 8192, 1024),
                         desc_sw128(smem_u32(sm + R_WT + ks * 32)), idesc, ks > 0);
            mma_commit(bar);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t off = ks * 32;
                mma_bf16(tbase + 256, desc_sw128(smem_u32(sm + R_P - 8192 + off)),
                         desc_sw128(smem_u32(sm + R_WT + off)), idesc_h, ks > 0);
                mma_bf16(tbase + 384, desc_sw128(smem_u32(sm + R_P + off)),
                         desc_sw128(smem_u32(sm + R_UT + off)), idesc_h, ks > 0);
            }
            mma_commit(bar2);
        }
        ok = mbar_wait(bar, phase) && ok;
        phase ^= 1u;
        tc_fence_after();

        // ---- the package image, staged in shared memory.  Warp (quadrant q =
        //      warp mod 4, slot s = warp / 4) does three 32-column jobs on the
        //      rows of its lane quadrant: X tile s; then, after bar2 (the image
        //      of N overwrites W^T / U~^T, which the second products read),
        //      columns 32 s .. 32 s + 31 of N, and O' tile s (q < 2, token
        //      rows) or those columns of Q' = Q^g - P W (q >= 2, token rows).
        {
            const int q = warp & 3, sl = warp >> 2;
            const uint32_t row = 32 * q + lane;
            const uint32_t taddr = tbase + ((uint32_t)(32 * q) << 16);
            tmem32_to_jtile_pairs(taddr + 128 + 32 * sl, sm + R_PKG + PKG_X + sl * 8192, row);
            ok = mbar_wait(bar2, phase2) && ok;
            tc_fence_after();
            const uint32_t kb = (uint32_t)sl >> 1, ch0 = 4 * ((uint32_t)sl & 1);
            tmem32_to_swizzled(taddr + 32 * sl, sm + R_PKG + PKG_B0 + kb * PKG_BK, row, ch0);
            if (q < 2) {
                tmem32_to_jtile(taddr + 384 + 32 * sl, sm + R_PKG + PKG_OP + sl * 4096, row);
            } else {
                const uint32_t t = row - 64;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float pw[16];
                    tmem_ld16(taddr + 256 + 32 * sl + 16 * q2, pw);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t ch = ch0 + 2 * q2 + hh;
                        float qg[8], o8[8];
                        unpack8(*reinterpret_cast<const uint4*>(sm + R_QG + kb * 8192 + sw128(t, ch)), qg);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o8[e] = qg[e] - pw[8 * hh + e];
                        *reinterpret_cast<uint4*>(sm + R_PKG + PKG_B0 + kb * PKG_BK +
                                                  sw128(128 + t, ch)) = pack8(o8);
                    }
                }
            }
            if (tid < 128)
                reinterpret_cast<float*>(sm + R_PKG + PKG_LAM)[tid] = small[SM_LAM + tid];
            phase2 ^= 1u;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g(pkg, sm + R_PKG, 49152);
            bulk_s2g(pkg + 49152, sm + R_PKG + 49152, PKG_BYTES - 49152);
            bulk_commit();
        }
        item = nitem;
        slot = nslot;
        head = nhead;
        t0 = nt0;
        len = nlen;
    }
    if (!ok) set_status(status, kErrPrepWait);
    if (tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<512>(tbase);
    }
}

// ============================================================================
// state_pass: one CTA per (sequence, head, column tile), sequential over the
// sequence's chunks.  The update warps hold the tile S[c][j0 .. j0+31] in fp32
// registers, two threads per row c.  Per chunk two tcgen05 products
// read the bf16 copy of the tile's S^T: D_S[c][j] = (N S)[c][j] and D_O[t][j]
// = (Q' S)[t][j] (N=32, K=128; M=128 and M=64).  S^T is double-buffered so that chunk m + 1's update can write the
// next copy while chunk m's O product still reads the current one.
//
// Barriers (phase k of a per-chunk barrier belongs to the k-th chunk using it):
//   full[m % 4]     [N ; Q'] of chunk m landed            (1 arrival + bytes)
//   sdone[m & 1]    chunk m's S product done              (1 commit)
//   odone[m & 1]    chunk m's O product done              (1 commit)
//   sfree[m % 4]    chunk m's products no longer read its stage (1 commit)
//   stready[p]      S^T copy p written by the update of the chunk before (8 warps)
//   dfree[m & 1]    chunk m's accumulators read           (12 warps)
// X, O' and lam bypass shared memory: the warps that use them load their own
// pieces straight into registers two chunks ahead.
// ============================================================================
// Update-warp fragment of a 128 x 32 tile of S (rows c, tile columns j): warp
// w holds rows 32 q4 .. 32 q4 + 31 (q4 = w mod 4) and tile columns jh .. jh +
// 15 (jh = 16 ((w / 4) mod 2)) in the layout of a 16x256b TMEM load: element e
// (0..15) of a thread is
//   row    32 q4 + 16 (e >> 3) + 8 ((e >> 1) & 1) + lane / 4,
//   column jh + 8 ((e >> 2) & 1) + 2 (lane mod 4) + (e & 1),
// so elements 2i and 2i + 1 are adjacent columns of one row.
struct Frag {
    int q4, jh, lane;
    __device__ __forceinline__ Frag(int warp, int lane_)
        : q4(warp & 3), jh(16 * ((warp >> 2) & 1)), lane(lane_) {}
    __device__ __forceinline__ int row(int e) const {
        return 32 * q4 + 16 * (e >> 3) + 8 * ((e >> 1) & 1) + (lane >> 2);
    }
    __device__ __forceinline__ int col(int e) const {
        return jh + 8 * ((e >> 2) & 1) + 2 * (lane & 3) + (e & 1);
    }
};

// Writes the fragment `st` as copy `p` of the tile's S^T, the bf16 B operand
// of the state products (rows j, 128-byte-swizzled K-major over c; copies 8 KB
// apart from `st_base`): per 16-row half hh one transposing stmatrix of the
// four 8 x 8 matrices (m, k) = (i / 2, i mod 2), rows c = 32 q4 + 16 hh + 8 k ..,
// columns j = jh + 8 m ..  Thread t gives stored row j = jh + 8 m + t mod 8 of
// matrix i = t / 8.
__device__ __forceinline__ void write_st_copy(uint8_t* st_base, int p, const Frag& f,
                                              const float (&st)[16]) {
    const int i = f.lane >> 3, m = i >> 1, k = i & 1, jrow = f.jh + 8 * m + (f.lane & 7);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int c0 = 32 * f.q4 + 16 * hh + 8 * k;
        uint32_t rg[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
            const int e = 8 * hh + 4 * (ii >> 1) + 2 * (ii & 1);
            rg[ii] = pack_bf16x2(st[e], st[e + 1]);
        }
        stmatrix_x4_trans(smem_u32(st_base + p * 8192 + (c0 >> 6) * 4096 + sw128(jrow, (c0 & 63) >> 3)), rg);
    }
}

// X at a fragment's element pairs and lam at its four rows, for one chunk.
struct XRegs {
    uint32_t x[8];
    float lam[4];
};
__device__ __forceinline__ void load_x_frag(const uint8_t* pk, int tile, const Frag& f, XRegs& r) {
    const uint8_t* xt = pk + PKG_X + tile * 8192;
    // row(8 hh + 2 k): columns 2w, 2w + 1 (m = 0) and 8 + 2w, 9 + 2w (m = 1) of
    // the warp's 16-column group, 8 contiguous bytes in the package's pair
    // order (w = lane mod 4)
    const uint32_t xoff = 8u * (f.lane & 1);
    const int xch = 2 * (f.jh >> 4) + ((f.lane & 3) >> 1);
#pragma unroll
    for (int hk = 0; hk < 4; ++hk) {
        const int e = 8 * (hk >> 1) + 2 * (hk & 1);
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(xt + jtile_off(f.row(e), xch) + xoff));
        r.x[e >> 1] = v.x;
        r.x[(e + 4) >> 1] = v.y;
    }
#pragma unroll
    for (int hk = 0; hk < 4; ++hk)
        r.lam[hk] = __ldg(reinterpret_cast<const float*>(pk + PKG_LAM) + f.row(2 * hk + ((hk >> 1) * 4)));
}

// st <- lam (.) st + x - d on the fragment (x omitted when `with_x` is false).
__device__ __forceinline__ void update_frag(float (&st)[16], const float (&d)[16], const XRegs& xr,
                                            bool with_x) {
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        const float2 x = with_x ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xr.x[e >> 1]))
                                : make_float2(0.f, 0.f);
        const float lam = xr.lam[2 * (e >> 3) + ((e >> 1) & 1)];
        st[e] = fmaf(lam, st[e], x.x - d[e]);
        st[e + 1] = fmaf(lam, st[e + 1], x.y - d[e + 1]);
    }
}

__device__ __forceinline__ void issue_stage(uint8_t* stg, const uint8_t* pkg, uint64_t* full) {
    mbar_expect_tx(full, ST_BYTES);
    bulk_g2s(stg, pkg + PKG_B0, ST_BYTES, full);
}

// Asks L2 for the parts of a package that one column-tile CTA copies.
__device__ __forceinline__ void prefetch_stage(const uint8_t* pkg, int tile) {
    bulk_prefetch_l2(pkg + PKG_B0, 49152);
    bulk_prefetch_l2(pkg + PKG_X + tile * 8192, 8192);
    bulk_prefetch_l2(pkg + PKG_OP + tile * 4096, 4096);
    bulk_prefetch_l2(pkg + PKG_LAM, 512);
}

// Bounded wait that also gives up as soon as another role of the CTA has
// raised `abort`.
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 30); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && (*abort || global_ns() - t0 > 2000000000ull)) break;
    }
    return false;
}

// Segments of the segment-parallel prefill: sequence n is split into G
// segments of cps chunks; segment g starts from S_start[(n H + h)(G - 1) + g - 1]
// (g >= 1) or from S0 (g = 0).  G = 1 is the plain pass.
struct SegSpec {
    int G = 1;
    int cps = 0x7fffffff;           // chunks per segment
    const float* S_start = nullptr;  // [N, H, G - 1, d_k, d_v] fp32
};

__global__ void __launch_bounds__(kStateThreads, 1)
state_pass_kernel(const uint8_t* __restrict__ ws, __nv_bfloat16* __restrict__ o,
                  const float* __restrict__ S0, float* __restrict__ S1, SeqMap map, int H,
                  int dk, int dv, CheckpointSpec ck, SegSpec seg, const float* __restrict__ Scarry) {
    const int tile = blockIdx.x, n = blockIdx.y / seg.G, g = blockIdx.y % seg.G, h = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = tile * kJ;

    int64_t bos, eos, bos_seq;
    const int64_t slot_seq = seq_slot_base(map, n, bos, eos, bos_seq);
    const int nc_seq = (int)((eos - bos + kC - 1) / kC);
    const int c0 = (int)((int64_t)g * seg.cps < nc_seq ? (int64_t)g * seg.cps : nc_seq);
    const int nc = (nc_seq - c0) < seg.cps ? (nc_seq - c0) : seg.cps;   // this segment's chunks
    const int64_t slot0 = slot_seq + c0;
    const bool last_seg = g == seg.G - 1;
    uint32_t* status = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(ws));
    const uint8_t* pkgs = ws + WS_HEADER;
    auto pkg_of = [&](int chunk) { return pkgs + ((size_t)(slot0 + chunk) * H + h) * PKG_BYTES; };

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S_BAR);        // [4]
    uint64_t* sfree = full + kStages;                                  // [4]
    uint64_t* sdone = sfree + kStages;                                 // [2]
    uint64_t* odone = sdone + 2;                                       // [2]
    uint64_t* stready = odone + 2;                                     // [2]
    uint64_t* dfree = stready + 2;                                     // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dfree + 2);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    const Frag f(warp, lane);
    const bool upd = warp < kUpdWarps;
    // this tile of S0 / S1 ([d_k][d_v] per (n, h)); rows d_k .. 127 of a
    // narrower head stay 0 on chip and are neither read nor written
    const size_t smat = ((size_t)n * H + h) * dk * dv + j0;
    // A sequence that started in an earlier window continues from the carried state.
    const float* S_first = bos == bos_seq ? S0 : Scarry;
    const float* S_in = g == 0 ? (S_first ? S_first + smat : nullptr)
                               : seg.S_start + (((size_t)n * H + h) * (seg.G - 1) + (g - 1)) * dk * dv + j0;
    float st[16];
    auto store_state = [&](float* mat) {                             // mat: S of (n, h) + j0
#pragma unroll
        for (int e = 0; e < 16; e += 2)
            if (f.row(e) < dk)
                *reinterpret_cast<float2*>(mat + (size_t)f.row(e) * dv + f.col(e)) = make_float2(st[e], st[e + 1]);
    };
    if (upd) {
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            const float2 v = S_in && f.row(e) < dk
                                 ? __ldg(reinterpret_cast<const float2*>(S_in + (size_t)f.row(e) * dv + f.col(e)))
                                 : make_float2(0.f, 0.f);
            st[e] = v.x;
            st[e + 1] = v.y;
        }
    }
    if (nc <= 0 || (smem_u32(smem_raw) & 1023u) != 0) {
        if (nc > 0 && tid == 0) set_status(status, kErrSmemAlign);
        if (S1 && upd && last_seg) store_state(S1 + smat);
        return;
    }

    if (warp == 0) tmem_alloc<kTmemCols>(tslot);
    if (tid == 32) {
        for (int p = 0; p < kStages; ++p) {
            mbar_init(full + p, 1);
            mbar_init(sfree + p, 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(sdone + p, 1);
            mbar_init(odone + p, 1);
            mbar_init(stready + p, kUpdWarps);
            mbar_init(dfree + p, kUpdWarps + kOutWarps);
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (upd) write_st_copy(sm + S_ST, 0, f, st);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp == 14) {
        // ---------------------------------------------------- package copies
        if (lane == 0) {
            int m = 0;
            for (; m < kStages && m < nc; ++m) issue_stage(sm + m * ST_BYTES, pkg_of(m), full + m);
            for (int p = kStages; p < kL2Ahead && p < nc; ++p) prefetch_stage(pkg_of(p), tile);
            for (; m < nc; ++m) {
                // chunk m goes into chunk m - 4's stage once that chunk's products are done
                ok = role_wait(sfree + m % kStages, ((m - kStages) / kStages) & 1, abort) && ok;
                if (!ok) break;
                issue_stage(sm + (m % kStages) * ST_BYTES, pkg_of(m), full + m % kStages);
                if (m + kL2Ahead - kStages < nc) prefetch_stage(pkg_of(m + kL2Ahead - kStages), tile);
            }
            if (!ok) {
                *abort = 1;
                // Let the copies in flight land (bounded) before the CTA exits.
                for (int k = m > kStages ? m - kStages : 0; k < m; ++k)
                    mbar_wait(full + k % kStages, (k / kStages) & 1);
            }
        }
    } else if (warp == 12) {
        // ------------------------------------------- S product D_S = N S^T'
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, kJ);
            int cc = 0;
            for (; cc < nc; ++cc) {
                const int b = cc & 1;
                // accumulator buffer b was last read for chunk cc - 2
                if (cc >= 2) ok = role_wait(dfree + b, ((cc - 2) >> 1) & 1, abort) && ok;
                ok = role_wait(full + cc % kStages, (cc / kStages) & 1, abort) && ok;
                if (cc >= 1) ok = role_wait(stready + b, ((cc - 1) >> 1) & 1, abort) && ok;
                if (!ok) break;
                tc_fence_after();
                const uint64_t bdesc0 = desc_sw128(smem_u32(sm + S_ST + b * 8192));
                const uint64_t adesc0 = desc_sw128(smem_u32(sm + (cc % kStages) * ST_BYTES));
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + b * kDBuf, adesc0 + ((kb * PKG_BK + off) >> 4),
                             bdesc0 + ((kb * 4096 + off) >> 4), idesc, ks > 0);
                }
                mma_commit(sdone + b);
            }
            if (!ok) {
                *abort = 1;
                if (cc > 0) mbar_wait(sdone + ((cc - 1) & 1), ((cc - 1) >> 1) & 1);
            }
        }
    } else if (warp == 13) {
        // ------------------------- O product D_O = Q' S^T' (M=64), after D_S
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(64, kJ);
            int cc = 0;
            for (; cc < nc; ++cc) {
                const int b = cc & 1;
                ok = role_wait(sdone + b, (cc >> 1) & 1, abort) && ok;
                if (!ok) break;
                tc_fence_after();
                const uint64_t bdesc0 = desc_sw128(smem_u32(sm + S_ST + b * 8192));
                const uint64_t adesc0 = desc_sw128(smem_u32(sm + (cc % kStages) * ST_BYTES + 16384));
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + b * kDBuf + 32, adesc0 + ((kb * PKG_BK + off) >> 4),
                             bdesc0 + ((kb * 4096 + off) >> 4), idesc, ks > 0);
                }
                mma_commit(odone + b);
                mma_commit(sfree + cc % kStages);   // the S product finished before these began
            }
            if (!ok) {
                *abort = 1;
                if (cc > 0) mbar_wait(odone + ((cc - 1) & 1), ((cc - 1) >> 1) & 1);
            }
        }
    } else if (!upd) {
        // ------------------------------- outputs o = Q' S + O' (warps 8-11)
        const int t = 16 * (warp & 3) + lane;              // token row, lanes 0..15
        const bool act = lane < 16;
        const uint32_t tl = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
        // O'[t][0 .. 31] of chunk m, loaded two chunks ahead of its use
        auto load_op = [&](int m, uint4 (&r)[4]) {
            const uint8_t* tp = pkg_of(m) + PKG_OP + tile * 4096;
#pragma unroll
            for (int q = 0; q < 4; ++q) r[q] = __ldg(reinterpret_cast<const uint4*>(tp + jtile_off(t, q)));
        };
        auto step = [&](int cc, uint4 (&r)[4]) -> bool {
            const int b = cc & 1;
            ok = role_wait(odone + b, (cc >> 1) & 1, abort) && ok;
            if (!ok) return false;
            tc_fence_after();
            float ov[32];
            tmem_ld16(tl + b * kDBuf + 32, *reinterpret_cast<float(*)[16]>(ov));
            tmem_ld16(tl + b * kDBuf + 48, *reinterpret_cast<float(*)[16]>(ov + 16));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree + b);
            const int64_t t0 = bos + (int64_t)(c0 + cc) * kC;
            if (act && t < eos - t0) {
                uint4* dst = reinterpret_cast<uint4*>(o + ((size_t)(t0 + t) * H + h) * dv + j0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float op[8], o8[8];
                    unpack8(r[q], op);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o8[e] = ov[8 * q + e] + op[e];
                    __stcs(dst + q, pack8(o8));
                }
            }
            if (act && cc + 2 < nc) load_op(cc + 2, r);
            return true;
        };
        uint4 ra[4], rb[4];
        if (act) {
            load_op(0, ra);
            if (nc > 1) load_op(1, rb);
        }
        for (int cc = 0; cc < nc; cc += 2) {
            if (!step(cc, ra)) break;
            if (cc + 1 < nc && !step(cc + 1, rb)) break;
        }
        if (!ok) *abort = 1;
    } else {
        // ------------------------------- state S <- lam (.) S - (N S) + X
        const uint32_t tl = tbase + ((uint32_t)(32 * f.q4) << 16) + f.jh;
        auto step = [&](int cc, XRegs& xr) -> bool {
            const int b = cc & 1;
            ok = role_wait(sdone + b, (cc >> 1) & 1, abort) && ok;
            if (!ok) return false;
            tc_fence_after();
            float d[16];
            tmem_ld_16x256b_x2(tl + b * kDBuf, *reinterpret_cast<float(*)[8]>(d));
            tmem_ld_16x256b_x2(tl + (16u << 16) + b * kDBuf, *reinterpret_cast<float(*)[8]>(d + 8));
            tmem_wait_ld();
            update_frag(st, d, xr, true);
            if (cc + 1 < nc) {
                // S^T copy (cc + 1) & 1 is still read by chunk cc - 1's O product
                if (cc >= 1) ok = role_wait(odone + ((cc - 1) & 1), ((cc - 1) >> 1) & 1, abort) && ok;
                write_st_copy(sm + S_ST, (cc + 1) & 1, f, st);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (cc + 1 < nc) mbar_arrive(stready + ((cc + 1) & 1));
                mbar_arrive(dfree + b);
            }
            if (cc + 2 < nc) load_x_frag(pkg_of(cc + 2), tile, f, xr);
            // Checkpoint: the state after every `ck.every` tokens of this sequence
            // (bos - bos_seq of them precede this window).
            if (ck.out) {
                const int64_t done = (int64_t)(c0 + cc + 1) * kC;
                const int64_t at = (bos - bos_seq) + done;
                if (done <= eos - bos && at % ck.every == 0 && at / ck.every <= ck.max_count)
                    store_state(ck.out + (((size_t)n * H + h) * ck.max_count + (at / ck.every - 1)) * dk * dv + j0);
            }
            return true;
        };
        XRegs xa, xb;
        load_x_frag(pkg_of(0), tile, f, xa);
        if (nc > 1) load_x_frag(pkg_of(1), tile, f, xb);
        for (int cc = 0; cc < nc; cc += 2) {
            if (!step(cc, xa)) break;
            if (cc + 1 < nc && !step(cc + 1, xb)) break;
        }
        if (!ok) *abort = 1;
        if (S1 && last_seg) store_state(S1 + smat);
    }
    if (!ok) set_status(status, kErrStateWait);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTmemCols>(tbase);
    }
}

// ============================================================================
// Segment-parallel prefill ("Kimi K3 architecture: how an open model with a
// million-token context competes with market leaders", section "GPU level: the
// long-context scheduler": the segments of a long sequence are processed in
// parallel and merged into the exact state; the pair kept per segment is the
// context-parallel pair of "How Kimi K3 is built: 2.8 trillion parameters,
// linear attention and agents for a million tokens", section "How to serve two
// different caches").  Per chunk the state moves by S <- F_c S + X_c with
// F_c = Diag(lam_c) - N_c, so over segment g the state goes to M_g S_in + X_g
// with M_g = prod F_c and X_g = the segment's end state from a zero start.
//   trans_pass   per (sequence, head, segment g < G - 1) the chain over
//                Y = [X | M] (d_v + d_k columns) from Y0 = [0 | I]:
//                Y <- Diag(lam) Y - N Y + [X_c | 0]; one CTA per 32-column tile
//                of Y, no outputs.
//   seg_combine  S_start(g + 1) = M_g S_start(g) + X_g in fp32, sequential over
//                the segments (S_start(0) = the initial state).
//   state_pass   the plain pass, one CTA per (segment, 32-column tile of S),
//                from S_start(g): outputs of the segment's tokens, final state
//                from the last segment.
// The transition pass needs neither Q' nor O': only update warps, an MMA
// issuer and a copy warp, with a two-stage ring of the N operand, so that two
// of its CTAs share an SM.
// ============================================================================
constexpr int kTransThreads = 32 * 10;
constexpr int kTStages = 2;
constexpr uint32_t TST_BYTES = 32768;               // N only: two K-blocks of 128 rows
constexpr uint32_t T_ST = kTStages * TST_BYTES;     // then two S^T copies of 8 KB
constexpr uint32_t T_BAR = T_ST + 2 * 8192;
constexpr uint32_t T_SMEM = T_BAR + 256 + 1024;     // + slack for aligning the base
constexpr uint32_t kTTmemCols = 64;                 // two 32-column accumulators
constexpr uint32_t SEG_Y_COLS = 256;                // row pitch of a stored [X | M] (fp32)
constexpr size_t SEG_Y_BYTES = (size_t)128 * SEG_Y_COLS * 4;   // per (sequence, head, segment)
constexpr size_t SEG_S_BYTES = (size_t)128 * 128 * 4;          // room for one start state
static_assert(T_SMEM * 2 <= 232448, "two transition-pass CTAs per SM");

__device__ __forceinline__ void issue_nstage(uint8_t* stg, const uint8_t* pkg, uint64_t* full) {
    mbar_expect_tx(full, TST_BYTES);
    bulk_g2s(stg, pkg + PKG_B0, 16384, full);                  // N rows of K-block 0
    bulk_g2s(stg + 16384, pkg + PKG_B0 + PKG_BK, 16384, full);  // and of K-block 1
}

__global__ void __launch_bounds__(kTransThreads, 2)
trans_pass_kernel(uint8_t* __restrict__ ws, float* __restrict__ Y_out, SeqMap map, int H, int dk,
                  int dv, SegSpec seg) {
    const int tile = blockIdx.x, n = blockIdx.y / (seg.G - 1), g = blockIdx.y % (seg.G - 1);
    const int h = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nx = dv / kJ;                          // tiles of the X part; the rest are M
    const bool mpart = tile >= nx;
    const int m0 = kJ * (tile - nx);                 // first identity column of an M tile
    const int ycol0 = mpart ? 128 + m0 : kJ * tile;  // its first column in the stored Y

    int64_t bos, eos;
    const int64_t slot_seq = seq_slot_base(map, n, bos, eos);
    const int nc_seq = (int)((eos - bos + kC - 1) / kC);
    const int c0 = (int)((int64_t)g * seg.cps < nc_seq ? (int64_t)g * seg.cps : nc_seq);
    const int nc = (nc_seq - c0) < seg.cps ? (nc_seq - c0) : seg.cps;
    const int64_t slot0 = slot_seq + c0;
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    const uint8_t* pkgs = ws + WS_HEADER;
    auto pkg_of = [&](int chunk) { return pkgs + ((size_t)(slot0 + chunk) * H + h) * PKG_BYTES; };

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + T_BAR);        // [2]
    uint64_t* sfree = full + kTStages;                                 // [2]
    uint64_t* sdone = sfree + kTStages;                                // [2]
    uint64_t* stready = sdone + 2;                                     // [2]
    uint64_t* dfree = stready + 2;                                     // [2]
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dfree + 2);
    volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);

    const Frag f(warp, lane);
    const bool upd = warp < kUpdWarps;
    float st[16];
    if (upd) {
#pragma unroll
        for (int e = 0; e < 16; ++e) st[e] = (mpart && f.row(e) == m0 + f.col(e)) ? 1.f : 0.f;
    }
    float* ydst = Y_out + (((size_t)n * H + h) * (seg.G - 1) + g) * 128 * SEG_Y_COLS + ycol0;
    auto store_y = [&]() {
#pragma unroll
        for (int e = 0; e < 16; e += 2)
            if (f.row(e) < dk)
                *reinterpret_cast<float2*>(ydst + (size_t)f.row(e) * SEG_Y_COLS + f.col(e)) =
                    make_float2(st[e], st[e + 1]);
    };
    if (nc <= 0) {
        if (upd) store_y();
        return;
    }

    if (warp == 0) tmem_alloc<kTTmemCols>(tslot);
    if (tid == 32) {
        for (int p = 0; p < kTStages; ++p) {
            mbar_init(full + p, 1);
            mbar_init(sfree + p, 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(sdone + p, 1);
            mbar_init(stready + p, kUpdWarps);
            mbar_init(dfree + p, kUpdWarps);
        }
        *abort = 0;
        fence_mbar_init();
    }
    if (upd) write_st_copy(sm + T_ST, 0, f, st);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp == 9) {
        // ------------------------------------------------ N operand copies
        if (lane == 0) {
            int m = 0;
            for (; m < kTStages && m < nc; ++m) issue_nstage(sm + m * TST_BYTES, pkg_of(m), full + m);
            for (int p = kTStages; p < kL2Ahead && p < nc; ++p) {
                bulk_prefetch_l2(pkg_of(p) + PKG_B0, 16384);
                bulk_prefetch_l2(pkg_of(p) + PKG_B0 + PKG_BK, 16384);
            }
            for (; m < nc; ++m) {
                ok = role_wait(sfree + m % kTStages, ((m - kTStages) / kTStages) & 1, abort) && ok;
                if (!ok) break;
                issue_nstage(sm + (m % kTStages) * TST_BYTES, pkg_of(m), full + m % kTStages);
                const int pf = m + kL2Ahead - kTStages;
                if (pf < nc) {
                    bulk_prefetch_l2(pkg_of(pf) + PKG_B0, 16384);
                    bulk_prefetch_l2(pkg_of(pf) + PKG_B0 + PKG_BK, 16384);
                }
            }
            if (!ok) {
                *abort = 1;
                for (int k = m > kTStages ? m - kTStages : 0; k < m; ++k)
                    mbar_wait(full + k % kTStages, (k / kTStages) & 1);
            }
        }
    } else if (warp == 8) {
        // ----------------------------------------------- product D = N Y^T'
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, kJ);
            int cc = 0;
            for (; cc < nc; ++cc) {
                const int b = cc & 1;
                if (cc >= 2) ok = role_wait(dfree + b, ((cc - 2) >> 1) & 1, abort) && ok;
                ok = role_wait(full + cc % kTStages, (cc / kTStages) & 1, abort) && ok;
                if (cc >= 1) ok = role_wait(stready + b, ((cc - 1) >> 1) & 1, abort) && ok;
                if (!ok) break;
                tc_fence_after();
                const uint64_t bdesc0 = desc_sw128(smem_u32(sm + T_ST + b * 8192));
                const uint64_t adesc0 = desc_sw128(smem_u32(sm + (cc % kTStages) * TST_BYTES));
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, off = (ks & 3) * 32;
                    mma_bf16(tbase + b * kJ, adesc0 + ((kb * 16384 + off) >> 4),
                             bdesc0 + ((kb * 4096 + off) >> 4), idesc, ks > 0);
                }
                mma_commit(sdone + b);
                mma_commit(sfree + cc % kTStages);
            }
            if (!ok) {
                *abort = 1;
                if (cc > 0) mbar_wait(sdone + ((cc - 1) & 1), ((cc - 1) >> 1) & 1);
            }
        }
    } else if (upd) {
        // -------------------------------- Y <- lam (.) Y - (N Y) + [X | 0]
        const uint32_t tl = tbase + ((uint32_t)(32 * f.q4) << 16) + f.jh;
        const int xtile = mpart ? 0 : tile;
        auto step = [&](int cc, XRegs& xr) -> bool {
            const int b = cc & 1;
            ok = role_wait(sdone + b, (cc >> 1) & 1, abort) && ok;
            if (!ok) return false;
            tc_fence_after();
            float d[16];
            tmem_ld_16x256b_x2(tl + b * kJ, *reinterpret_cast<float(*)[8]>(d));
            tmem_ld_16x256b_x2(tl + (16u << 16) + b * kJ, *reinterpret_cast<float(*)[8]>(d + 8));
            tmem_wait_ld();
            update_frag(st, d, xr, !mpart);
            // copy (cc + 1) & 1 was last read by chunk cc - 1's product, which
            // completed before chunk cc's (sdone above)
            if (cc + 1 < nc) write_st_copy(sm + T_ST, (cc + 1) & 1, f, st);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (cc + 1 < nc) mbar_arrive(stready + ((cc + 1) & 1));
                mbar_arrive(dfree + b);
            }
            if (cc + 2 < nc) load_x_frag(pkg_of(cc + 2), xtile, f, xr);
            return true;
        };
        XRegs xa, xb;
        load_x_frag(pkg_of(0), xtile, f, xa);
        if (nc > 1) load_x_frag(pkg_of(1), xtile, f, xb);
        for (int cc = 0; cc < nc; cc += 2) {
            if (!step(cc, xa)) break;
            if (cc + 1 < nc && !step(cc + 1, xb)) break;
        }
        if (!ok) *abort = 1;
        store_y();
    }
    if (!ok) set_status(status, kErrStateWait);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<kTTmemCols>(tbase);
    }
}

// S_start(g + 1) = M_g S_start(g) + X_g for g = 0 .. G - 2 in fp32, per
// (sequence, head, 8-column tile of S); S_start(0) is the initial state (zeros
// when there is none).  M_g and this tile of X_g are staged in shared memory
// (M rows at a pitch of 132 floats), two buffers deep: the copies of step g + 1
// (cp.async, each thread its own 16-byte pieces) run while step g multiplies,
// so no step waits on global memory.  Every thread forms one row c times four
// columns.
constexpr int kCombCols = 8;
constexpr int kMPitch = 132;
constexpr uint32_t COMB_BUF = 128 * kMPitch + 128 * kCombCols;           // floats per buffer
constexpr uint32_t COMB_SMEM = (2 * COMB_BUF + 128 * kCombCols) * 4;

__device__ __forceinline__ void comb_issue(float* buf, const float* Yg, int dk, int j0, int tid) {
    float* Ms = buf;
    float* Xs = buf + 128 * kMPitch;
    for (int i = tid; i < 128 * 32; i += 256) {
        const int row = i >> 5, c4 = i & 31;
        if (row < dk && 4 * c4 < dk)
            cp_async16(Ms + row * kMPitch + 4 * c4, Yg + (size_t)row * SEG_Y_COLS + 128 + 4 * c4, 16);
    }
    {   // X_g[c][j0 .. j0 + 7]: two 16-byte pieces per row, one per thread
        const int row = tid >> 1, half = tid & 1;
        if (row < dk) cp_async16(Xs + row * kCombCols + 4 * half, Yg + (size_t)row * SEG_Y_COLS + j0 + 4 * half, 16);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(256)
seg_combine_kernel(const float* __restrict__ Y, const float* __restrict__ S0,
                   float* __restrict__ S_start, int H, int dk, int dv, int G) {
    const int j0 = blockIdx.x * kCombCols, n = blockIdx.y, h = blockIdx.z, tid = threadIdx.x;
    extern __shared__ float comb_smem[];
    float* cur = comb_smem + 2 * COMB_BUF;                      // S_start(g) [128][8]
    const int c = tid >> 1, jq = 4 * (tid & 1);
    const bool row_ok = c < dk;
    auto Yof = [&](int g) { return Y + (((size_t)n * H + h) * (G - 1) + g) * 128 * SEG_Y_COLS; };
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S0 && row_ok)
        s = *reinterpret_cast<const float4*>(S0 + (((size_t)n * H + h) * dk + c) * dv + j0 + jq);
    *reinterpret_cast<float4*>(cur + c * kCombCols + jq) = s;
    if (G > 1) comb_issue(comb_smem, Yof(0), dk, j0, tid);
    for (int g = 0; g + 1 < G; ++g) {
        float* buf = comb_smem + (g & 1) * COMB_BUF;
        // step g + 1's copies go to the other buffer, whose last reader (step
        // g - 1) is behind the barrier that closed that step
        if (g + 2 < G) {
            comb_issue(comb_smem + ((g + 1) & 1) * COMB_BUF, Yof(g + 1), dk, j0, tid);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();                          // M_g, X_g and S_start(g) in place
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row_ok) {
            acc = *reinterpret_cast<const float4*>(buf + 128 * kMPitch + c * kCombCols + jq);
            const float* mrow = buf + c * kMPitch;
            for (int cp = 0; cp < dk; cp += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float m = mrow[cp + u];
                    const float4 x = *reinterpret_cast<const float4*>(cur + (cp + u) * kCombCols + jq);
                    acc.x = fmaf(m, x.x, acc.x);
                    acc.y = fmaf(m, x.y, acc.y);
                    acc.z = fmaf(m, x.z, acc.z);
                    acc.w = fmaf(m, x.w, acc.w);
                }
            }
        }
        __syncthreads();                          // every read of step g's buffers and S_start(g) done
        *reinterpret_cast<float4*>(cur + c * kCombCols + jq) = acc;
        if (row_ok)
            *reinterpret_cast<float4*>(S_start + ((((size_t)n * H + h) * (G - 1) + g) * dk + c) * dv +
                                       j0 + jq) = acc;
    }
}

}  // namespace tc

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point so
// that the library does not link against the driver library directly.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map of one [T_total][H][d] bf16 input (d <= 128, 2 d a multiple of
// 16 bytes) with box_rows x 1 x 128 boxes: channels d .. 127 of a box lie
// outside the tensor and arrive as zeros.
bool make_rows_tensor_map(void* map, const void* base, int64_t T_total, int H, int d, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T_total};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {128, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
static bool make_input_map(CUtensorMap* m, const void* base, int64_t T_total, int H, int d) {
    return make_rows_tensor_map(m, base, T_total, H, d, tc::kC);
}

// Chunks per segment and the segment count actually used when a fixed-length
// batch of T tokens per sequence is split into (at most) G segments.
static void segment_shape(int64_t T, int G, int& cps, int& G_eff) {
    const int64_t nc = (T + tc::kC - 1) / tc::kC;
    if (G <= 1 || nc <= 1) {
        cps = 0x7fffffff;
        G_eff = 1;
        return;
    }
    const int64_t c = (nc + G - 1) / G;
    cps = (int)c;
    G_eff = (int)((nc + c - 1) / c);
}

int chunked_tc_segments_used(int64_t T, int G) {
    int cps, Ge;
    segment_shape(T, G, cps, Ge);
    return Ge;
}

size_t chunked_tc_workspace_bytes(int n_seqs, int64_t T_total, int H, int64_t T_seq, int G) {
    const int64_t slots = T_total / tc::kC + n_seqs + 1;
    size_t bytes = tc::WS_HEADER + (size_t)slots * H * tc::PKG_BYTES;
    const int Ge = chunked_tc_segments_used(T_seq, G);
    if (Ge > 1) bytes += (size_t)n_seqs * H * (Ge - 1) * (tc::SEG_Y_BYTES + tc::SEG_S_BYTES);
    return bytes;
}

// The segment count kda_chunk_prefill picks for a fixed-length batch: more
// than one only when the plain state pass would leave most SMs idle.  Costs in
// chain steps of the plain pass (measured on the long-context shapes): the
// plain pass walks the whole chain once; a segmented one walks a segment's
// chain in the transition pass (two CTAs per SM, each step about 1.5 times
// slower than a plain step), then in the final pass (one CTA per SM), in waves,
// plus about two steps per segment for the sequential combine.  Segments keep
// at least 16 chunks.
int chunked_tc_auto_segments(int B, int64_t T, int H, int dk, int dv, int num_sms) {
    if (B <= 0 || T <= 0 || H <= 0) return 1;
    const int64_t nc = (T + tc::kC - 1) / tc::kC;
    const int64_t nx = dv / tc::kJ, nm = (dk + tc::kJ - 1) / tc::kJ;
    const int64_t plain = (int64_t)B * H * nx;
    if (plain * 2 > num_sms) return 1;
    auto waves = [](int64_t n, int64_t slots) { return (n + slots - 1) / slots; };
    int best = 1;
    int64_t best_cost = nc * waves(plain, num_sms);
    for (int G = 2; G <= 64; ++G) {
        int cps, Ge;
        segment_shape(T, G, cps, Ge);
        if (cps < 16 || (int64_t)B * Ge > 65535) break;
        const int64_t ab = (int64_t)B * H * (Ge - 1) * (nx + nm), d = (int64_t)B * H * Ge * nx;
        const int64_t cost = (int64_t)cps * (3 * waves(ab, 2 * (int64_t)num_sms) + 2 * waves(d, num_sms)) / 2 +
                             2 * (Ge - 1);
        if (cost < best_cost) {
            best = Ge;
            best_cost = cost;
        }
    }
    return best;
}

cudaError_t run_chunked_tc(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, void* o, const float* S0, float* S1,
                           const float* Scarry, const int32_t* cu, int n_seqs, int64_t T,
                           int64_t rows, int64_t w0, int64_t w1, int H, int dk, int dv,
                           void* workspace, const CheckpointSpec& ck, cudaStream_t stream,
                           int num_sms, int n_segments) {
    constexpr int kMaxDevices = 64;
    static bool attr_done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        e = cudaFuncSetAttribute(tc::chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::P_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::state_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::S_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::trans_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::T_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::COMB_SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    e = cudaMemsetAsync(ws, 0, tc::WS_HEADER, stream);
    if (e != cudaSuccess) return e;
    tc::SeqMap map{cu, T, rows, n_seqs, w0, w1};
    using bf = __nv_bfloat16;
    profile_event(0, stream);
    const int64_t win_tokens = cu ? (w1 - w0) : (int64_t)n_seqs * (w1 - w0);
    const int64_t slots = win_tokens / tc::kC + n_seqs + 1;
    if (win_tokens > 0) {
        tc::InputMaps maps;
        if (!make_input_map(&maps.q, q, rows, H, dk) || !make_input_map(&maps.k, k, rows, H, dk) ||
            !make_input_map(&maps.v, v, rows, H, dv) || !make_input_map(&maps.z, z, rows, H, dk))
            return cudaErrorInvalidValue;
        const int64_t n_items = slots * H;
        const int64_t grid = n_items < num_sms ? n_items : num_sms;
        tc::chunk_prep_kernel<<<(unsigned)grid, tc::kPrepThreads, tc::P_SMEM, stream>>>(
            maps, static_cast<const bf*>(beta), A, ws, map, H, dk, n_items);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    profile_event(1, stream);
    tc::SegSpec seg;
    int cps = 0x7fffffff, Ge = 1;
    if (cu == nullptr) segment_shape(w1 - w0, n_segments, cps, Ge);
    if (Ge > 1) {
        // [X | M] per (sequence, head, segment < G - 1), then the start states
        float* Y = reinterpret_cast<float*>(ws + tc::WS_HEADER + (size_t)slots * H * tc::PKG_BYTES);
        float* S_start = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(Y) +
                                                  (size_t)n_seqs * H * (Ge - 1) * tc::SEG_Y_BYTES);
        seg.G = Ge;
        seg.cps = cps;
        seg.S_start = S_start;
        const int nm = (dk + tc::kJ - 1) / tc::kJ;
        dim3 grid_t((unsigned)(dv / tc::kJ + nm), (unsigned)(n_seqs * (Ge - 1)), (unsigned)H);
        tc::trans_pass_kernel<<<grid_t, tc::kTransThreads, tc::T_SMEM, stream>>>(ws, Y, map, H, dk, dv, seg);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        profile_event(2, stream);
        dim3 grid_c((unsigned)(dv / tc::kCombCols), (unsigned)n_seqs, (unsigned)H);
        // Segments are for fixed-length batches, whose sequences all start in the
        // first window: later windows start from the carried states.
        tc::seg_combine_kernel<<<grid_c, 256, tc::COMB_SMEM, stream>>>(Y, w0 == 0 ? S0 : Scarry,
                                                                       S_start, H, dk, dv, Ge);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        profile_event(3, stream);
    }
    dim3 grid_s((unsigned)(dv / tc::kJ), (unsigned)(n_seqs * Ge), (unsigned)H);
    tc::state_pass_kernel<<<grid_s, tc::kStateThreads, tc::S_SMEM, stream>>>(
        ws, static_cast<bf*>(o), S0, S1, map, H, dk, dv, ck, seg, Scarry);
    e = cudaGetLastError();
    profile_event(Ge > 1 ? 4 : 2, stream);
    return e;
}

}  // namespace kda
