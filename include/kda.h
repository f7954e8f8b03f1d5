/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention layer library.
 *
 * The layer (per sequence n and head h; S is a d_k x d_v state):
 *
 *   g_t   = -5 * sigmoid(exp(A_h) (.) z_t)          (per channel, g_min = -5)
 *   a_t   = exp(g_t)                                 (forget factor in [e^-5, 1])
 *   S_t   = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T
 *   o_t   = S_t^T q_t
 *
 * Sources: the gate is the forget-coefficient parametrisation of
 * "How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens",
 * section "Sequence: three KDA to one global MLA" (g = g_min*sigmoid(exp(A)*z),
 * alpha = exp(g), g_min = -5).  The state update is the delta rule of
 * "Kimi K3 architecture: how an open model with a million-token context competes with market leaders",
 * section "How the Kimi K3 architecture holds a million tokens of context": a
 * fixed state that each token partly erases and then writes, beta the write
 * strength, alpha the forget factor, alpha bounded to [e^-5, 1].  Both pages
 * make the forget gate per channel.
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers owned by the caller, unless stated.
 *     The library allocates no device memory, keeps no pointer after a call
 *     returns, and launches its kernels asynchronously on `stream`.
 *   - Layouts are row-major and dense:
 *       q, k, z      [tokens, H, d_k]      (tokens = B*T, or packed T_total)
 *       v, o         [tokens, H, d_v]
 *       beta         [tokens, H]           (a scalar write strength in (0,1))
 *       A            [H, d_k] fp32
 *       states       [N, H, d_k, d_v] fp32 (d_v contiguous)
 *     q, k, v, z, beta and o share one dtype (KDA_DTYPE_F32 or KDA_DTYPE_BF16).
 *     The caller L2-normalises q and k if it wants unit keys; there is no
 *     query scale.
 *   - Every tensor pointer must be 16-byte aligned.
 *   - Argument errors are reported before anything is launched.  Launch
 *     failures are reported as KDA_ERR_CUDA.  Kernels never trap or assert;
 *     kda_last_error() gives a one-line description of the last failure on
 *     the calling thread.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or layout    */
    KDA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d_k > 128)     */
    KDA_ERR_CUDA = 3,          /* a CUDA call or kernel launch failed            */
    KDA_ERR_WORKSPACE = 4      /* workspace missing or smaller than required     */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

/* Which kernels kda_chunk_prefill runs for a given shape. */
typedef enum {
    KDA_PATH_RECURRENT = 0,    /* SIMT fp32, token by token, any d_k, d_v <= 128     */
    KDA_PATH_CHUNKED_TC = 1,   /* chunked WY/UT form on tcgen05: bf16, chunk 64,
                                  d_k a multiple of 16 and d_v a multiple of 32,
                                  both <= 128 (zero-padded to 128 on chip)      */
    KDA_PATH_CHUNK16_TC = 2    /* the same form over 16-token chunks, one fused
                                  tcgen05 kernel per (sequence, head): bf16,
                                  chunk 16, d_k and d_v multiples of 16, <= 128 */
} kda_prefill_path;

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_string(kda_status s);

/* Description of the last non-OK status returned on this thread ("" if none). */
const char *kda_last_error(void);

/*
 * kda_gate -- the forget gate on its own.
 *   g[t, h, c] = clamp(-5 * sigmoid(exp(A[h, c]) * z[t, h, c]), -5, 0)   (fp32 out)
 * Defined by the gate formula of the first page above (g_min = -5); the clamp
 * only guards the rounding of sigmoid and never moves an exact value.
 *   z        [n_tokens, H, d_k] in z_dtype
 *   A        [H, d_k] fp32
 *   g        [n_tokens, H, d_k] fp32 (written)
 * n_tokens may be 0 (nothing is launched).  Prefill and decode compute the gate
 * inline from z and never read g.
 */
kda_status kda_gate(const void *z, const float *A, float *g, int64_t n_tokens, int H, int d_k,
                    kda_dtype z_dtype, cudaStream_t stream);

/*
 * kda_chunk_prefill -- o and (optionally) the final state for a batch of
 * sequences, by the chunked form: tokens of one chunk in parallel, then the
 * state passed from chunk to chunk (second page above, section "Chip level:
 * the specialised FlashKDA kernel"; the g_min bound that keeps every causal
 * block a dense product is from the first page, same section as the gate).
 *
 * Fixed-length batch: cu_seqlens == NULL, inputs [B, T, H, d], N = B = n_seqs.
 * Packed batch:       cu_seqlens != NULL (device int32 [n_seqs + 1], rising
 *                     from 0 to T), B must be 1, inputs [1, T, H, d],
 *                     N = n_seqs.  Chunk boundaries restart at every sequence.
 *                     Malformed offsets are clamped into [0, T] on the device:
 *                     results are then unspecified but no access leaves the
 *                     buffers.
 *   initial_state  nullable; [N, H, d_k, d_v] fp32 (read).  NULL means zeros.
 *   final_state    nullable; [N, H, d_k, d_v] fp32 (written).
 *   o              [B, T, H, d_v] in `dtype` (written).
 *   chunk          16 or 64 (the exact result does not depend on it).
 *                  bf16 with chunk 64, d_k a multiple of 16 and d_v a multiple
 *                  of 32 (both <= 128) runs on the 64-token tensor-core path;
 *                  bf16 with chunk 16, d_k and d_v multiples of 16 (<= 128)
 *                  on the 16-token tensor-core path (one fused kernel per
 *                  (sequence, head), the state handed on every 16 tokens);
 *                  everything else on the fp32 SIMT recurrence
 *                  (kda_chunk_prefill_path says which path a shape takes).  The
 *                  64-token path takes fewer than 2^31 tokens in all
 *                  (KDA_ERR_UNSUPPORTED otherwise).
 *   workspace      device scratch of at least kda_chunk_prefill_workspace_size()
 *                  bytes (may be NULL when that size is 0); 256-byte aligned;
 *                  contents on entry are ignored.  Its first 32-bit word is the
 *                  call's device status: the call clears it, and a kernel that
 *                  gives up a bounded wait (about 2 s; nothing in a correct
 *                  run waits that long) sets a nonzero bit there and returns
 *                  instead of hanging.  Read it after the stream has finished:
 *                  nonzero means o and the states of that call are not valid.
 *                  The fp32 SIMT recurrence needs no workspace: if one of its
 *                  bounded waits gives up, o from that point of the sequence
 *                  and that sequence's final state are NaN instead.
 * T == 0 (or every sequence empty) writes only the final states (copies of the
 * initial ones, or zeros).
 * A fixed-length batch whose (sequence, head) chains would leave most SMs idle
 * in the state pass (few sequences and heads, long T) is split into segments
 * automatically (see kda_chunk_prefill_segmented); the workspace size returned
 * by kda_chunk_prefill_workspace_size includes what that needs, and a
 * workspace that only covers the plain pass makes the call run unsegmented.
 */
kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const void *z,
                             const void *beta, const float *A, void *o,
                             const float *initial_state, float *final_state,
                             const int32_t *cu_seqlens, int n_seqs, int B, int64_t T, int H,
                             int d_k, int d_v, int chunk, kda_dtype dtype, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_prefill_segmented -- kda_chunk_prefill for a fixed-length batch
 * with each sequence split into n_segments segments whose state passes run in
 * parallel ("Kimi K3 architecture: how an open model with a million-token
 * context competes with market leaders", section "GPU level: the long-context
 * scheduler": segments of a long sequence computed on otherwise idle SMs and
 * merged into the exact final state; the per-segment pair of transition and
 * state-from-zero is the context-parallel pair of "How Kimi K3 is built",
 * section "How to serve two different caches").
 *
 * With F_c = Diag(lam_c) - N_c the per-chunk state map S <- F_c S + X_c of the
 * chunked form, segment g maps its start state S_g to M_g S_g + X_g
 * (M_g = product of its F_c, X_g = its end state from zero).  The call forms
 * every (M_g, X_g) in parallel, scans S_{g+1} = M_g S_g + X_g in fp32 from the
 * initial state, then runs every segment from its S_g, writing o and, from the
 * last segment, the final state.  The result equals kda_chunk_prefill up to
 * rounding.  It pays when B * H * d_v / 32 is well below the SM count and T is
 * long: each segment's chain is walked twice, but the segments run at once.
 *   n_segments  >= 1; segments hold ceil(ceil(T / 64) / n_segments) chunks, so
 *               fewer may be used (kda_chunk_prefill_auto_segments reports the
 *               count kda_chunk_prefill picks).  1 is the plain pass.
 *   workspace   kda_chunk_prefill_segmented_workspace_size() bytes, 256-byte
 *               aligned; word 0 is the device status as for kda_chunk_prefill.
 * Other arguments as for kda_chunk_prefill with cu_seqlens == NULL and
 * n_seqs == B.  Only the tensor-core shapes (bf16, chunk 64, d_k a multiple of
 * 16 and d_v a multiple of 32, both <= 128) are taken (KDA_ERR_UNSUPPORTED
 * otherwise), with B * segments <= 65535.
 */
kda_status kda_chunk_prefill_segmented(const void *q, const void *k, const void *v, const void *z,
                                       const void *beta, const float *A, void *o,
                                       const float *initial_state, float *final_state, int B,
                                       int64_t T, int H, int d_k, int d_v, int chunk,
                                       kda_dtype dtype, int n_segments, void *workspace,
                                       size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes of kda_chunk_prefill_segmented (0 for shapes it does not take). */
size_t kda_chunk_prefill_segmented_workspace_size(int B, int64_t T, int H, int d_k, int d_v,
                                                  int chunk, kda_dtype dtype, int n_segments);

/* The segment count kda_chunk_prefill uses for a fixed-length batch of these
 * sizes on the current device (1: unsegmented). */
int kda_chunk_prefill_auto_segments(int B, int64_t T, int H, int d_k, int d_v, int chunk,
                                    kda_dtype dtype);

/*
 * kda_chunk_prefill_checkpoints -- kda_chunk_prefill that also emits
 * intermediate states ("checkpoint states") at fixed token boundaries.
 *
 * Serving with a prefix cache keeps states only at some boundaries and copies a
 * saved state before continuing from it ("How Kimi K3 is built", section "How
 * to serve two different caches": checkpoint states are immutable and copied
 * into the request's own state before it continues).  This call writes, for
 * every sequence n and head h, the state after (i + 1) * checkpoint_every of
 * that sequence's tokens into checkpoints[n, h, i] for
 * i < min(len_n / checkpoint_every, max_checkpoints).  Slots past that are not
 * written.  Continuing a prefill from checkpoints[n, h, i] (as initial_state)
 * gives the same result as the uninterrupted run.
 *   checkpoints       nullable (then this is kda_chunk_prefill); [N, H,
 *                     max_checkpoints, d_k, d_v] fp32, 16-byte aligned
 *   checkpoint_every  tokens between checkpoints, a positive multiple of chunk
 *   max_checkpoints   slots per (sequence, head), >= 1
 * Everything else is as for kda_chunk_prefill.
 */
kda_status kda_chunk_prefill_checkpoints(const void *q, const void *k, const void *v,
                                         const void *z, const void *beta, const float *A, void *o,
                                         const float *initial_state, float *final_state,
                                         const int32_t *cu_seqlens, int n_seqs, int B, int64_t T,
                                         int H, int d_k, int d_v, int chunk, kda_dtype dtype,
                                         float *checkpoints, int64_t checkpoint_every,
                                         int max_checkpoints, void *workspace,
                                         size_t workspace_bytes, cudaStream_t stream);

/*
 * kda_chunk_prefill_from_host -- kda_chunk_prefill for a fixed-length batch
 * whose inputs and output live in host memory, with the transfers overlapped
 * with the kernels.  The layer computed is the one of kda_chunk_prefill; the
 * pages describe no host interface, so this entry has no counterpart there.
 *
 * Each sequence is processed in segments of segment_tokens tokens: the
 * segment's q, k, v, z, beta are copied to the device on h2d_stream, prefilled
 * on `stream` (continuing from the state the previous segment left in
 * final_state), and its o is copied back on d2h_stream, so that the copies of
 * one segment run while another is computed.  The result equals one
 * kda_chunk_prefill call on the whole batch.
 *   q_h, k_h, v_h, z_h, beta_h  host inputs [B, T, H, d] (beta [B, T, H]) in
 *                 `dtype`; page-locked (cudaHostAlloc) for the copies to
 *                 overlap.
 *   o_h           host output [B, T, H, d_v], page-locked.
 *   q_d .. beta_d, o_d  device buffers of the same shapes (staging), written.
 *   A             device [H, d_k] fp32.
 *   initial_state nullable device [B, H, d_k, d_v] fp32 (read before the
 *                 first segment of each sequence writes final_state, so it
 *                 may equal final_state).
 *   final_state   device [B, H, d_k, d_v] fp32, required: it carries the
 *                 state from segment to segment and ends as the final state.
 *   segment_tokens  a positive multiple of 64.
 *   workspace     as for kda_chunk_prefill with B = 1, T = segment_tokens.
 * Only shapes of the tensor-core path (bf16, chunk 64, d_k a multiple of 16
 * and d_v a multiple of 32, both <= 128); anything else returns
 * KDA_ERR_UNSUPPORTED.  The three streams must differ; h2d_stream and
 * d2h_stream first wait for the work already queued on `stream`, and `stream`
 * finishes only after the last copy back, so synchronising `stream` covers
 * the whole call.  Each call creates and destroys two CUDA events.
 */
kda_status kda_chunk_prefill_from_host(const void *q_h, const void *k_h, const void *v_h,
                                       const void *z_h, const void *beta_h, const float *A,
                                       void *o_h, void *q_d, void *k_d, void *v_d, void *z_d,
                                       void *beta_d, void *o_d, const float *initial_state,
                                       float *final_state, int B, int64_t T, int H, int d_k,
                                       int d_v, kda_dtype dtype, int64_t segment_tokens,
                                       void *workspace, size_t workspace_bytes,
                                       cudaStream_t stream, cudaStream_t h2d_stream,
                                       cudaStream_t d2h_stream);

/*
 * Bytes of workspace kda_chunk_prefill needs for these sizes (0 if none).
 * For packed batches pass B = 1, T = total tokens and the sequence count; the
 * bound does not depend on the individual lengths.
 */
size_t kda_chunk_prefill_workspace_size(int n_seqs, int B, int64_t T, int H, int d_k, int d_v,
                                        int chunk, kda_dtype dtype);

/* The kernel path kda_chunk_prefill takes for these sizes. */
kda_prefill_path kda_chunk_prefill_path(int d_k, int d_v, int chunk, kda_dtype dtype);

/*
 * kda_decode_step -- one token for each of B independent sequences, updating
 * the state in place.  The fixed-size state replaces a KV cache, and the first
 * page above notes, in "How to serve two different caches", that reading this
 * state is the cost of decoding:
 *   S' = Diag(a) S,  u = b (v - S'^T k),  S <- S' + k u^T,  o = S'^T q + u (k^T q)
 * which equals o = S_new^T q.
 *   q, k, z  [B, H, d_k];  v, o [B, H, d_v];  beta [B, H]  (dtype)
 *   A        [H, d_k] fp32
 *   state    [B, H, d_k, d_v] fp32, read and overwritten
 * Supports d_k <= 128 and d_v <= 128 with d_v a multiple of 4.  B == 0 is a
 * no-op.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *z,
                           const void *beta, const float *A, float *state, void *o, int B, int H,
                           int d_k, int d_v, kda_dtype dtype, cudaStream_t stream);

/*
 * kda_chunk_prefill_static_workspace -- kda_chunk_prefill for callers that
 * cannot allocate device memory.
 *
 * The pages describe no counterpart to this entry point; it exists for
 * deployment.  The chunked tensor-core path needs device scratch, which
 * kda_chunk_prefill takes from its caller.  Some callers cannot allocate it:
 * a plugin hosted by a runtime that owns every device allocation and forbids
 * its plugins from calling cudaMalloc, or a serving loop whose memory plan is
 * fixed at start-up.  This entry point takes the same arguments minus the
 * workspace and uses a library-owned __device__ array of
 * KDA_STATIC_WORKSPACE_BYTES instead.  It allocates nothing.
 *
 *   - Every GPU that loads the library holds that array until the process exits.
 *   - Sizes whose workspace (kda_chunk_prefill_workspace_size) exceeds
 *     KDA_STATIC_WORKSPACE_BYTES are rejected with KDA_ERR_UNSUPPORTED before
 *     any launch; kda_last_error() says how much they would need.
 *   - The array lives on the current device: make the device that owns the
 *     pointers and `stream` current before the call.  Each call looks up the
 *     array's device address there (cudaGetSymbolAddress), so a reset device
 *     or a second context gets its own array.  The first call on a device also
 *     loads the library's kernels there; make it before any stream capture.
 *   - The device status word of the call (see `workspace` above) sits in the
 *     array; kda_static_workspace_status copies it out.
 *   - All calls share the one array and it keeps the last call's contents (the
 *     kernels clear what must start at zero).  Calls whose kernels overlap on
 *     the GPU -- concurrent streams, or several host threads -- race on it;
 *     serialise them.
 * Arguments, layouts and errors are otherwise those of kda_chunk_prefill.
 */
#define KDA_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)

kda_status kda_chunk_prefill_static_workspace(const void *q, const void *k, const void *v,
                                              const void *z, const void *beta, const float *A,
                                              void *o, const float *initial_state,
                                              float *final_state, const int32_t *cu_seqlens,
                                              int n_seqs, int B, int64_t T, int H, int d_k,
                                              int d_v, int chunk, kda_dtype dtype,
                                              cudaStream_t stream);

/*
 * kda_static_workspace_status -- copies the device status word of the last
 * kda_chunk_prefill_static_workspace call on the current device (word 0 of
 * the library's array; 0 = every bounded wait was satisfied) into *status,
 * asynchronously on `stream`.  Issue it on the stream of that call (or after
 * it), then read *status once the stream has finished.  Nonzero means the
 * call's outputs are not valid.  The next static-workspace call clears the
 * word again.  The pages have no counterpart; this only reports.
 *   status  uint32_t, device or page-locked host memory, 4-byte aligned
 *           (written).
 * Returns KDA_ERR_INVALID_ARG for a null or misaligned pointer and
 * KDA_ERR_CUDA if the lookup or the copy cannot be queued.
 */
kda_status kda_static_workspace_status(uint32_t *status, cudaStream_t stream);

/*
 * kda_spec_verify / kda_spec_commit -- speculative decoding without a state
 * copy per draft token.  "How Kimi K3 is built", section "How to serve two
 * different caches": K3 keeps the small input projections of the draft tokens
 * and recomputes the accepted span on chip, which is cheaper than reading the
 * large recurrent state again for every draft token.
 *
 * kda_spec_verify runs T draft tokens per sequence from `state` and writes
 * their outputs.  The state is read once and NOT modified:
 *   q, k, z  [B, T, H, d_k];  v, o [B, T, H, d_v];  beta [B, T, H]  (dtype)
 *   A        [H, d_k] fp32;   state [B, H, d_k, d_v] fp32 (read only)
 * kda_spec_commit advances each sequence's state by its first n_accept[b]
 * draft tokens (recomputed from k, v, z, beta) and writes it once, in place:
 *   n_accept device int32 [B]; values are clamped into [0, T]; 0 leaves the
 *   state untouched.
 * Both take 1 <= T <= 16, d_k <= 128, d_v <= 128 with d_v a multiple of 4.
 * Arithmetic: commit, verify of fp32 inputs and verify of at most 5 draft
 * tokens run token by token in fp32 (commit with n_accept = T equals T decode
 * steps to fp32 rounding, so a state advanced by speculative decoding carries
 * no extra rounding).  verify of more than 5 bf16 tokens with d_k and d_v
 * multiples of 16 takes the span as one 16-token chunk of the chunked form on
 * the tensor cores (the state's products in bf16, as in the tensor-core
 * prefill; outputs within the same bound, 2e-2 of max |o|); if one of its
 * bounded waits gives up, the outputs of that (b, h) and of the other pairs
 * its CTA has still to walk are NaN.
 */
kda_status kda_spec_verify(const void *q, const void *k, const void *v, const void *z,
                           const void *beta, const float *A, const float *state, void *o, int B,
                           int T, int H, int d_k, int d_v, kda_dtype dtype, cudaStream_t stream);

kda_status kda_spec_commit(const void *k, const void *v, const void *z, const void *beta,
                           const float *A, float *state, const int32_t *n_accept, int B, int T,
                           int H, int d_k, int d_v, kda_dtype dtype, cudaStream_t stream);

/*
 * Instrumentation (not part of the layer's arithmetic).  While `events` is
 * non-NULL, every later prefill, decode or speculative call made on this
 * thread records events[0] on its stream before its first kernel and
 * events[i] after its i-th kernel, for i < n_events; the caller then reads
 * per-kernel times with cudaEventElapsedTime.  The events stay owned by the
 * caller.  Pass NULL to switch recording off.  Returns KDA_OK, or
 * KDA_ERR_INVALID_ARG for n_events < 0.
 */
kda_status kda_set_profile_events(cudaEvent_t *events, int n_events);

/*
 * kda_selftest_bounded_wait -- failure detection, exercised without a fault
 * (not part of the layer's arithmetic; the pages have no counterpart).  The
 * tensor-core kernels bound every mbarrier wait: after about 2 s the wait
 * gives up, the kernel sets a bit in the workspace status word and returns,
 * and the context stays usable.  This launches one thread that waits through
 * that same bounded wait on an mbarrier nothing arrives on (arrive == 0; the
 * call's kernel then runs for about 2 s) or on one that its own arrival
 * completes (arrive != 0), and writes the outcome to *status: 1 if the wait
 * gave up, 0 if it was satisfied.
 *   status  device uint32_t, 4-byte aligned, owned by the caller (written).
 * Asynchronous on `stream`.  Returns KDA_ERR_INVALID_ARG for a null or
 * misaligned status, KDA_ERR_CUDA if the launch fails.
 */
kda_status kda_selftest_bounded_wait(uint32_t *status, int arrive, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
