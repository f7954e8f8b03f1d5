// kda_internal.h -- host-side launchers behind the C ABI (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Records `status` with a printf-style reason for kda_last_error() and returns it.
kda_status report(kda_status status, const char* fmt, ...);

// Records the caller-supplied profiling event i (if any) on `stream`.
void profile_event(int i, cudaStream_t stream);

cudaError_t run_gate(const void* z, const float* A, float* g, int64_t n_tokens, int H, int dk,
                     bool bf16, cudaStream_t stream, int num_sms);

cudaError_t run_decode(const void* q, const void* k, const void* v, const void* z,
                       const void* beta, const float* A, float* state, void* o, int B, int H,
                       int dk, int dv, bool bf16, cudaStream_t stream);

// Speculative decoding over Tn <= 16 draft tokens per sequence: verify (outputs,
// state untouched) or commit (state advanced by n_accept[b] tokens, in place).
cudaError_t run_spec(const void* q, const void* k, const void* v, const void* z, const void* beta,
                     const float* A, float* state, void* o, const int32_t* n_accept, int B, int Tn,
                     int H, int dk, int dv, bool bf16, bool verify, cudaStream_t stream);

// Optional emission of intermediate states: for each sequence, the state after
// (i + 1) * every tokens goes to out[((n * H + h) * max_count + i)], i < max_count.
struct CheckpointSpec {
    float* out = nullptr;       // [N, H, max_count, d_k, d_v] fp32, or null
    int64_t every = 0;          // tokens between checkpoints (a multiple of the chunk)
    int max_count = 0;
};

// Token-by-token SIMT path (fp32 arithmetic), any d_k, d_v <= 128.
cudaError_t run_recurrent(const void* q, const void* k, const void* v, const void* z,
                          const void* beta, const float* A, void* o, const float* S0, float* S1,
                          const int32_t* cu, int n_seqs, int64_t T, int64_t T_total, int H,
                          int dk, int dv, bool bf16, const CheckpointSpec& ck,
                          cudaStream_t stream);

// Chunked tensor-core path (bf16, chunk 64; d_k a multiple of 16 and d_v a
// multiple of 32, both <= 128, zero-padded to 128 on chip).
// A fixed-length batch (T tokens per sequence) may be split into segments
// for the segment-parallel state pass; G = 1 is the plain pass.  The workspace
// covers the packages plus, for G_eff > 1, the per-segment pairs and start
// states (T_seq is the per-sequence length, G the requested segment count).
size_t chunked_tc_workspace_bytes(int n_seqs, int64_t T_total, int H, int64_t T_seq, int G);
int chunked_tc_segments_used(int64_t T_seq, int G);
int chunked_tc_auto_segments(int B, int64_t T, int H, int dk, int dv, int num_sms);
// One launch covers a window of tokens: positions [w0, w1) of every sequence
// of a fixed-length batch (T tokens each), or rows [w0, w1) of a packed one
// (`rows` token rows in all).  A sequence that starts inside the window reads
// S0; one that started before reads Scarry (the state the previous window
// left there); every sequence's state at the window's end goes to S1.
cudaError_t run_chunked_tc(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, void* o, const float* S0,
                           float* S1, const float* Scarry, const int32_t* cu, int n_seqs,
                           int64_t T, int64_t rows, int64_t w0, int64_t w1, int H, int dk,
                           int dv, void* workspace, const CheckpointSpec& ck,
                           cudaStream_t stream, int num_sms, int n_segments);

// The 64-token path runs at most this many tokens at a time (B sequences of a
// fixed-length batch take kWindowTokens / B positions each, rounded down to a
// multiple of 64; a packed batch takes rows), the state carried from window to
// window, so that its workspace is bounded by one window's packages.
constexpr int64_t kWindowTokens = 262144;

// Tensor map (a CUtensorMap, written to `map`) of a [T_total][H][d] bf16
// tensor (2 d a multiple of 16 bytes) with boxes of box_rows tokens x 1 head x
// 128 channels; channels d .. 127 and tokens past T_total read as zeros.
// False if the driver's encoder is unavailable or rejects the description.
bool make_rows_tensor_map(void* map, const void* base, int64_t T_total, int H, int d, int box_rows);

// Chunked tensor-core path with 16-token chunks (bf16; d_k and d_v multiples
// of 16, at most 128): one fused kernel per (sequence, head), no package
// workspace; the workspace holds only the device status word.
constexpr size_t CHUNK16_WORKSPACE_BYTES = 1024;
cudaError_t run_chunk16_tc(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, void* o, const float* S0, float* S1,
                           const int32_t* cu, int n_seqs, int64_t T, int64_t T_total, int H,
                           int dk, int dv, void* workspace, const CheckpointSpec& ck,
                           cudaStream_t stream);

// Speculative verify on the tensor cores: bf16, Tn <= 16, d_k and d_v
// multiples of 16 (<= 128); the Tn draft tokens are one 16-token chunk taken
// from the state (read only).
cudaError_t run_spec_verify_tc(const void* q, const void* k, const void* v, const void* z,
                               const void* beta, const float* A, const float* state, void* o, int B,
                               int Tn, int H, int dk, int dv, cudaStream_t stream);

}  // namespace kda
