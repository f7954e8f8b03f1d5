// kda_api.cu -- the C ABI: argument validation, path choice and launches.
//
// Every check happens on the host before anything is launched; nothing here
// reads device memory.  Each entry point returns a kda_status and records a
// one-line reason for the last failure in thread-local storage.
#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

thread_local char g_last_error[512] = "";
thread_local cudaEvent_t* g_prof_events = nullptr;
thread_local int g_prof_n = 0;

kda_status fail(kda_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

kda_status ok() {
    g_last_error[0] = '\0';
    return KDA_OK;
}

kda_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 148;
    return sms > 0 ? sms : 148;
}

bool valid_dtype(kda_dtype d) { return d == KDA_DTYPE_F32 || d == KDA_DTYPE_BF16; }

// A pointer that must be present and 16-byte aligned.
#define KDA_REQUIRE_PTR(p)                                                              \
    do {                                                                                \
        if ((p) == nullptr) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", #p);         \
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
    } while (0)

#define KDA_OPTIONAL_PTR(p)                                                             \
    do {                                                                                \
        if ((p) != nullptr && !aligned16(p))                                            \
            return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p);          \
    } while (0)

// The tensor-core path: bf16, chunk 64, d_k a multiple of 16 and d_v a
// multiple of 32 (one 32-column state tile per CTA of the state pass), both
// at most 128; narrower heads are zero-padded to 128 on chip.
bool use_chunked_tc(int dk, int dv, int chunk, kda_dtype dtype) {
    return dtype == KDA_DTYPE_BF16 && chunk == 64 && dk >= 16 && dk <= 128 && dk % 16 == 0 &&
           dv >= 32 && dv <= 128 && dv % 32 == 0;
}

// The 16-token tensor-core path: bf16, chunk 16, d_k and d_v multiples of 16
// in [16, 128].
bool use_chunk16_tc(int dk, int dv, int chunk, kda_dtype dtype) {
    return dtype == KDA_DTYPE_BF16 && chunk == 16 && dk >= 16 && dk <= 128 && dk % 16 == 0 &&
           dv >= 16 && dv <= 128 && dv % 16 == 0;
}

}  // namespace

namespace kda {
kda_status report(kda_status status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

void profile_event(int i, cudaStream_t stream) {
    if (g_prof_events && i < g_prof_n) cudaEventRecord(g_prof_events[i], stream);
}
}  // namespace kda

extern "C" {

kda_status kda_set_profile_events(cudaEvent_t* events, int n_events) {
    if (n_events < 0) return fail(KDA_ERR_INVALID_ARG, "n_events must be >= 0");
    g_prof_events = n_events > 0 ? events : nullptr;
    g_prof_n = events ? n_events : 0;
    return ok();
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error(void) { return g_last_error; }

kda_status kda_gate(const void* z, const float* A, float* g, int64_t n_tokens, int H, int d_k,
                    kda_dtype z_dtype, cudaStream_t stream) {
    if (!valid_dtype(z_dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)z_dtype);
    if (n_tokens < 0 || H <= 0 || d_k <= 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes n_tokens=%lld H=%d d_k=%d",
                    (long long)n_tokens, H, d_k);
    if (n_tokens == 0) return ok();
    KDA_REQUIRE_PTR(z);
    KDA_REQUIRE_PTR(A);
    KDA_REQUIRE_PTR(g);
    return cuda_status(kda::run_gate(z, A, g, n_tokens, H, d_k, z_dtype == KDA_DTYPE_BF16, stream,
                                     device_sm_count()),
                       "kda_gate launch");
}

kda_prefill_path kda_chunk_prefill_path(int d_k, int d_v, int chunk, kda_dtype dtype) {
    if (use_chunked_tc(d_k, d_v, chunk, dtype)) return KDA_PATH_CHUNKED_TC;
    if (use_chunk16_tc(d_k, d_v, chunk, dtype)) return KDA_PATH_CHUNK16_TC;
    return KDA_PATH_RECURRENT;
}

// Window of the 64-token path (see kda::kWindowTokens): for a fixed-length
// batch of B sequences, the positions per sequence (a multiple of 64, so that
// B of them hold at most kWindowTokens tokens); for a packed batch, rows.
static int64_t window_len(bool fixed, int B) {
    if (!fixed || B <= 1) return kda::kWindowTokens;
    const int64_t w = kda::kWindowTokens / B / 64 * 64;
    return w < 64 ? 64 : w;
}
static int64_t window_span(bool fixed, int B, int64_t T) {
    const int64_t w = window_len(fixed, B);
    return T < w ? T : w;
}

// Segment count for kda_chunk_prefill: automatic for fixed-length batches on
// the tensor-core path (n_seqs == B marks a fixed-length query), 1 otherwise.
static int auto_segments(int n_seqs, int B, int64_t T, int H, int d_k, int d_v) {
    if (n_seqs != B) return 1;
    return kda::chunked_tc_auto_segments(B, window_span(true, B, T), H, d_k, d_v, device_sm_count());
}

// Workspace of the 64-token path for a fixed-length batch (`fixed`: B sequences
// of T tokens) or a packed one (T tokens in all): one window's packages, the
// segment records (fixed length only) and, when the call runs in several
// windows, a carry area for the states between them (at the end).
static size_t carry_bytes(int n_seqs, int H) { return (size_t)n_seqs * H * 128 * 128 * 4; }
static size_t tc_workspace(bool fixed, int n_seqs, int B, int64_t T, int H, int G) {
    const int64_t w = window_span(fixed, B, T);
    size_t bytes = fixed ? kda::chunked_tc_workspace_bytes(n_seqs, (int64_t)B * w, H, w, G)
                         : kda::chunked_tc_workspace_bytes(n_seqs, w, H, w, 1);
    if (T > w) bytes += carry_bytes(n_seqs, H);
    return bytes;
}

size_t kda_chunk_prefill_workspace_size(int n_seqs, int B, int64_t T, int H, int d_k, int d_v,
                                        int chunk, kda_dtype dtype) {
    if (n_seqs <= 0 || B <= 0 || T < 0 || H <= 0) return 0;
    if (use_chunk16_tc(d_k, d_v, chunk, dtype)) return kda::CHUNK16_WORKSPACE_BYTES;
    if (!use_chunked_tc(d_k, d_v, chunk, dtype)) return 0;
    // n_seqs == B is read as a fixed-length batch; a packed batch's need is the
    // larger one only when it holds a single sequence, so return the larger.
    const size_t fixed = tc_workspace(n_seqs == B, n_seqs, B, T, H,
                                      auto_segments(n_seqs, B, T, H, d_k, d_v));
    const size_t packed = tc_workspace(false, n_seqs, 1, (int64_t)B * T, H, 1);
    return n_seqs == B && B == 1 && packed > fixed ? packed : fixed;
}

size_t kda_chunk_prefill_segmented_workspace_size(int B, int64_t T, int H, int d_k, int d_v,
                                                  int chunk, kda_dtype dtype, int n_segments) {
    if (B <= 0 || T < 0 || H <= 0 || n_segments <= 0) return 0;
    if (!use_chunked_tc(d_k, d_v, chunk, dtype)) return 0;
    return tc_workspace(true, B, B, T, H, n_segments);
}

int kda_chunk_prefill_auto_segments(int B, int64_t T, int H, int d_k, int d_v, int chunk,
                                    kda_dtype dtype) {
    if (B <= 0 || T <= 0 || H <= 0 || !use_chunked_tc(d_k, d_v, chunk, dtype)) return 1;
    return kda::chunked_tc_segments_used(window_span(true, B, T), auto_segments(B, B, T, H, d_k, d_v));
}

static kda_status prefill_impl(const void* q, const void* k, const void* v, const void* z,
                               const void* beta, const float* A, void* o,
                               const float* initial_state, float* final_state,
                               const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                               int d_k, int d_v, int chunk, kda_dtype dtype, void* workspace,
                               size_t workspace_bytes, const kda::CheckpointSpec& ck,
                               cudaStream_t stream, int n_segments = 0) {
    if (!valid_dtype(dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B <= 0 || T < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || n_seqs <= 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes B=%d T=%lld H=%d d_k=%d d_v=%d n_seqs=%d", B,
                    (long long)T, H, d_k, d_v, n_seqs);
    if (chunk != 16 && chunk != 64)
        return fail(KDA_ERR_INVALID_ARG, "chunk must be 16 or 64, got %d", chunk);
    if (cu_seqlens) {
        if (B != 1) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens requires B == 1 (got %d)", B);
        if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens is not 4-byte aligned");
    } else if (n_seqs != B) {
        return fail(KDA_ERR_INVALID_ARG, "without cu_seqlens n_seqs must equal B (%d vs %d)",
                    n_seqs, B);
    }
    if (d_k > 128 || d_v > 128)
        return fail(KDA_ERR_UNSUPPORTED, "head sizes above 128 are not supported (d_k=%d d_v=%d)",
                    d_k, d_v);
    if (H > 65535 || n_seqs > 65535)
        return fail(KDA_ERR_UNSUPPORTED, "H and n_seqs must be <= 65535");
    const int64_t T_total = (int64_t)B * T;
    if (T_total > 0) {
        KDA_REQUIRE_PTR(q);
        KDA_REQUIRE_PTR(k);
        KDA_REQUIRE_PTR(v);
        KDA_REQUIRE_PTR(z);
        KDA_REQUIRE_PTR(beta);
        KDA_REQUIRE_PTR(o);
    }
    KDA_REQUIRE_PTR(A);
    KDA_OPTIONAL_PTR(initial_state);
    KDA_OPTIONAL_PTR(final_state);
    const bool bf16 = dtype == KDA_DTYPE_BF16;

    if (use_chunked_tc(d_k, d_v, chunk, dtype)) {
        // TMA tile coordinates are 32-bit: token indices must fit.
        if (T_total > (int64_t)INT32_MAX - 64)
            return fail(KDA_ERR_UNSUPPORTED, "the tensor-core path takes fewer than 2^31 tokens (%lld)",
                        (long long)T_total);
        // Segments: n_segments > 0 asks for that many (fixed-length batches
        // only); 0 picks them automatically, falling back to the plain pass when
        // the workspace only covers that.
        const bool fixed = cu_seqlens == nullptr;
        int G = 1;
        if (n_segments > 0) {
            if (!fixed && n_segments > 1)
                return fail(KDA_ERR_UNSUPPORTED, "segments need a fixed-length batch (cu_seqlens == NULL)");
            if ((int64_t)B * kda::chunked_tc_segments_used(window_span(true, B, T), n_segments) > 65535)
                return fail(KDA_ERR_UNSUPPORTED, "B x segments must be <= 65535");
            G = n_segments;
        } else if (fixed) {
            G = auto_segments(n_seqs, B, T, H, d_k, d_v);
            if (G > 1 && workspace_bytes < tc_workspace(true, n_seqs, B, T, H, G)) G = 1;
        }
        const size_t need = fixed ? tc_workspace(true, n_seqs, B, T, H, G)
                                  : tc_workspace(false, n_seqs, 1, T_total, H, 1);
        if (workspace == nullptr || workspace_bytes < need)
            return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu at %p", need,
                        workspace_bytes, workspace);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
        // Windows: at most kWindowTokens tokens per launch pair (window_len
        // positions of every sequence when fixed, rows when packed).  The states
        // cross windows in final_state, or in the workspace's carry area when the
        // caller wants no final state.
        const int64_t span = fixed ? T : T_total;
        const int64_t W = window_len(fixed, B);
        float* carry = final_state;
        if (span > W && carry == nullptr)
            carry = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + need -
                                             carry_bytes(n_seqs, H));
        int64_t w0 = 0;
        do {
            const int64_t w1 = span - w0 < W ? span : w0 + W;
            const cudaError_t e = kda::run_chunked_tc(
                q, k, v, z, beta, A, o, initial_state, carry, carry, cu_seqlens, n_seqs, T,
                T_total, w0, w1, H, d_k, d_v, workspace, ck, stream, device_sm_count(), G);
            if (e != cudaSuccess) return cuda_status(e, "kda_chunk_prefill (chunked tensor-core path)");
            w0 = w1;
        } while (w0 < span);
        return ok();
    }
    if (use_chunk16_tc(d_k, d_v, chunk, dtype)) {
        if (workspace == nullptr || workspace_bytes < kda::CHUNK16_WORKSPACE_BYTES)
            return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu at %p",
                        kda::CHUNK16_WORKSPACE_BYTES, workspace_bytes, workspace);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(KDA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
        if (n_segments > 1) return fail(KDA_ERR_UNSUPPORTED, "segments run on the 64-token path only");
        if (T_total > (int64_t)INT32_MAX - 16)
            return fail(KDA_ERR_UNSUPPORTED, "the tensor-core path takes fewer than 2^31 tokens (%lld)",
                        (long long)T_total);
        return cuda_status(kda::run_chunk16_tc(q, k, v, z, beta, A, o, initial_state, final_state,
                                               cu_seqlens, n_seqs, T, T_total, H, d_k, d_v,
                                               workspace, ck, stream),
                           "kda_chunk_prefill (16-token tensor-core path)");
    }
    kda::profile_event(0, stream);
    const cudaError_t e = kda::run_recurrent(q, k, v, z, beta, A, o, initial_state, final_state,
                                             cu_seqlens, n_seqs, T, T_total, H, d_k, d_v, bf16,
                                             ck, stream);
    kda::profile_event(1, stream);
    return cuda_status(e, "kda_chunk_prefill (recurrent path)");
}

kda_status kda_chunk_prefill(const void* q, const void* k, const void* v, const void* z,
                             const void* beta, const float* A, void* o,
                             const float* initial_state, float* final_state,
                             const int32_t* cu_seqlens, int n_seqs, int B, int64_t T, int H,
                             int d_k, int d_v, int chunk, kda_dtype dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    return prefill_impl(q, k, v, z, beta, A, o, initial_state, final_state, cu_seqlens, n_seqs, B,
                        T, H, d_k, d_v, chunk, dtype, workspace, workspace_bytes,
                        kda::CheckpointSpec{}, stream);
}

kda_status kda_chunk_prefill_segmented(const void* q, const void* k, const void* v, const void* z,
                                       const void* beta, const float* A, void* o,
                                       const float* initial_state, float* final_state, int B,
                                       int64_t T, int H, int d_k, int d_v, int chunk,
                                       kda_dtype dtype, int n_segments, void* workspace,
                                       size_t workspace_bytes, cudaStream_t stream) {
    if (n_segments <= 0)
        return fail(KDA_ERR_INVALID_ARG, "n_segments must be >= 1 (got %d)", n_segments);
    if (!use_chunked_tc(d_k, d_v, chunk, dtype))
        return fail(KDA_ERR_UNSUPPORTED, "segments run on the tensor-core path only (bf16, chunk 64, "
                                         "d_k a multiple of 16 and d_v a multiple of 32, both <= 128)");
    return prefill_impl(q, k, v, z, beta, A, o, initial_state, final_state, nullptr, B, B, T, H,
                        d_k, d_v, chunk, dtype, workspace, workspace_bytes, kda::CheckpointSpec{},
                        stream, n_segments);
}

kda_status kda_chunk_prefill_from_host(const void* q_h, const void* k_h, const void* v_h,
                                       const void* z_h, const void* beta_h, const float* A,
                                       void* o_h, void* q_d, void* k_d, void* v_d, void* z_d,
                                       void* beta_d, void* o_d, const float* initial_state,
                                       float* final_state, int B, int64_t T, int H, int d_k,
                                       int d_v, kda_dtype dtype, int64_t segment_tokens,
                                       void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream, cudaStream_t h2d_stream,
                                       cudaStream_t d2h_stream) {
    if (!valid_dtype(dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B <= 0 || T < 0 || H <= 0 || H > 65535)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes B=%d T=%lld H=%d", B, (long long)T, H);
    if (!use_chunked_tc(d_k, d_v, 64, dtype))
        return fail(KDA_ERR_UNSUPPORTED, "kda_chunk_prefill_from_host supports the tensor-core "
                                         "path only: bf16, d_k a multiple of 16 and d_v a multiple "
                                         "of 32, both <= 128 (d_k=%d d_v=%d dtype=%d)",
                    d_k, d_v, (int)dtype);
    if (segment_tokens <= 0 || segment_tokens % 64 != 0)
        return fail(KDA_ERR_INVALID_ARG, "segment_tokens must be a positive multiple of 64, got %lld",
                    (long long)segment_tokens);
    if (stream == h2d_stream || stream == d2h_stream || h2d_stream == d2h_stream)
        return fail(KDA_ERR_INVALID_ARG, "the compute, host-to-device and device-to-host streams "
                                         "must differ");
    KDA_REQUIRE_PTR(A);
    KDA_REQUIRE_PTR(final_state);
    KDA_OPTIONAL_PTR(initial_state);
    if (T == 0)
        return prefill_impl(nullptr, nullptr, nullptr, nullptr, nullptr, A, nullptr, initial_state,
                            final_state, nullptr, B, B, 0, H, d_k, d_v, 64, dtype, workspace,
                            workspace_bytes, kda::CheckpointSpec{}, stream);
    if (!q_h || !k_h || !v_h || !z_h || !beta_h || !o_h)
        return fail(KDA_ERR_INVALID_ARG, "a host input or output pointer is NULL");
    KDA_REQUIRE_PTR(q_d);
    KDA_REQUIRE_PTR(k_d);
    KDA_REQUIRE_PTR(v_d);
    KDA_REQUIRE_PTR(z_d);
    KDA_REQUIRE_PTR(beta_d);
    KDA_REQUIRE_PTR(o_d);
    const int64_t seg = segment_tokens < T ? segment_tokens : T;
    const size_t need = tc_workspace(true, 1, 1, seg, H, 1);
    if (workspace == nullptr || workspace_bytes < need)
        return fail(KDA_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu", need,
                    workspace_bytes);

    const size_t es = 2;                                    // bf16
    const size_t qb = (size_t)H * d_k * es, vb = (size_t)H * d_v * es, bb = (size_t)H * es;
    const size_t sb = (size_t)H * d_k * d_v;                // floats per sequence state
    cudaEvent_t ev_in = nullptr, ev_out = nullptr;
    cudaError_t e = cudaEventCreateWithFlags(&ev_in, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_out, cudaEventDisableTiming);
    // The copy streams start after the work already queued on `stream`.
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h2d_stream, ev_in, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d2h_stream, ev_in, 0);
    kda_status st = KDA_OK;
    auto cp = [&](void* dst, const void* src, size_t off, size_t n, cudaMemcpyKind kind,
                  cudaStream_t s) {
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off,
                                n, kind, s);
    };
    for (int b = 0; b < B && e == cudaSuccess && st == KDA_OK; ++b) {
        for (int64_t t0 = 0; t0 < T && e == cudaSuccess && st == KDA_OK; t0 += seg) {
            const int64_t len = (T - t0) < seg ? (T - t0) : seg;
            const size_t tok = (size_t)b * T + t0;
            cp(q_d, q_h, tok * qb, len * qb, cudaMemcpyHostToDevice, h2d_stream);
            cp(k_d, k_h, tok * qb, len * qb, cudaMemcpyHostToDevice, h2d_stream);
            cp(v_d, v_h, tok * vb, len * vb, cudaMemcpyHostToDevice, h2d_stream);
            cp(z_d, z_h, tok * qb, len * qb, cudaMemcpyHostToDevice, h2d_stream);
            cp(beta_d, beta_h, tok * bb, len * bb, cudaMemcpyHostToDevice, h2d_stream);
            if (e == cudaSuccess) e = cudaEventRecord(ev_in, h2d_stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev_in, 0);
            if (e != cudaSuccess) break;
            float* S = final_state + (size_t)b * sb;
            const float* S_in = t0 == 0 ? (initial_state ? initial_state + (size_t)b * sb : nullptr) : S;
            st = prefill_impl(static_cast<const char*>(q_d) + tok * qb,
                              static_cast<const char*>(k_d) + tok * qb,
                              static_cast<const char*>(v_d) + tok * vb,
                              static_cast<const char*>(z_d) + tok * qb,
                              static_cast<const char*>(beta_d) + tok * bb, A,
                              static_cast<char*>(o_d) + tok * vb, S_in, S, nullptr, 1, 1, len, H,
                              d_k, d_v, 64, dtype, workspace, workspace_bytes,
                              kda::CheckpointSpec{}, stream, 1);
            if (st != KDA_OK) break;
            if (e == cudaSuccess) e = cudaEventRecord(ev_out, stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(d2h_stream, ev_out, 0);
            cp(o_h, o_d, tok * vb, len * vb, cudaMemcpyDeviceToHost, d2h_stream);
        }
    }
    // `stream` finishes after the last copy back.
    if (e == cudaSuccess) e = cudaEventRecord(ev_out, d2h_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev_out, 0);
    if (ev_in) cudaEventDestroy(ev_in);
    if (ev_out) cudaEventDestroy(ev_out);
    if (st != KDA_OK) return st;
    return cuda_status(e, "kda_chunk_prefill_from_host");
}

kda_status kda_chunk_prefill_checkpoints(const void* q, const void* k, const void* v,
                                         const void* z, const void* beta, const float* A, void* o,
                                         const float* initial_state, float* final_state,
                                         const int32_t* cu_seqlens, int n_seqs, int B, int64_t T,
                                         int H, int d_k, int d_v, int chunk, kda_dtype dtype,
                                         float* checkpoints, int64_t checkpoint_every,
                                         int max_checkpoints, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream) {
    kda::CheckpointSpec ck;
    if (checkpoints != nullptr) {
        if (!aligned16(checkpoints))
            return fail(KDA_ERR_INVALID_ARG, "checkpoints is not 16-byte aligned");
        if (chunk != 16 && chunk != 64)
            return fail(KDA_ERR_INVALID_ARG, "chunk must be 16 or 64, got %d", chunk);
        if (checkpoint_every <= 0 || checkpoint_every % chunk != 0)
            return fail(KDA_ERR_INVALID_ARG,
                        "checkpoint_every must be a positive multiple of the chunk (%lld, chunk %d)",
                        (long long)checkpoint_every, chunk);
        if (max_checkpoints <= 0)
            return fail(KDA_ERR_INVALID_ARG, "max_checkpoints must be positive (got %d)",
                        max_checkpoints);
        ck.out = checkpoints;
        ck.every = checkpoint_every;
        ck.max_count = max_checkpoints;
    }
    return prefill_impl(q, k, v, z, beta, A, o, initial_state, final_state, cu_seqlens, n_seqs, B,
                        T, H, d_k, d_v, chunk, dtype, workspace, workspace_bytes, ck, stream);
}

kda_status kda_decode_step(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, float* state, void* o, int B, int H,
                           int d_k, int d_v, kda_dtype dtype, cudaStream_t stream) {
    if (!valid_dtype(dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || H <= 0 || d_k <= 0 || d_v <= 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes B=%d H=%d d_k=%d d_v=%d", B, H, d_k, d_v);
    if (d_k > 128 || d_v > 128 || d_v % 4 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "decode needs d_k <= 128 and d_v <= 128, d_v %% 4 == 0 "
                    "(d_k=%d d_v=%d)", d_k, d_v);
    if ((int64_t)B * H > 0x7fffffffLL)
        return fail(KDA_ERR_UNSUPPORTED, "B*H too large");
    if (B == 0) return ok();
    KDA_REQUIRE_PTR(q);
    KDA_REQUIRE_PTR(k);
    KDA_REQUIRE_PTR(v);
    KDA_REQUIRE_PTR(z);
    KDA_REQUIRE_PTR(beta);
    KDA_REQUIRE_PTR(A);
    KDA_REQUIRE_PTR(state);
    KDA_REQUIRE_PTR(o);
    kda::profile_event(0, stream);
    const cudaError_t e = kda::run_decode(q, k, v, z, beta, A, state, o, B, H, d_k, d_v,
                                          dtype == KDA_DTYPE_BF16, stream);
    kda::profile_event(1, stream);
    return cuda_status(e, "kda_decode_step launch");
}

}  // extern "C"

extern "C" {

static kda_status spec_checks(int B, int T, int H, int d_k, int d_v, kda_dtype dtype) {
    if (!valid_dtype(dtype)) return fail(KDA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || H <= 0 || d_k <= 0 || d_v <= 0 || T <= 0)
        return fail(KDA_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d d_k=%d d_v=%d", B, T, H, d_k,
                    d_v);
    if (T > 16) return fail(KDA_ERR_UNSUPPORTED, "at most 16 draft tokens per call (got %d)", T);
    if (d_k > 128 || d_v > 128 || d_v % 4 != 0)
        return fail(KDA_ERR_UNSUPPORTED, "needs d_k <= 128 and d_v <= 128, d_v %% 4 == 0 "
                    "(d_k=%d d_v=%d)", d_k, d_v);
    if ((int64_t)B * H > 0x7fffffffLL) return fail(KDA_ERR_UNSUPPORTED, "B*H too large");
    return KDA_OK;
}

kda_status kda_spec_verify(const void* q, const void* k, const void* v, const void* z,
                           const void* beta, const float* A, const float* state, void* o, int B,
                           int T, int H, int d_k, int d_v, kda_dtype dtype, cudaStream_t stream) {
    const kda_status st = spec_checks(B, T, H, d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (B == 0) return ok();
    KDA_REQUIRE_PTR(q);
    KDA_REQUIRE_PTR(k);
    KDA_REQUIRE_PTR(v);
    KDA_REQUIRE_PTR(z);
    KDA_REQUIRE_PTR(beta);
    KDA_REQUIRE_PTR(A);
    KDA_REQUIRE_PTR(state);
    KDA_REQUIRE_PTR(o);
    kda::profile_event(0, stream);
    // bf16 heads with d_k and d_v multiples of 16 and more than 5 draft tokens:
    // the draft span is one 16-token chunk on the tensor cores; otherwise token
    // by token in fp32 (up to 5 tokens that is faster: 0.128 against 0.203 ms at
    // T = 1, 0.175 against 0.208 ms at T = 4, 0.201 against 0.210 ms at T = 5,
    // against 0.214 / 0.212 ms at T = 6, for B = 256, H = 32).
    const bool tc = dtype == KDA_DTYPE_BF16 && d_k % 16 == 0 && d_v % 16 == 0 && T > 5;
    const cudaError_t e =
        tc ? kda::run_spec_verify_tc(q, k, v, z, beta, A, state, o, B, T, H, d_k, d_v, stream)
           : kda::run_spec(q, k, v, z, beta, A, const_cast<float*>(state), o, nullptr, B, T, H, d_k,
                           d_v, dtype == KDA_DTYPE_BF16, true, stream);
    kda::profile_event(1, stream);
    return cuda_status(e, "kda_spec_verify launch");
}

kda_status kda_spec_commit(const void* k, const void* v, const void* z, const void* beta,
                           const float* A, float* state, const int32_t* n_accept, int B, int T,
                           int H, int d_k, int d_v, kda_dtype dtype, cudaStream_t stream) {
    const kda_status st = spec_checks(B, T, H, d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (B == 0) return ok();
    KDA_REQUIRE_PTR(k);
    KDA_REQUIRE_PTR(v);
    KDA_REQUIRE_PTR(z);
    KDA_REQUIRE_PTR(beta);
    KDA_REQUIRE_PTR(A);
    KDA_REQUIRE_PTR(state);
    if (n_accept == nullptr) return fail(KDA_ERR_INVALID_ARG, "n_accept is NULL");
    if ((reinterpret_cast<uintptr_t>(n_accept) & 3u) != 0)
        return fail(KDA_ERR_INVALID_ARG, "n_accept is not 4-byte aligned");
    kda::profile_event(0, stream);
    const cudaError_t e = kda::run_spec(nullptr, k, v, z, beta, A, state, nullptr, n_accept, B, T,
                                        H, d_k, d_v, dtype == KDA_DTYPE_BF16, false, stream);
    kda::profile_event(1, stream);
    return cuda_status(e, "kda_spec_commit launch");
}

}  // extern "C"
