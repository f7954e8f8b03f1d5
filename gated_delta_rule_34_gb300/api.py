"""Thin Python binding of the KDA C ABI (include/kda.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, and their data pointers plus the current CUDA stream are handed
to ``libkda.so``.  Every step of the layer runs in the library's kernels; there
is no fallback of any kind, and calling an op without the built library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
PATH_NAMES = {0: "recurrent", 1: "chunked_tc", 2: "chunk16_tc"}
STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
          4: "KDA_ERR_WORKSPACE"}


class KDAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def _declare(lib):
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.kda_status_string.argtypes = [i32]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_gate.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp]
    lib.kda_gate.restype = i32
    lib.kda_chunk_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64,
                                      i32, i32, i32, i32, i32, vp, sz, vp]
    lib.kda_chunk_prefill.restype = i32
    lib.kda_chunk_prefill_checkpoints.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                  i32, i64, i32, i32, i32, i32, i32, vp, i64, i32,
                                                  vp, sz, vp]
    lib.kda_chunk_prefill_checkpoints.restype = i32
    lib.kda_chunk_prefill_workspace_size.argtypes = [i32, i32, i64, i32, i32, i32, i32, i32]
    lib.kda_chunk_prefill_workspace_size.restype = sz
    lib.kda_chunk_prefill_path.argtypes = [i32, i32, i32, i32]
    lib.kda_chunk_prefill_path.restype = i32
    lib.kda_chunk_prefill_from_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                vp, vp, vp, i32, i64, i32, i32, i32, i32, i64, vp,
                                                sz, vp, vp, vp]
    lib.kda_chunk_prefill_from_host.restype = i32
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
    lib.kda_decode_step.restype = i32
    lib.kda_chunk_prefill_static_workspace.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                       i32, i32, i64, i32, i32, i32, i32, i32,
                                                       vp]
    lib.kda_chunk_prefill_static_workspace.restype = i32
    lib.kda_spec_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                    vp]
    lib.kda_spec_verify.restype = i32
    lib.kda_spec_commit.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.kda_spec_commit.restype = i32
    lib.kda_set_profile_events.argtypes = [vp, i32]
    lib.kda_set_profile_events.restype = i32
    lib.kda_selftest_bounded_wait.argtypes = [vp, i32, vp]
    lib.kda_selftest_bounded_wait.restype = i32
    lib.kda_chunk_prefill_segmented.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32,
                                                i32, i32, i32, i32, i32, vp, sz, vp]
    lib.kda_chunk_prefill_segmented.restype = i32
    lib.kda_chunk_prefill_segmented_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32,
                                                               i32]
    lib.kda_chunk_prefill_segmented_workspace_size.restype = sz
    lib.kda_chunk_prefill_auto_segments.argtypes = [i32, i64, i32, i32, i32, i32, i32]
    lib.kda_chunk_prefill_auto_segments.restype = i32
    lib.kda_static_workspace_status.argtypes = [vp, vp]
    lib.kda_static_workspace_status.restype = i32
    return lib


def lib():
    """The loaded ``libkda.so``; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"KDA CUDA library not found at {path}; build it with "
                "`python -m gated_delta_rule_34_gb300.build` (there is no fallback path)")
        _LIB = _declare(ctypes.CDLL(path))
    return _LIB


def _check(status: int):
    if status != 0:
        raise KDAError(status, lib().kda_last_error().decode())


def _on(device):
    """Makes ``device`` current for the duration of a library call: the library launches
    on the current device and resolves its per-device state there."""
    return torch.cuda.device(device)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return KDA_DTYPE_F32
    if t == torch.bfloat16:
        return KDA_DTYPE_BF16
    raise TypeError(f"KDA inputs must be float32 or bfloat16, got {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("KDA ops take CUDA tensors")
            if not t.is_contiguous():
                raise ValueError("KDA ops take contiguous tensors")


def gate(z: torch.Tensor, A: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """g = clamp(-5 * sigmoid(exp(A) * z), -5, 0) in fp32; z is [..., H, d_k], A is [H, d_k]."""
    H, dk = z.shape[-2], z.shape[-1]
    n_tokens = z.numel() // (H * dk) if z.numel() else 0
    if out is None:
        out = torch.empty(z.shape, dtype=torch.float32, device=z.device)
    _need_cuda(z, A, out)
    with _on(z.device):
        _check(lib().kda_gate(_ptr(z), _ptr(A), _ptr(out), n_tokens, H, dk, _dtype_code(z.dtype),
                              _stream(z.device)))
    return out


def prefill_path(d_k: int, d_v: int, chunk: int, dtype: torch.dtype) -> str:
    """Name of the kernel path kda_chunk_prefill takes for these sizes."""
    return PATH_NAMES[lib().kda_chunk_prefill_path(d_k, d_v, chunk, _dtype_code(dtype))]


def workspace_size(n_seqs: int, B: int, T: int, H: int, d_k: int, d_v: int, chunk: int,
                   dtype: torch.dtype) -> int:
    return int(lib().kda_chunk_prefill_workspace_size(n_seqs, B, T, H, d_k, d_v, chunk,
                                                      _dtype_code(dtype)))


def chunk_prefill(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None, chunk: int = 64,
                  output_final_state: bool = True, out=None, final_state=None, workspace=None,
                  checkpoints=None, checkpoint_every: int = 0):
    """Prefill through kda_chunk_prefill.

    q, k, z: [B, T, H, d_k]; v: [B, T, H, d_v]; beta: [B, T, H] (one dtype, fp32 or bf16);
    A: [H, d_k] fp32; initial_state: [N, H, d_k, d_v] fp32 or None; cu_seqlens: int32
    [N + 1] on the device for a packed batch (then B must be 1).
    Returns (o, final_state or None).  A workspace of the required size is allocated
    with torch if none is given.  With ``checkpoints`` (fp32 [N, H, n_slots, d_k, d_v])
    the state after every ``checkpoint_every`` tokens of each sequence is written too
    (kda_chunk_prefill_checkpoints).
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    need = workspace_size(n_seqs, B, T, H, dk, dv, chunk, q.dtype)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    _need_cuda(q, k, v, z, beta, A, out, initial_state, final_state, cu_seqlens, workspace,
               checkpoints)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if checkpoints is None:
        with _on(q.device):
            _check(lib().kda_chunk_prefill(
                _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(out),
                _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), n_seqs, B, T, H, dk, dv,
                chunk, _dtype_code(q.dtype), _ptr(workspace), ws_bytes, _stream(q.device)))
    else:
        if checkpoints.dtype != torch.float32 or checkpoints.dim() != 5:
            raise ValueError("checkpoints must be fp32 [N, H, max_checkpoints, d_k, d_v]")
        with _on(q.device):
            _check(lib().kda_chunk_prefill_checkpoints(
                _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(out),
                _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), n_seqs, B, T, H, dk, dv,
                chunk, _dtype_code(q.dtype), _ptr(checkpoints), int(checkpoint_every),
                checkpoints.shape[2], _ptr(workspace), ws_bytes, _stream(q.device)))
    return out, final_state


def auto_segments(B: int, T: int, H: int, d_k: int, d_v: int, chunk: int = 64,
                  dtype: torch.dtype = torch.bfloat16) -> int:
    """Segment count kda_chunk_prefill uses for a fixed-length batch on the current device."""
    return int(lib().kda_chunk_prefill_auto_segments(B, T, H, d_k, d_v, chunk, _dtype_code(dtype)))


def segmented_workspace_size(B: int, T: int, H: int, d_k: int, d_v: int, n_segments: int,
                             chunk: int = 64, dtype: torch.dtype = torch.bfloat16) -> int:
    return int(lib().kda_chunk_prefill_segmented_workspace_size(B, T, H, d_k, d_v, chunk,
                                                                _dtype_code(dtype), n_segments))


def chunk_prefill_segmented(q, k, v, z, beta, A, n_segments: int, initial_state=None,
                            chunk: int = 64, out=None, final_state=None, workspace=None):
    """Prefill through kda_chunk_prefill_segmented: each of the B fixed-length sequences is
    split into ``n_segments`` segments whose state passes run in parallel.  Same tensors as
    ``chunk_prefill`` without cu_seqlens.  Returns (o, final_state)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = segmented_workspace_size(B, T, H, dk, dv, n_segments, chunk, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _need_cuda(q, k, v, z, beta, A, out, initial_state, final_state, workspace)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(q.device):
        _check(lib().kda_chunk_prefill_segmented(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(out),
            _ptr(initial_state), _ptr(final_state), B, T, H, dk, dv, chunk, _dtype_code(q.dtype),
            int(n_segments), _ptr(workspace), ws_bytes, _stream(q.device)))
    return out, final_state


def chunk_prefill_from_host(q, k, v, z, beta, A, initial_state=None, segment_tokens: int = 8192,
                            out=None, final_state=None, staging=None, workspace=None,
                            copy_streams=None):
    """Prefill through kda_chunk_prefill_from_host: q, k, v, z, beta and the returned o are
    page-locked host tensors ([B, T, H, d] bf16, beta [B, T, H]); A and initial_state are on
    the device.  The host copies of each ``segment_tokens``-token segment overlap the
    kernels of another.  Returns (o on the host, final_state on the device).  Device staging
    buffers, the workspace and the two copy streams are made with torch when not given
    (``staging`` is a dict with q, k, v, z, beta, o device tensors of the host shapes).
    The call is asynchronous on the current stream; ``out`` is valid after it syncs.
    """
    dev = A.device
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    for t in (q, k, v, z, beta):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("host inputs must be contiguous page-locked CPU tensors")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype).pin_memory()
    if final_state is None:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=dev)
    if staging is None:
        staging = {n: torch.empty(t.shape, dtype=t.dtype, device=dev)
                   for n, t in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta), ("o", out))}
    seg = max(64, min(int(segment_tokens), T))
    need = workspace_size(1, 1, seg, H, dk, dv, 64, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if copy_streams is None:
        copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    _need_cuda(A, initial_state, final_state, workspace, *staging.values())
    ws_bytes = workspace.numel() * workspace.element_size()
    with _on(dev):
        _check(lib().kda_chunk_prefill_from_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(out),
            _ptr(staging["q"]), _ptr(staging["k"]), _ptr(staging["v"]), _ptr(staging["z"]),
            _ptr(staging["beta"]), _ptr(staging["o"]), _ptr(initial_state), _ptr(final_state),
            B, T, H, dk, dv, _dtype_code(q.dtype), int(segment_tokens), _ptr(workspace), ws_bytes,
            _stream(dev), ctypes.c_void_p(copy_streams[0].cuda_stream),
            ctypes.c_void_p(copy_streams[1].cuda_stream)))
    return out, final_state


def decode_step(q, k, v, z, beta, A, state, out=None):
    """One token per sequence; updates ``state`` [B, H, d_k, d_v] fp32 in place, returns o."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, z, beta, A, state, out)
    with _on(q.device):
        _check(lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                     _ptr(state), _ptr(out), B, H, dk, dv, _dtype_code(q.dtype),
                                     _stream(q.device)))
    return out


def set_profile_events(events) -> None:
    """Makes later calls on this thread record ``events[0]`` before their first kernel and
    ``events[i]`` after their i-th kernel (torch.cuda.Event objects); None switches it off."""
    if events is None:
        _check(lib().kda_set_profile_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    set_profile_events._keep = arr
    _check(lib().kda_set_profile_events(arr, len(events)))


def selftest_bounded_wait(status: torch.Tensor, arrive: bool) -> None:
    """kda_selftest_bounded_wait: one thread waits through the kernels' bounded mbarrier
    wait, on a barrier nothing arrives on (arrive False: gives up after about 2 s) or one it
    completes itself; writes 1 (gave up) or 0 into ``status`` (an int32 CUDA tensor)."""
    _need_cuda(status)
    if status.dtype != torch.int32 or status.numel() < 1:
        raise ValueError("status must be an int32 CUDA tensor")
    with _on(status.device):
        _check(lib().kda_selftest_bounded_wait(_ptr(status), int(bool(arrive)),
                                               _stream(status.device)))


def chunk_prefill_static_workspace(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None,
                                   chunk: int = 64, output_final_state: bool = True, out=None,
                                   final_state=None):
    """chunk_prefill through kda_chunk_prefill_static_workspace: the library's own fixed
    scratch array replaces the caller workspace, so nothing is allocated for it (the
    outputs are still allocated here unless passed in)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    n_seqs = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if output_final_state and final_state is None:
        final_state = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    if not output_final_state:
        final_state = None
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    _need_cuda(q, k, v, z, beta, A, out, initial_state, final_state, cu_seqlens)
    with _on(q.device):
        _check(lib().kda_chunk_prefill_static_workspace(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(out),
            _ptr(initial_state), _ptr(final_state), _ptr(cu_seqlens), n_seqs, B, T, H, dk, dv, chunk,
            _dtype_code(q.dtype), _stream(q.device)))
    return out, final_state


def spec_verify(q, k, v, z, beta, A, state, out=None):
    """Outputs of T draft tokens per sequence from ``state`` (not modified).

    q, k, z: [B, T, H, d_k]; v: [B, T, H, d_v]; beta: [B, T, H]; state [B, H, d_k, d_v].
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _need_cuda(q, k, v, z, beta, A, state, out)
    with _on(q.device):
        _check(lib().kda_spec_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
                                     _ptr(state), _ptr(out), B, T, H, dk, dv, _dtype_code(q.dtype),
                                     _stream(q.device)))
    return out


def spec_commit(k, v, z, beta, A, state, n_accept):
    """Advances ``state`` in place by the first n_accept[b] draft tokens of each sequence."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if n_accept.dtype != torch.int32:
        raise TypeError("n_accept must be int32")
    _need_cuda(k, v, z, beta, A, state, n_accept)
    with _on(k.device):
        _check(lib().kda_spec_commit(_ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(state),
                                     _ptr(n_accept), B, T, H, dk, dv, _dtype_code(k.dtype),
                                     _stream(k.device)))
    return state


def static_workspace_status(out: torch.Tensor) -> torch.Tensor:
    """kda_static_workspace_status: copies the device status word of the last
    static-workspace prefill on ``out``'s device into ``out`` (an int32 CUDA tensor),
    on the current stream.  0 after the stream finishes means every bounded wait of
    that call was satisfied."""
    _need_cuda(out)
    if out.dtype != torch.int32 or out.numel() < 1:
        raise ValueError("out must be an int32 CUDA tensor")
    with _on(out.device):
        _check(lib().kda_static_workspace_status(_ptr(out), _stream(out.device)))
    return out
