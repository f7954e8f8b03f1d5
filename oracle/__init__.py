"""fp64 CPU oracle of the Kimi Delta Attention (KDA) layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
leg of the benchmark may import this package.  It shares no code with the CUDA
library and never imports it; the two meet only in the seeded input
generator, which holds none of the layer's arithmetic.

Contents
  gate(z, A)            g = -5 * sigmoid(exp(A) * z), fp64 ("How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents for a million tokens",
                        section "Sequence: three KDA to one global MLA").
  recurrent(...)        the delta-rule recurrence token by token in fp64 (kda_oracle.c;
                        the state update of "Kimi K3 architecture: how an open model with a million-token context competes with market leaders",
                        section "How the Kimi K3 architecture holds a million tokens of
                        context", with the channel-wise gate of the page above).
  chunked(...)          an independently written chunked form (oracle/chunked.py)
                        used to cross-check the recurrence.

Each function takes inputs exactly as handed to the GPU (fp32, or bf16 given as
torch bf16 tensors / numpy uint16 bit patterns) and converts them exactly to
fp64.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build
from .chunked import chunked, chunked_pair  # noqa: F401

_LIB = None

REF_F32 = 0
REF_BF16 = 1


def load_library(path: str):
    """Loads an oracle shared library and declares its C signatures."""
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    fp = ctypes.POINTER(ctypes.c_float)
    vp = ctypes.c_void_p
    lib.kda_ref_gate_scalar.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.kda_ref_gate_scalar.restype = ctypes.c_double
    lib.kda_ref_gate.argtypes = [vp, ctypes.c_int, fp, dp, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_int]
    lib.kda_ref_gate.restype = None
    lib.kda_ref_recurrent.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, fp, fp, i64p,
                                      ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, i64p, ctypes.c_int64, dp, dp,
                                      ctypes.c_int]
    lib.kda_ref_recurrent.restype = ctypes.c_int
    lib.kda_ref_default_threads.argtypes = []
    lib.kda_ref_default_threads.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = load_library(_build.build())
    return _LIB


def default_threads() -> int:
    """Threads the oracle uses when n_threads <= 0 (one per online core)."""
    return int(_lib().kda_ref_default_threads())


def _as_raw(x):
    """Returns (contiguous numpy array, dtype code) for fp32 or bf16 input."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), REF_BF16
            if x.dtype == torch.float32:
                return x.numpy(), REF_F32
            raise TypeError(f"oracle takes fp32 or bf16 inputs, got {x.dtype}")
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, REF_BF16
    if x.dtype == np.float32:
        return x, REF_F32
    raise TypeError(f"oracle takes float32 or bf16 bit patterns (uint16), got {x.dtype}")


def to_f64(x) -> np.ndarray:
    """Exact conversion of an fp32 / bf16 input to fp64."""
    raw, code = _as_raw(x)
    if code == REF_BF16:
        return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return raw.astype(np.float64)


def _f32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().float().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.float32)


def gate_scalar(a: float, z: float) -> float:
    return float(_lib().kda_ref_gate_scalar(float(a), float(z)))


def gate(z, A) -> np.ndarray:
    """g[t, h, c] = -5 * sigmoid(exp(A[h, c]) * z[t, h, c]) in fp64; z is [T, H, dk]."""
    zr, code = _as_raw(z)
    if zr.ndim != 3:
        raise ValueError("z must be [tokens, H, dk]")
    n, H, dk = zr.shape
    Af = _f32(A)
    if Af.shape != (H, dk):
        raise ValueError("A must be [H, dk]")
    out = np.empty((n, H, dk), dtype=np.float64)
    _lib().kda_ref_gate(zr.ctypes.data, code, Af.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), n, H, dk)
    return out


def _flatten_tokens(x, trailing: int):
    """[B, T, ...] or [T_total, ...] -> [B*T, ...] without copying."""
    return x.reshape((-1,) + tuple(x.shape[-trailing:])) if trailing else x.reshape(-1)


def recurrent(q, k, v, z, beta, A, S0=None, cu_seqlens=None, pairs=None, want_o=True,
              n_threads: int = 0):
    """Runs the fp64 recurrence.

    q, k, z: [B, T, H, dk] or packed [T_total, H, dk]; v: [..., H, dv]; beta: [..., H];
    A: [H, dk]; S0: [N, H, dk, dv] fp32 or None; cu_seqlens: [N + 1] token offsets for the
    packed layout (None means fixed length: N = B sequences of T tokens).
    pairs: None for every (seq, head), else an int array [P, 2] of (seq, head).

    Returns (o, S): with pairs None, o is [T_total, H, dv] fp64 (None if not want_o) and
    S is [N, H, dk, dv]; with pairs given, o is a list of [len, dv] arrays and S is
    [P, dk, dv].
    """
    qr, code = _as_raw(q)
    kr, c2 = _as_raw(k)
    vr, c3 = _as_raw(v)
    zr, c4 = _as_raw(z)
    br, c5 = _as_raw(beta)
    if len({code, c2, c3, c4, c5}) != 1:
        raise TypeError("q, k, v, z, beta must share one dtype")
    H, dk = qr.shape[-2], qr.shape[-1]
    dv = vr.shape[-1]
    if cu_seqlens is None:
        if qr.ndim != 4:
            raise ValueError("without cu_seqlens inputs are [B, T, H, d]")
        B, T = qr.shape[0], qr.shape[1]
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
    N = len(cu) - 1
    qr, kr, zr = (np.ascontiguousarray(_flatten_tokens(x, 2)) for x in (qr, kr, zr))
    vr = np.ascontiguousarray(_flatten_tokens(vr, 2))
    br = np.ascontiguousarray(br.reshape(-1, H))
    T_total = qr.shape[0]
    if cu[0] != 0 or cu[-1] != T_total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must rise from 0 to the token count")
    Af = _f32(A)
    S0f = None if S0 is None else _f32(S0).reshape(N, H, dk, dv)

    all_pairs = pairs is None
    if all_pairs:
        pr = np.stack(np.meshgrid(np.arange(N), np.arange(H), indexing="ij"), -1).reshape(-1, 2)
    else:
        pr = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    pr = np.ascontiguousarray(pr, dtype=np.int64)
    lens = cu[pr[:, 0] + 1] - cu[pr[:, 0]]
    o_buf = np.empty(int(lens.sum()) * dv, dtype=np.float64) if want_o else None
    S_buf = np.empty((len(pr), dk, dv), dtype=np.float64)

    dp = ctypes.POINTER(ctypes.c_double)
    fp = ctypes.POINTER(ctypes.c_float)
    i64p = ctypes.POINTER(ctypes.c_int64)
    rc = _lib().kda_ref_recurrent(
        qr.ctypes.data, kr.ctypes.data, vr.ctypes.data, zr.ctypes.data, br.ctypes.data, code,
        Af.ctypes.data_as(fp), None if S0f is None else S0f.ctypes.data_as(fp),
        cu.ctypes.data_as(i64p), N, H, dk, dv, pr.ctypes.data_as(i64p), len(pr),
        None if o_buf is None else o_buf.ctypes.data_as(dp), S_buf.ctypes.data_as(dp),
        int(n_threads))
    if rc != 0:
        raise RuntimeError("kda_ref_recurrent rejected its arguments")

    offs = np.concatenate([[0], np.cumsum(lens * dv)])
    if all_pairs:
        S = S_buf.reshape(N, H, dk, dv)
        if not want_o:
            return None, S
        o = np.empty((T_total, H, dv), dtype=np.float64)
        for p, (n, h) in enumerate(pr):
            o[cu[n]:cu[n + 1], h, :] = o_buf[offs[p]:offs[p + 1]].reshape(-1, dv)
        return o, S
    o_list = None
    if want_o:
        o_list = [o_buf[offs[p]:offs[p + 1]].reshape(-1, dv) for p in range(len(pr))]
    return o_list, S_buf


__all__ = ["gate", "gate_scalar", "recurrent", "chunked", "chunked_pair", "to_f64",
           "default_threads"]
