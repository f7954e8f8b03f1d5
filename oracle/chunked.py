"""Chunked form of the KDA recurrence, written independently of kda_oracle.c (fp64, numpy).

TEST INFRASTRUCTURE ONLY: it exists to cross-check the token-by-token oracle.

The pages say the kernel runs the tokens of one chunk in parallel and then
passes the state on ("Kimi K3 architecture: how an open model with a
million-token context competes with market leaders", section "Chip level: the
specialised FlashKDA kernel") but print no equations, so the algebra here is
derived directly from the recurrence S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,
o_t = S_t^T q_t.  Inside a chunk with start state S0 and G_t = sum_{s<=t} g_s
(per channel, cumulative log-decay from the chunk start):

  delta  u_t = b_t (v_t - (Diag(a_t) S_{t-1})^T k_t),  so  S_t = Diag(a_t) S_{t-1} + k_t u_t^T
  unroll S_t = Diag(e^{G_t}) S0 + sum_{s<=t} Diag(e^{G_t - G_s}) k_s u_s^T
  hence  (I + A) U = Diag(b) (V - K^g S0),  A_ts = b_t sum_c k_tc k_sc e^{G_tc - G_sc}  (s < t)
         O = Q^g S0 + P U,                   P_ts = sum_c q_tc k_sc e^{G_tc - G_sc}      (s <= t)
         S_C = Diag(e^{G_C}) S0 + (K^C)^T U, K^C_s = k_s (.) e^{G_C - G_s}
  with K^g_t = k_t (.) e^{G_t}, Q^g_t = q_t (.) e^{G_t}.

The decay factors are taken directly as e^{G_t - G_s} (a difference, never
factored), and (I + A) is solved by forward substitution.  The last chunk of a
sequence may be short; chunk size does not change the exact result.
"""
from __future__ import annotations

import numpy as np


def _gate64(z: np.ndarray, A: np.ndarray) -> np.ndarray:
    """g = -5 * sigmoid(exp(A) * z) in fp64.

    "How Kimi K3 is built: 2.8 trillion parameters, linear attention and agents
    for a million tokens", section "Sequence: three KDA to one global MLA".
    """
    x = np.exp(A) * z
    with np.errstate(over="ignore"):
        return -5.0 / (1.0 + np.exp(-x))


def chunked_pair(q, k, v, g, beta, S0, C: int):
    """One (sequence, head).  q, k, g: [L, dk]; v: [L, dv]; beta: [L]; S0: [dk, dv]; all fp64."""
    L, dk = q.shape
    dv = v.shape[1]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((L, dv))
    for t0 in range(0, L, C):
        sl = slice(t0, min(t0 + C, L))
        qc, kc, vc, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        n = qc.shape[0]
        G = np.cumsum(gc, axis=0)
        E = np.exp(G[:, None, :] - G[None, :, :])          # [t, s, c] = e^{G_tc - G_sc}
        A = np.tril(bc[:, None] * np.einsum("tc,sc,tsc->ts", kc, kc, E), -1)
        P = np.tril(np.einsum("tc,sc,tsc->ts", qc, kc, E))
        Kg = kc * np.exp(G)
        Qg = qc * np.exp(G)
        R = bc[:, None] * (vc - Kg @ S)
        U = np.zeros((n, dv))
        for t in range(n):                                  # (I + A) U = R, unit lower
            U[t] = R[t] - A[t, :t] @ U[:t]
        o[sl] = Qg @ S + P @ U
        Kc = kc * np.exp(G[-1][None, :] - G)
        S = np.exp(G[-1])[:, None] * S + Kc.T @ U
    return o, S


def chunked(q, k, v, z, beta, A, S0=None, cu_seqlens=None, C: int = 64):
    """Every (sequence, head) through chunked_pair.

    Inputs as for oracle.recurrent (fp32 or bf16, converted exactly to fp64).
    Returns o [T_total, H, dv] and S [N, H, dk, dv] in fp64.
    """
    from . import to_f64
    qf, kf, vf, zf, bf = (to_f64(x) for x in (q, k, v, z, beta))
    H, dk = qf.shape[-2], qf.shape[-1]
    dv = vf.shape[-1]
    if cu_seqlens is None:
        B, T = qf.shape[0], qf.shape[1]
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                        dtype=np.int64)
    qf, kf, zf = (x.reshape(-1, H, dk) for x in (qf, kf, zf))
    vf = vf.reshape(-1, H, dv)
    bf = bf.reshape(-1, H)
    Af = to_f64(A.float() if hasattr(A, "float") else np.asarray(A, np.float32))
    N = len(cu) - 1
    S0f = np.zeros((N, H, dk, dv)) if S0 is None else to_f64(
        S0.float() if hasattr(S0, "float") else np.asarray(S0, np.float32)).reshape(N, H, dk, dv)
    g = _gate64(zf, Af[None, :, :])
    o = np.zeros((qf.shape[0], H, dv))
    S = np.zeros((N, H, dk, dv))
    for n in range(N):
        sl = slice(int(cu[n]), int(cu[n + 1]))
        for h in range(H):
            o[sl, h], S[n, h] = chunked_pair(qf[sl, h], kf[sl, h], vf[sl, h], g[sl, h],
                                             bf[sl, h], S0f[n, h], C)
    return o, S
