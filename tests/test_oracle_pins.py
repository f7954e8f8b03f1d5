"""Pins the fp64 oracle to facts that do not come from the oracle itself.

Every check here is CPU-only.  The pins are chosen so that a plausible slip in
the oracle (a dropped decay, erase and decay swapped, a wrong sign, o read
before the update, S transposed, a wrong token or head index) fails at least
one of them; tests/test_oracle_mutants.py plants such slips in a copy of the
oracle and checks that they are caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = float("-inf")


def _val(x):
    table = {"inf": math.inf, "-inf": -math.inf, "ln3": math.log(3.0), "ln2": math.log(2.0),
             "ln3/2": math.log(3.0) / 2, "-ln3/2": -math.log(3.0) / 2}
    return table[x] if isinstance(x, str) else float(x)


# --------------------------------------------------------------------------- gate
def test_gate_golden_points():
    with open(os.path.join(GOLDEN, "gate_points.json")) as f:
        gold = json.load(f)
    assert gold["g_min"] == -5.0
    for p in gold["points"]:
        g = oracle.gate_scalar(_val(p["A"]), _val(p["z"]))
        assert g == pytest.approx(p["g"], abs=1e-15), p


def test_gate_range_and_alpha_bound():
    rng = np.random.default_rng(0)
    z = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 50, 4000),
                        [0.0, 1e30, -1e30, 8.0, -8.0]]).astype(np.float32)
    A = rng.normal(0, 2, (1, len(z))).astype(np.float32)
    g = oracle.gate(z.reshape(1, 1, -1), A)
    assert np.all(g >= -5.0) and np.all(g <= 0.0)
    alpha = np.exp(g)
    assert np.all(alpha >= math.exp(-5.0)) and np.all(alpha <= 1.0)


def test_gate_array_matches_scalar_and_indexing():
    # A is per (head, channel): check head/channel indexing of the array form.
    z = np.array([[[0.0, 1.0], [0.0, -1.0]]], dtype=np.float32)      # [T=1, H=2, dk=2]
    A = np.array([[0.0, math.log(2.0)], [math.log(3.0), 0.0]], dtype=np.float32)
    g = oracle.gate(z, A)
    for h in range(2):
        for c in range(2):
            assert g[0, h, c] == oracle.gate_scalar(float(A[h, c]), float(z[0, h, c]))
    assert g[0, 0, 0] == -2.5 and g[0, 1, 0] == -2.5


def test_bf16_inputs_convert_exactly():
    vals = torch.tensor([1.0, -2.5, 3.140625, 1e-3, 65280.0], dtype=torch.bfloat16)
    assert np.array_equal(oracle.to_f64(vals), vals.float().double().numpy())


# --------------------------------------------------------------- helpers for pins
def _rand_case(T, dk, dv, H=1, B=1, seed=0, s0=True, dtype=torch.float32, beta=None,
               z_inf=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, dk, generator=g)
    k = torch.randn(B, T, H, dk, generator=g)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(B, T, H, dv, generator=g)
    z = torch.randn(B, T, H, dk, generator=g) * 2
    b = torch.rand(B, T, H, generator=g) if beta is None else torch.full((B, T, H), beta)
    A = torch.randn(H, dk, generator=g) * 0.5
    S0 = torch.randn(B, H, dk, dv, generator=g) if s0 else None
    if z_inf is not None:
        z = torch.full_like(z, z_inf)
    return dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), z=z.to(dtype),
                beta=b.to(dtype), A=A, S0=S0)


def _alpha(z, A):
    return np.exp(oracle.gate(z, A))


# ------------------------------------------------------ hand-worked examples
def test_hand_example_no_decay():
    # z = -inf makes every gate 0 (alpha = 1).  Worked by hand with dyadic numbers:
    # t=1: k=(1,0) v=(2,3) b=1/2 q=(1,0), S0=0  -> S1=[[1,1.5],[0,0]], o1=(1,1.5)
    # t=2: k=(1/2,1/2) v=(1,-1) b=1/4 q=(0,1)   -> k^T S1 = (1/2, 3/4)
    #      S2 = S1 - 1/4 k (1/2,3/4) + 1/4 k (1,-1) = [[1.0625,1.28125],[0.0625,-0.21875]]
    #      o2 = S2^T q2 = (0.0625, -0.21875)
    q = torch.tensor([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    k = torch.tensor([[[[1.0, 0.0]], [[0.5, 0.5]]]])
    v = torch.tensor([[[[2.0, 3.0]], [[1.0, -1.0]]]])
    z = torch.full((1, 2, 1, 2), NEG_INF)
    b = torch.tensor([[[0.5], [0.25]]])
    A = torch.zeros(1, 2)
    o, S = oracle.recurrent(q, k, v, z, b, A)
    assert np.array_equal(o[:, 0, :], [[1.0, 1.5], [0.0625, -0.21875]])
    assert np.array_equal(S[0, 0], [[1.0625, 1.28125], [0.0625, -0.21875]])


def test_hand_example_channel_decay():
    # Channel 0 at the floor (z=+inf: alpha=e^-5), channel 1 undecayed (z=-inf: alpha=1).
    # S0=[[1,2],[3,4]], k=(1,0), b=1/2, v=(2,3), q=(1,1):
    #   D = Diag(e,1) S0 = [[e,2e],[3,4]],  k^T D = (e, 2e)
    #   S1 = D - 1/2 k (e,2e) + 1/2 k (2,3) = [[e/2+1, e+3/2],[3,4]]
    #   o1 = S1^T q = (4 + e/2, 11/2 + e)
    e = math.exp(-5.0)
    q = torch.tensor([[[[1.0, 1.0]]]])
    k = torch.tensor([[[[1.0, 0.0]]]])
    v = torch.tensor([[[[2.0, 3.0]]]])
    z = torch.tensor([[[[math.inf, NEG_INF]]]])
    b = torch.tensor([[[0.5]]])
    A = torch.zeros(1, 2)
    S0 = torch.tensor([[[[1.0, 2.0], [3.0, 4.0]]]])
    o, S = oracle.recurrent(q, k, v, z, b, A, S0=S0)
    np.testing.assert_allclose(o[0, 0], [4 + e / 2, 5.5 + e], rtol=1e-15)
    np.testing.assert_allclose(S[0, 0], [[e / 2 + 1, e + 1.5], [3.0, 4.0]], rtol=1e-15)


# ------------------------------------------------------------- closed form T<=3
def _closed_form_T3(q, k, v, beta, alpha, S0):
    """Hand-unrolled delta form for three tokens (no loop over t).

    u_t is the write each token makes; D_t = Diag(alpha_t).
      u1 = b1 (v1 - (D1 S0)^T k1)
      u2 = b2 (v2 - (D2 D1 S0)^T k2 - (k2^T D2 k1) u1)
      u3 = b3 (v3 - (D3 D2 D1 S0)^T k3 - (k3^T D3 D2 k1) u1 - (k3^T D3 k2) u2)
      S1 = D1 S0 + k1 u1^T
      S2 = D2 D1 S0 + (D2 k1) u1^T + k2 u2^T
      S3 = D3 D2 D1 S0 + (D3 D2 k1) u1^T + (D3 k2) u2^T + k3 u3^T
      o_t = S_t^T q_t
    """
    a1, a2, a3 = alpha
    q1, q2, q3 = q
    k1, k2, k3 = k
    v1, v2, v3 = v
    b1, b2, b3 = beta
    P1 = a1[:, None] * S0
    P2 = a2[:, None] * P1
    P3 = a3[:, None] * P2
    u1 = b1 * (v1 - P1.T @ k1)
    u2 = b2 * (v2 - P2.T @ k2 - (k2 @ (a2 * k1)) * u1)
    u3 = b3 * (v3 - P3.T @ k3 - (k3 @ (a3 * a2 * k1)) * u1 - (k3 @ (a3 * k2)) * u2)
    S1 = P1 + np.outer(k1, u1)
    S2 = P2 + np.outer(a2 * k1, u1) + np.outer(k2, u2)
    S3 = P3 + np.outer(a3 * a2 * k1, u1) + np.outer(a3 * k2, u2) + np.outer(k3, u3)
    return [S1.T @ q1, S2.T @ q2, S3.T @ q3], [S1, S2, S3]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_closed_form_three_tokens(seed, dtype):
    dk, dv = 5, 3                       # non-square so a transposed S cannot pass
    c = _rand_case(3, dk, dv, seed=seed, dtype=dtype)
    o, S = oracle.recurrent(c["q"], c["k"], c["v"], c["z"], c["beta"], c["A"], S0=c["S0"])
    q, k, v, z, b = (oracle.to_f64(c[n])[0, :, 0] for n in ("q", "k", "v", "z", "beta"))
    alpha = np.exp(oracle.gate(c["z"][0], c["A"]))[:, 0]
    o_cf, S_cf = _closed_form_T3(q, k, v, b, alpha, c["S0"].double().numpy()[0, 0])
    for t in range(3):
        np.testing.assert_allclose(o[t, 0], o_cf[t], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S[0, 0], S_cf[2], rtol=1e-12, atol=1e-13)
    # Shorter prefixes are the T=1 and T=2 closed forms.
    for T in (1, 2):
        sub = {n: (c[n][:, :T] if n in ("q", "k", "v", "z", "beta") else c[n]) for n in c}
        _, S_T = oracle.recurrent(sub["q"], sub["k"], sub["v"], sub["z"], sub["beta"],
                                  sub["A"], S0=sub["S0"])
        np.testing.assert_allclose(S_T[0, 0], S_cf[T - 1], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ invariants
def test_beta_zero_no_decay_keeps_state():
    c = _rand_case(17, 6, 4, H=2, seed=3, beta=0.0, z_inf=NEG_INF)
    o, S = oracle.recurrent(c["q"], c["k"], c["v"], c["z"], c["beta"], c["A"], S0=c["S0"])
    S0 = c["S0"].double().numpy()
    np.testing.assert_array_equal(S[0], S0[0])
    q = c["q"].double().numpy()[0]
    for h in range(2):
        np.testing.assert_allclose(o[:, h], q[:, h] @ S0[0, h], rtol=1e-13, atol=1e-14)


def test_beta_zero_pure_decay_closed_form():
    # beta = 0: S_t = Diag(exp(G_t)) S0 with G_t the running sum of gates.
    c = _rand_case(9, 4, 3, seed=4, beta=0.0)
    o, S = oracle.recurrent(c["q"], c["k"], c["v"], c["z"], c["beta"], c["A"], S0=c["S0"])
    g = oracle.gate(c["z"][0], c["A"])[:, 0]                  # [T, dk]
    G = np.cumsum(g, axis=0)
    S0 = c["S0"].double().numpy()[0, 0]
    q = c["q"].double().numpy()[0, :, 0]
    for t in range(9):
        St = np.exp(G[t])[:, None] * S0
        np.testing.assert_allclose(o[t, 0], St.T @ q[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S[0, 0], np.exp(G[-1])[:, None] * S0, rtol=1e-12)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_orthonormal_keys_recall_values(T):
    # alpha = 1, beta = 1, orthonormal keys: (I - k_j k_j^T) k_i = k_i for j != i,
    # so the final state returns v_i when queried with k_i.
    dk, dv = 8, 5
    rng = np.random.default_rng(T)
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    keys = Qm[:, :T].T.astype(np.float32)                      # rows orthonormal (in fp64)
    k = torch.from_numpy(keys).reshape(1, T, 1, dk)
    v = torch.randn(1, T, 1, dv, generator=torch.Generator().manual_seed(T))
    q = torch.randn(1, T, 1, dk, generator=torch.Generator().manual_seed(T + 100))
    z = torch.full((1, T, 1, dk), NEG_INF)
    b = torch.ones(1, T, 1)
    A = torch.zeros(1, dk)
    S0 = torch.randn(1, 1, dk, dv, generator=torch.Generator().manual_seed(7)) \
        if T == 8 else None                                    # T = dk: S0 is fully overwritten
    _, S = oracle.recurrent(q, k, v, z, b, A, S0=S0)
    kf = keys.astype(np.float64)
    # fp32 keys are orthonormal only to ~1e-7; the recall error is of that order.
    np.testing.assert_allclose(S[0, 0].T @ kf.T, v.double().numpy()[0, :, 0].T, atol=2e-6)


def test_contraction_of_state_differences():
    # With |k| = 1 and beta in [0, 1], (I - b k k^T) Diag(alpha) has spectral norm <= 1,
    # so two runs that differ only in S0 never drift apart.
    c = _rand_case(40, 8, 6, seed=5)
    S0b = c["S0"] + torch.randn(c["S0"].shape, generator=torch.Generator().manual_seed(9))
    _, Sa = oracle.recurrent(c["q"], c["k"], c["v"], c["z"], c["beta"], c["A"], S0=c["S0"])
    _, Sb = oracle.recurrent(c["q"], c["k"], c["v"], c["z"], c["beta"], c["A"], S0=S0b)
    d0 = np.linalg.norm((S0b - c["S0"]).double().numpy())
    assert np.linalg.norm(Sb - Sa) <= d0 * (1 + 1e-12)


# --------------------------------------------------- structure: segments, varlen
def test_segment_split_equals_whole():
    c = _rand_case(50, 6, 5, H=3, seed=6)
    args = [c[n] for n in ("q", "k", "v", "z", "beta")]
    o, S = oracle.recurrent(*args, c["A"], S0=c["S0"])
    first = [x[:, :23] for x in args]
    second = [x[:, 23:] for x in args]
    o1, S1 = oracle.recurrent(*first, c["A"], S0=c["S0"])
    o2, S2 = oracle.recurrent(*second, c["A"], S0=torch.from_numpy(S1).float())
    # S1 is rounded to fp32 when carried over; allow for that rounding.
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(S2, S, rtol=1e-5, atol=1e-6)


def test_state_dependence_is_affine():
    # run(S0, x) = M S0 + run(0, x) for a linear M (the segment pair of the
    # context-parallel decomposition: each segment is a pair of an accumulated
    # transformation and a state built from zero, per the page "How Kimi K3 is built: 2.8 trillion para...").
    c = _rand_case(30, 5, 4, seed=8)
    args = [c[n] for n in ("q", "k", "v", "z", "beta")]
    Sa = c["S0"]
    Sb = torch.randn(Sa.shape, generator=torch.Generator().manual_seed(11))
    _, Rz = oracle.recurrent(*args, c["A"], S0=None)
    _, Ra = oracle.recurrent(*args, c["A"], S0=Sa)
    _, Rb = oracle.recurrent(*args, c["A"], S0=Sb)
    _, Rab = oracle.recurrent(*args, c["A"], S0=Sa + Sb)
    np.testing.assert_allclose(Rab - Rz, (Ra - Rz) + (Rb - Rz), rtol=1e-10, atol=1e-12)


def test_packed_equals_separate_runs():
    lens = [5, 1, 17, 9]
    dk, dv, H = 6, 4, 2
    g = torch.Generator().manual_seed(12)
    Tt = sum(lens)
    q = torch.randn(Tt, H, dk, generator=g)
    k = torch.randn(Tt, H, dk, generator=g)
    v = torch.randn(Tt, H, dv, generator=g)
    z = torch.randn(Tt, H, dk, generator=g)
    b = torch.rand(Tt, H, generator=g)
    A = torch.randn(H, dk, generator=g)
    S0 = torch.randn(len(lens), H, dk, dv, generator=g)
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.recurrent(q, k, v, z, b, A, S0=S0, cu_seqlens=cu)
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        on, Sn = oracle.recurrent(q[sl][None], k[sl][None], v[sl][None], z[sl][None],
                                  b[sl][None], A, S0=S0[n:n + 1])
        np.testing.assert_array_equal(o[sl], on[:, :, :])
        np.testing.assert_array_equal(S[n], Sn[0])


def test_selected_pairs_match_full_run():
    c = _rand_case(12, 4, 3, H=3, B=2, seed=13)
    args = [c[n] for n in ("q", "k", "v", "z", "beta")]
    o, S = oracle.recurrent(*args, c["A"], S0=c["S0"])
    pairs = [(1, 2), (0, 1)]
    ol, Sl = oracle.recurrent(*args, c["A"], S0=c["S0"], pairs=pairs)
    for i, (n, h) in enumerate(pairs):
        np.testing.assert_array_equal(ol[i], o.reshape(2, 12, 3, 3)[n, :, h])
        np.testing.assert_array_equal(Sl[i], S[n, h])


# ------------------------------------------------------- chunked form agreement
@pytest.mark.parametrize("C", [1, 2, 16, 64])
def test_chunked_form_matches_recurrence(C):
    lens = [70, 1, 64, 33]            # a ragged tail, a one-token sequence, an exact chunk
    dk, dv, H = 16, 8, 2
    g = torch.Generator().manual_seed(20 + C)
    Tt = sum(lens)
    q = torch.randn(Tt, H, dk, generator=g)
    q = q / q.norm(dim=-1, keepdim=True)
    k = torch.randn(Tt, H, dk, generator=g)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(Tt, H, dv, generator=g)
    z = torch.randn(Tt, H, dk, generator=g) * 3
    z[:, :, : dk // 2] = 8.0          # half the channels at the -5 floor
    b = torch.sigmoid(torch.randn(Tt, H, generator=g))
    A = torch.randn(H, dk, generator=g) * 0.5
    S0 = torch.randn(len(lens), H, dk, dv, generator=g) * 0.02
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.recurrent(q, k, v, z, b, A, S0=S0, cu_seqlens=cu)
    oc, Sc = oracle.chunked(q, k, v, z, b, A, S0=S0, cu_seqlens=cu, C=C)
    scale_o = np.abs(o).max()
    scale_s = np.abs(S).max()
    assert np.abs(oc - o).max() <= 1e-12 * scale_o
    assert np.abs(Sc - S).max() <= 1e-12 * scale_s
