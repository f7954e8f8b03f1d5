"""GPU parity of kda_chunk_prefill against the fp64 oracle (through the C ABI).

Small cases run the whole oracle.  The full-size workloads also compare every
(sequence, head) pair with the oracle, element by element, in batches of heads.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import TOL, assert_parity, cuda, rel_err, report

pytestmark = pytest.mark.gpu


def run_gpu(x, chunk, output_final_state=True):
    xc = cuda(x)
    cu = xc.get("cu_seqlens")
    o, S = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                             initial_state=xc["S0"], cu_seqlens=cu, chunk=chunk,
                             output_final_state=output_final_state)
    torch.cuda.synchronize()
    return o, S


def run_oracle(x, pairs=None):
    cu = x.get("cu_seqlens")
    q, k, v, z, b = (x[n] for n in ("q", "k", "v", "z", "beta"))
    if cu is not None:
        q, k, v, z, b = (t[0] for t in (q, k, v, z, b))
    return oracle.recurrent(q, k, v, z, b, x["A"], S0=x["S0"], cu_seqlens=cu, pairs=pairs)


def check_full(x, chunk, dtype, what, o_tol=None, s_tol=None):
    o, S = run_gpu(x, chunk)
    ro, rS = run_oracle(x)
    eo = assert_parity(o.reshape(ro.shape), ro, dtype, f"{what} o", tol=o_tol)
    es = assert_parity(S, rS, dtype, f"{what} final state", tol=s_tol)
    return eo, es


def test_tiny_fp32_workload():
    w = WORKLOADS[0]
    x = make_inputs(w)
    assert kda.prefill_path(w.dk, w.dv, w.chunk, w.dtype) == "recurrent"
    check_full(x, w.chunk, w.dtype, "workload 0")


@pytest.mark.parametrize("chunk", [16, 64])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(128, 128), (32, 64), (20, 12), (64, 128), (17, 13), (128, 65)])
def test_fixed_length_shapes(dtype, dk, dv, chunk):
    w = replace(WORKLOADS[1], dk=dk, dv=dv, dtype=dtype, H=3, seed=dk + dv + chunk,
                initial_state=True)
    x = make_inputs(w, B=2, T=150)
    check_full(x, chunk, dtype, f"B=2 T=150 dk={dk} dv={dv} C={chunk}")


@pytest.mark.parametrize("lengths", [[1, 64, 65, 130, 0, 7], [200], [0, 0, 3]])
def test_packed_sequences(lengths):
    w = replace(WORKLOADS[4], H=2, seed=len(lengths) + sum(lengths))
    x = make_inputs(w, lengths=lengths)
    check_full(x, 64, torch.bfloat16, f"packed {lengths}")


@pytest.mark.parametrize("dtype,d", [(torch.float32, 128), (torch.bfloat16, 48)])
def test_packed_sequences_recurrent(dtype, d):
    # The fp32 recurrence on a packed batch (empty, one-token and ragged sequences;
    # runs of 8 tokens and 16-token tiles cut at every sequence start).
    lengths = [1, 64, 65, 130, 0, 7, 23]
    w = replace(WORKLOADS[4], H=2, dk=d, dv=d, dtype=dtype, seed=90 + d)
    x = make_inputs(w, lengths=lengths)
    assert kda.prefill_path(d, d, 64, dtype) == "recurrent"
    check_full(x, 64, dtype, f"packed {lengths} {dtype} d={d}")


def test_no_initial_state_and_no_final_state():
    w = replace(WORKLOADS[1], H=2, seed=77)
    x = make_inputs(w, B=1, T=90)
    assert x["S0"] is None
    o, S = run_gpu(x, 64, output_final_state=False)
    assert S is None
    ro, _ = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "o without states")


def test_zero_tokens_passes_state_through():
    w = replace(WORKLOADS[1], H=2, seed=5, initial_state=True)
    x = make_inputs(w, B=1, T=0)
    o, S = run_gpu(x, 64)
    assert o.numel() == 0
    assert torch.equal(S.cpu(), x["S0"])


def test_resume_from_final_state():
    # prefill(T1) -> S; prefill(T2, S0 = S) equals prefill(T1 + T2)
    w = replace(WORKLOADS[1], H=2, seed=8, initial_state=True)
    x = make_inputs(w, B=1, T=300)
    first = {n: (x[n][:, :130].contiguous() if n in ("q", "k", "v", "z", "beta") else x[n])
             for n in x}
    second = {n: (x[n][:, 130:].contiguous() if n in ("q", "k", "v", "z", "beta") else x[n])
              for n in x}
    o1, S1 = run_gpu(first, 64)
    second["S0"] = S1.cpu()
    o2, S2 = run_gpu(second, 64)
    ro, rS = run_oracle(x)
    assert_parity(torch.cat([o1, o2], 1).reshape(ro.shape), ro, torch.bfloat16, "resumed o")
    assert_parity(S2, rS, torch.bfloat16, "resumed state")


def test_output_buffer_canaries():
    # Writes stay inside o and the state: guard regions around them keep their pattern.
    w = replace(WORKLOADS[1], H=2, seed=9, initial_state=True)
    x = cuda(make_inputs(w, B=1, T=77))
    pad = 4096
    o_buf = torch.full((pad * 2 + 77 * 2 * 128,), 7.0, device="cuda", dtype=torch.bfloat16)
    s_buf = torch.full((pad * 2 + 2 * 128 * 128,), 7.0, device="cuda")
    o = o_buf[pad:pad + 77 * 2 * 128].view(1, 77, 2, 128)
    S = s_buf[pad:pad + 2 * 128 * 128].view(1, 2, 128, 128)
    kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], initial_state=x["S0"],
                      chunk=64, out=o, final_state=S)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(s_buf[:pad] == 7.0) and torch.all(s_buf[-pad:] == 7.0)


# ----------------------------------------------------------- tensor-core path
def test_tensor_core_path_is_selected():
    assert kda.prefill_path(128, 128, 64, torch.bfloat16) == "chunked_tc"
    assert kda.prefill_path(128, 128, 16, torch.bfloat16) == "chunk16_tc"
    assert kda.prefill_path(128, 128, 64, torch.float32) == "recurrent"


def _run_with_status(x, chunk=64):
    """Runs prefill with a caller workspace and returns (o, S, device status word)."""
    xc = cuda(x)
    q = xc["q"]
    B, T, H, dk = q.shape
    cu = xc.get("cu_seqlens")
    n = B if cu is None else cu.numel() - 1
    need = kda.workspace_size(n, B, T, H, dk, xc["v"].shape[-1], chunk, q.dtype)
    ws = torch.full((max(need, 256),), 0xAB, dtype=torch.uint8, device="cuda")
    o, S = kda.chunk_prefill(q, xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                             initial_state=xc["S0"], cu_seqlens=cu, chunk=chunk, workspace=ws)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item()) if need > 0 else 0
    return o, S, status


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 1000])
def test_tensor_core_lengths(T):
    w = replace(WORKLOADS[2], H=2, seed=1000 + T)
    x = make_inputs(w, B=1, T=T)
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"TC T={T} o")
    assert_parity(S, rS, torch.bfloat16, f"TC T={T} state")


def test_tensor_core_zero_and_pure_decay_inputs():
    # beta = 0 everywhere: the state only decays, o_t = (Diag(e^{G_t}) S0)^T q_t.  The gate
    # inputs are shifted down so that 130 tokens of decay stay inside the fp32 range.
    w = replace(WORKLOADS[1], H=1, seed=55, initial_state=True)
    x = make_inputs(w, B=1, T=130)
    x["beta"] = torch.zeros_like(x["beta"])
    x["z"] = (x["z"].float() * 0.5 - 3.0).to(torch.bfloat16)
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "beta=0 o")
    assert_parity(S, rS, torch.bfloat16, "beta=0 state")


def _full_check(x, what, heads_per_batch, chunk=64):
    """Compares every (sequence, head) of one GPU call with the oracle, element by element.

    The oracle runs on batches of heads (every sequence of those heads at once), so that
    its fp64 output stays a few GB.  The bound is applied to the whole o and the whole final
    state (max |gpu - oracle| over max |oracle| of the tensor); the worst single (sequence,
    head) pair, measured against its own maximum, is reported beside it.
    """
    o, S, status = _run_with_status(x, chunk)
    assert status == 0
    q = x["q"]
    B, T, H = q.shape[:3]
    cu = x.get("cu_seqlens")
    cuv = (np.arange(B + 1, dtype=np.int64) * T if cu is None
           else cu.cpu().numpy().astype(np.int64))
    n_seqs = len(cuv) - 1
    dv = o.shape[-1]
    o_flat = o.reshape(-1, H, dv)
    nonempty = np.nonzero(np.diff(cuv) > 0)[0]
    d_o = r_o = d_s = r_s = 0.0
    worst_o = worst_s = 0.0
    for h0 in range(0, H, heads_per_batch):
        hs = torch.arange(h0, min(H, h0 + heads_per_batch), device=q.device)
        sub = {n: x[n].index_select(-2 if n != "beta" else -1, hs).cpu()
               for n in ("q", "k", "v", "z", "beta")}
        sub["A"] = x["A"][hs].cpu()
        sub["S0"] = None if x["S0"] is None else x["S0"][:, hs].cpu()
        if cu is not None:
            sub["cu_seqlens"] = cu.cpu()
        ro, rS = run_oracle(sub)                           # [T_total, hb, dv], [N, hb, dk, dv]
        go = o_flat.index_select(1, hs).cpu().double().numpy()
        assert np.all(np.isfinite(go)), f"{what}: non-finite o"
        dtok = np.abs(go - ro).max(axis=-1)                # [T_total, hb]
        rtok = np.abs(ro).max(axis=-1)
        del go, ro
        gS = S.index_select(1, hs).cpu().double().numpy()
        assert np.all(np.isfinite(gS)), f"{what}: non-finite state"
        dpair_s = np.abs(gS - rS).reshape(n_seqs, len(hs), -1).max(-1)
        rpair_s = np.abs(rS).reshape(n_seqs, len(hs), -1).max(-1)
        d_s, r_s = max(d_s, dpair_s.max()), max(r_s, rpair_s.max())
        worst_s = max(worst_s, float((dpair_s / np.maximum(rpair_s, 1e-30)).max()))
        if len(nonempty):
            dpair_o = np.maximum.reduceat(dtok, cuv[nonempty], axis=0)  # [seqs, hb]
            rpair_o = np.maximum.reduceat(rtok, cuv[nonempty], axis=0)
            d_o, r_o = max(d_o, dpair_o.max()), max(r_o, rpair_o.max())
            worst_o = max(worst_o, float((dpair_o / np.maximum(rpair_o, 1e-30)).max()))
    tol = TOL[torch.bfloat16]
    eo, es = d_o / r_o, d_s / r_s
    report(f"{what} o (all {n_seqs}x{H} pairs)", eo, tol, f" worst_pair={worst_o:.3e}")
    report(f"{what} final state (all {n_seqs}x{H} pairs)", es, tol, f" worst_pair={worst_s:.3e}")
    assert eo <= tol, f"{what} o: {eo:.3e} > {tol:.1e}"
    assert es <= tol, f"{what} final state: {es:.3e} > {tol:.1e}"
    return eo, es


def test_full_workload_prefill_b2_h8_t4096():
    x = make_inputs(WORKLOADS[1], device="cuda")
    _full_check(x, "workload 1", heads_per_batch=8)


def test_full_workload_long_prefill_h32_t65536():
    x = make_inputs(WORKLOADS[2], device="cuda")
    _full_check(x, "workload 2", heads_per_batch=16)


def test_full_workload_packed_64_sequences():
    x = make_inputs(WORKLOADS[4], device="cuda")
    _full_check(x, "workload 4", heads_per_batch=2)
