"""GPU parity of kda_chunk_prefill against the fp64 oracle (through the C ABI).

Small cases run the whole oracle; the full-size workloads compare a seeded
sample of (sequence, head) pairs, each of which the oracle computes on its own.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import TOL, assert_parity, cuda, rel_err

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
@pytest.mark.parametrize("dk,dv", [(128, 128), (32, 64), (20, 12), (64, 128)])
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
    assert kda.prefill_path(128, 128, 16, torch.bfloat16) == "recurrent"
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


def _sampled_check(x, pairs, what):
    """Compares the GPU result with the oracle on the given (sequence, head) pairs only."""
    xc = {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    o, S, status = _run_with_status(xc)
    assert status == 0
    heads = sorted({h for _, h in pairs})
    hidx = {h: i for i, h in enumerate(heads)}
    hs = torch.tensor(heads, device=xc["q"].device)
    sub = {n: xc[n].index_select(-2 if n != "beta" else -1, hs).cpu()
           for n in ("q", "k", "v", "z", "beta")}
    sub["A"] = xc["A"][hs].cpu()
    sub["S0"] = None if xc["S0"] is None else xc["S0"][:, hs].cpu()
    cu = x.get("cu_seqlens")
    if cu is not None:
        sub["cu_seqlens"] = cu.cpu()
    ro, rS = run_oracle(sub, pairs=[(n, hidx[h]) for n, h in pairs])
    ocpu = o.index_select(-2, hs).cpu()
    Scpu = S.cpu()
    B, T = xc["q"].shape[:2]
    cuv = np.arange(B + 1) * T if cu is None else cu.cpu().numpy()
    flat = ocpu.reshape(-1, len(heads), ocpu.shape[-1])
    errs = []
    for i, (n, h) in enumerate(pairs):
        got = flat[cuv[n]:cuv[n + 1], hidx[h]]
        errs.append(assert_parity(got, ro[i], torch.bfloat16, f"{what} o pair {(n, h)}"))
        assert_parity(Scpu[n, h], rS[i], torch.bfloat16, f"{what} state pair {(n, h)}")
    return max(errs)


def test_full_workload_prefill_b2_h8_t4096():
    w = WORKLOADS[1]
    x = make_inputs(w, device="cuda")
    pairs = [(b, h) for b in range(2) for h in range(8)]
    _sampled_check(x, pairs, "workload 1")


def test_full_workload_long_prefill_h32_t65536():
    w = WORKLOADS[2]
    x = make_inputs(w, device="cuda")
    _sampled_check(x, [(0, 0), (0, 13), (0, 31)], "workload 2")


def test_full_workload_packed_64_sequences():
    w = WORKLOADS[4]
    x = make_inputs(w, device="cuda")
    lens = x["lengths"]
    order = torch.argsort(lens)
    pairs = [(int(order[-1]), 0), (int(order[0]), 5), (int(order[32]), 15), (7, 9)]
    _sampled_check(x, pairs, "workload 4")
