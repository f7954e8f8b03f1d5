"""GPU parity of the 16-token tensor-core prefill (chunk = 16, bf16) against the fp64
oracle, through the C ABI.

The state is handed from chunk to chunk every 16 tokens inside one fused kernel per
(sequence, head).  Cases: lengths around the chunk size, packed batches with empty and
one-token sequences, narrower heads, no initial state, checkpoints every 16 tokens, guard
regions around the outputs, and the full-size prefill, long-context and packed workloads
compared with the oracle on every (sequence, head) pair.
"""
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda
from tests.test_gpu_prefill import _full_check, _run_with_status, run_oracle

pytestmark = pytest.mark.gpu


def test_chunk16_path_is_selected():
    assert kda.prefill_path(128, 128, 16, torch.bfloat16) == "chunk16_tc"
    assert kda.prefill_path(16, 16, 16, torch.bfloat16) == "chunk16_tc"
    assert kda.prefill_path(128, 128, 16, torch.float32) == "recurrent"
    assert kda.workspace_size(1, 1, 4096, 8, 128, 128, 16, torch.bfloat16) == 1024


@pytest.mark.parametrize("T", [1, 15, 16, 17, 100, 1000])
def test_chunk16_lengths(T):
    w = replace(WORKLOADS[2], H=2, seed=700 + T)
    x = make_inputs(w, B=1, T=T)
    o, S, status = _run_with_status(x, chunk=16)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"chunk16 T={T} o")
    assert_parity(S, rS, torch.bfloat16, f"chunk16 T={T} state")


@pytest.mark.parametrize("lengths", [[1, 16, 17, 0, 33, 200], [0, 0, 5], [64]])
def test_chunk16_packed(lengths):
    w = replace(WORKLOADS[4], H=2, seed=710 + sum(lengths))
    x = make_inputs(w, lengths=lengths)
    o, S, status = _run_with_status(x, chunk=16)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"chunk16 packed {lengths} o")
    assert_parity(S, rS, torch.bfloat16, f"chunk16 packed {lengths} state")


@pytest.mark.parametrize("dk,dv", [(16, 16), (48, 32), (128, 64), (64, 128), (32, 112)])
def test_chunk16_narrower_heads(dk, dv):
    w = replace(WORKLOADS[2], H=2, dk=dk, dv=dv, seed=720 + dk + dv)
    x = make_inputs(w, B=2, T=150)
    o, S, status = _run_with_status(x, chunk=16)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"chunk16 dk={dk} dv={dv} o")
    assert_parity(S, rS, torch.bfloat16, f"chunk16 dk={dk} dv={dv} state")


def test_chunk16_without_states_and_canaries():
    w = replace(WORKLOADS[1], H=2, seed=730)
    x = cuda(make_inputs(w, B=1, T=77))
    assert x["S0"] is None
    pad = 4096
    o_buf = torch.full((pad * 2 + 77 * 2 * 128,), 7.0, device="cuda", dtype=torch.bfloat16)
    o = o_buf[pad:pad + 77 * 2 * 128].view(1, 77, 2, 128)
    kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], chunk=16, out=o,
                      output_final_state=False)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    ro, _ = run_oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "chunk16 o without states")


def test_chunk16_checkpoints_every_16_tokens():
    w = replace(WORKLOADS[2], H=2, seed=740)
    T, every = 100, 16
    x = make_inputs(w, B=1, T=T)
    xc = cuda(x)
    slots = T // every
    ck = torch.full((1, 2, slots, 128, 128), float("nan"), device="cuda")
    kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                      initial_state=xc["S0"], chunk=16, checkpoints=ck, checkpoint_every=every)
    torch.cuda.synchronize()
    for i in range(slots):
        n = (i + 1) * every
        part = {k_: (v_[:, :n].contiguous() if k_ in ("q", "k", "v", "z", "beta") else v_)
                for k_, v_ in x.items()}
        _, rS = oracle.recurrent(part["q"], part["k"], part["v"], part["z"], part["beta"],
                                 part["A"], S0=part["S0"])
        assert_parity(ck[0, :, i], rS[0], torch.bfloat16, f"chunk16 checkpoint {i}")


def test_chunk16_agrees_with_chunk64():
    w = replace(WORKLOADS[2], H=3, seed=750)
    x = cuda(make_inputs(w, B=2, T=500))
    o16, S16, _ = _run_with_status(x, chunk=16)
    o64, S64, _ = _run_with_status(x, chunk=64)
    scale_o = o64.float().abs().max()
    assert (o16.float() - o64.float()).abs().max() <= 2e-2 * scale_o
    assert (S16 - S64).abs().max() <= 2e-2 * S64.abs().max()


def test_chunk16_full_workload_prefill_b2_h8_t4096():
    _full_check(make_inputs(WORKLOADS[1], device="cuda"), "workload 1 chunk 16", 8, chunk=16)


def test_chunk16_full_workload_long_prefill_h32_t65536():
    _full_check(make_inputs(WORKLOADS[2], device="cuda"), "workload 2 chunk 16", 16, chunk=16)


def test_chunk16_full_workload_packed_64_sequences():
    _full_check(make_inputs(WORKLOADS[4], device="cuda"), "workload 4 chunk 16", 2, chunk=16)
