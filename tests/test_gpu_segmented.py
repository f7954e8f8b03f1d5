"""GPU parity of the segment-parallel prefill (kda_chunk_prefill_segmented) against the
fp64 oracle, through the C ABI.

Each sequence is split into segments whose (transition, state-from-zero) pairs are formed
in parallel, scanned into the segments' start states and then finished from them.  The
result must match the recurrence to the bf16 bound for every segment count, including
segment counts that do not divide the chunk count, ragged last chunks, narrower heads and
the case with no initial state.
"""
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda

pytestmark = pytest.mark.gpu


def _oracle(x):
    return oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])


def _run_segmented(xc, G):
    B, T, H, dk = xc["q"].shape
    need = kda.segmented_workspace_size(B, T, H, dk, xc["v"].shape[-1], G)
    ws = torch.full((need,), 0xCD, dtype=torch.uint8, device="cuda")
    o, S = kda.chunk_prefill_segmented(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                                       G, initial_state=xc["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "a bounded wait gave up"
    return o, S


@pytest.mark.parametrize("T,G", [(1000, 2), (1000, 3), (2000, 5), (4096, 7), (130, 2), (777, 13)])
def test_segmented_matches_oracle(T, G):
    w = replace(WORKLOADS[2], H=2, seed=600 + T + G)
    x = make_inputs(w, B=2, T=T)
    o, S = _run_segmented(cuda(x), G)
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"segmented T={T} G={G} o")
    assert_parity(S, rS, torch.bfloat16, f"segmented T={T} G={G} state")


def test_segmented_without_initial_state():
    w = replace(WORKLOADS[1], H=3, seed=611)
    x = make_inputs(w, B=1, T=1500)
    assert x["S0"] is None
    o, S = _run_segmented(cuda(x), 4)
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "segmented, no S0, o")
    assert_parity(S, rS, torch.bfloat16, "segmented, no S0, state")


@pytest.mark.parametrize("dk,dv", [(64, 64), (48, 32), (128, 64), (32, 128)])
def test_segmented_narrower_heads(dk, dv):
    w = replace(WORKLOADS[2], H=2, dk=dk, dv=dv, seed=620 + dk + dv)
    x = make_inputs(w, B=1, T=1300)
    o, S = _run_segmented(cuda(x), 3)
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"segmented dk={dk} dv={dv} o")
    assert_parity(S, rS, torch.bfloat16, f"segmented dk={dk} dv={dv} state")


def test_one_segment_is_the_plain_pass():
    w = replace(WORKLOADS[2], H=2, seed=630)
    x = cuda(make_inputs(w, B=1, T=900))
    o1, S1 = _run_segmented(x, 1)
    B, T, H, dk = x["q"].shape
    ws = torch.empty(kda.segmented_workspace_size(B, T, H, dk, 128, 1), dtype=torch.uint8,
                     device="cuda")
    assert ws.numel() == kda.workspace_size(B, B, T, H, dk, 128, 64, torch.bfloat16)
    o0, S0 = kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                               initial_state=x["S0"], workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(S0, S1)


def test_segmented_checkpoints_through_kda_chunk_prefill():
    # H=1 makes kda_chunk_prefill segment on its own; checkpoints come from the final pass.
    w = replace(WORKLOADS[2], H=1, seed=640)
    T = 4096
    x = make_inputs(w, B=1, T=T)
    assert kda.auto_segments(1, T, 1, 128, 128) > 1
    xc = cuda(x)
    every = 512
    ck = torch.full((1, 1, T // every, 128, 128), float("nan"), device="cuda")
    o, S = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                             initial_state=xc["S0"], checkpoints=ck, checkpoint_every=every)
    torch.cuda.synchronize()
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "auto-segmented o")
    assert_parity(S, rS, torch.bfloat16, "auto-segmented state")
    for i in (0, 3, T // every - 1):
        n = (i + 1) * every
        part = {k_: (v_[:, :n].contiguous() if k_ in ("q", "k", "v", "z", "beta") else v_)
                for k_, v_ in x.items()}
        _, rck = _oracle(part)
        assert_parity(ck[0, 0, i], rck[0, 0], torch.bfloat16, f"auto-segmented checkpoint {i}")


def test_low_chain_long_prefill_all_heads():
    # B=1, H=8, T=65536: 32 column-tile chains on 152 SMs; every head against the oracle.
    w = replace(WORKLOADS[2], H=8, seed=650)
    x = make_inputs(w, device="cuda", B=1, T=65536)
    G = kda.auto_segments(1, 65536, 8, 128, 128)
    assert G > 1
    o, S = _run_segmented(x, G)
    ro, rS = _oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"B=1 H=8 T=65536 G={G} o (all heads)")
    assert_parity(S, rS, torch.bfloat16, f"B=1 H=8 T=65536 G={G} state (all heads)")
