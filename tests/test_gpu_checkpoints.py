"""kda_chunk_prefill_checkpoints: intermediate states against the fp64 oracle.

Checkpoint i of a sequence is the state after (i + 1) * every of its tokens; the
oracle gives it as the final state of that prefix.  Continuing from a
checkpoint must reproduce the rest of the uninterrupted run (the copy-before-
continue contract of the prefix cache).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import TOL, assert_parity, cuda

pytestmark = pytest.mark.gpu


def _prefix_state(x, n, p, cu=None):
    """Oracle state of sequence n after its first p tokens."""
    names = ("q", "k", "v", "z", "beta")
    if cu is None:
        sub = [x[nm][n:n + 1, :p] for nm in names]
        S0 = None if x["S0"] is None else x["S0"][n:n + 1]
        _, S = oracle.recurrent(*sub, x["A"], S0=S0)
    else:
        b = int(cu[n])
        sub = [x[nm][:, b:b + p] for nm in names]
        S0 = None if x["S0"] is None else x["S0"][n:n + 1]
        _, S = oracle.recurrent(*sub, x["A"], S0=S0)
    return S[0]


def _run(x, chunk, every, slots):
    xc = cuda(x)
    cu = xc.get("cu_seqlens")
    B, T, H, dk = xc["q"].shape
    n = B if cu is None else cu.numel() - 1
    ck = torch.full((n, H, slots, dk, xc["v"].shape[-1]), float("nan"), device="cuda")
    o, S = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                             initial_state=xc["S0"], cu_seqlens=cu, chunk=chunk,
                             checkpoints=ck, checkpoint_every=every)
    torch.cuda.synchronize()
    return o, S, ck.cpu()


@pytest.mark.parametrize("path", ["tensor_core", "recurrent_bf16", "recurrent_fp32"])
def test_checkpoints_fixed_length(path):
    if path == "tensor_core":
        w = replace(WORKLOADS[2], H=2, seed=71)
        chunk, every, dtype = 64, 128, torch.bfloat16
    elif path == "recurrent_bf16":
        w = replace(WORKLOADS[1], H=2, dk=64, dv=48, seed=72, initial_state=True)
        chunk, every, dtype = 16, 32, torch.bfloat16
    else:
        w = replace(WORKLOADS[0], H=2, dk=32, dv=32, seed=73, initial_state=True)
        chunk, every, dtype = 16, 48, torch.float32
    x = make_inputs(w, B=2, T=300)
    slots = 3
    o, S, ck = _run(x, chunk, every, slots)
    for n in range(2):
        for i in range(slots):
            p = (i + 1) * every
            if p <= 300:
                ref = _prefix_state(x, n, p)
                assert_parity(ck[n, :, i], ref, dtype, f"{path} seq {n} checkpoint {i}")
            else:
                assert torch.isnan(ck[n, :, i]).all(), "slot past the sequence was written"


def test_checkpoints_packed_and_resume():
    lengths = [700, 64, 129, 1]
    w = replace(WORKLOADS[4], H=2, seed=74)
    x = make_inputs(w, lengths=lengths)
    every, slots = 128, 4
    o, S, ck = _run(x, 64, every, slots)
    cu = x["cu_seqlens"]
    for n, L in enumerate(lengths):
        for i in range(slots):
            p = (i + 1) * every
            if p <= L:
                ref = _prefix_state(x, n, p, cu=cu)
                assert_parity(ck[n, :, i], ref, torch.bfloat16, f"packed seq {n} checkpoint {i}")
            else:
                assert torch.isnan(ck[n, :, i]).all()
    # Continue sequence 0 from its checkpoint at 384 tokens: the rest of the run matches.
    b, p = int(cu[0]), 3 * every
    rest = {nm: x[nm][:, b + p:b + lengths[0]].contiguous() for nm in ("q", "k", "v", "z", "beta")}
    rest["A"] = x["A"]
    rest["S0"] = ck[0:1, :, 2].clone()
    rc = cuda(rest)
    o2, S2 = kda.chunk_prefill(rc["q"], rc["k"], rc["v"], rc["z"], rc["beta"], rc["A"],
                               initial_state=rc["S0"], chunk=64)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(*[x[nm][:, b:b + lengths[0]] for nm in ("q", "k", "v", "z", "beta")],
                              x["A"], S0=x["S0"][0:1])
    assert_parity(o2.reshape(-1, 2, 128), ro[p:], torch.bfloat16, "resumed outputs")
    assert_parity(S2, rS, torch.bfloat16, "resumed final state")
    assert_parity(S[0], rS[0], torch.bfloat16, "uninterrupted final state")


def test_checkpoint_argument_checks():
    w = replace(WORKLOADS[2], H=1, seed=75)
    x = cuda(make_inputs(w, B=1, T=128))
    ck = torch.zeros(1, 1, 2, 128, 128, device="cuda")
    with pytest.raises(kda.KDAError, match="multiple of the chunk"):
        kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], chunk=64,
                          checkpoints=ck, checkpoint_every=96)
    with pytest.raises(kda.KDAError, match="multiple of the chunk"):
        kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], chunk=64,
                          checkpoints=ck, checkpoint_every=0)
