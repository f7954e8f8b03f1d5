"""The tensor-core prefill path on heads narrower than 128 (bf16, chunk 64).

d_k a multiple of 16 and d_v a multiple of 32, both at most 128: the kernels
work on 128-wide tiles whose extra channels arrive as zeros, and the state
pass runs d_v / 32 column tiles.  Parity against the fp64 oracle, with canary
regions around every output so that nothing past d_k or d_v is written.
"""
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda

pytestmark = pytest.mark.gpu

SHAPES = [(64, 64), (16, 32), (32, 128), (128, 64), (96, 96), (48, 32)]
NAMES = ("q", "k", "v", "z", "beta")
CANARY = 7.0


def _oracle(x):
    cu = x.get("cu_seqlens")
    q, k, v, z, b = (x[n] for n in NAMES)
    if cu is not None:
        q, k, v, z, b = (t[0] for t in (q, k, v, z, b))
    return oracle.recurrent(q, k, v, z, b, x["A"], S0=x["S0"], cu_seqlens=cu)


def _guarded(shape, dtype):
    """A view of `shape` inside a buffer whose 32 elements on each side hold CANARY."""
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 64,), CANARY, dtype=dtype, device="cuda")
    return buf, buf[32:32 + n].view(*shape)


def _canaries_intact(buf, what):
    assert bool((buf[:32] == CANARY).all()) and bool((buf[-32:] == CANARY).all()), \
        f"{what}: written outside its extent"


@pytest.mark.parametrize("dk,dv", SHAPES)
def test_fixed_length(dk, dv):
    assert kda.prefill_path(dk, dv, 64, torch.bfloat16) == "chunked_tc"
    B, T, H = 2, 200, 3
    w = replace(WORKLOADS[1], H=H, dk=dk, dv=dv, seed=7 * dk + dv, initial_state=True)
    x = make_inputs(w, B=B, T=T)
    xc = cuda(x)
    ob, o = _guarded((B, T, H, dv), torch.bfloat16)
    sb, S = _guarded((B, H, dk, dv), torch.float32)
    kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                      initial_state=xc["S0"], chunk=64, out=o, final_state=S)
    torch.cuda.synchronize()
    _canaries_intact(ob, "o")
    _canaries_intact(sb, "final state")
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, f"dk={dk} dv={dv} o")
    assert_parity(S, rS, torch.bfloat16, f"dk={dk} dv={dv} final state")


def test_packed_sequences_d64():
    lengths = [1, 64, 65, 130, 0, 7, 300]
    w = replace(WORKLOADS[4], H=2, dk=64, dv=64, seed=61)
    x = make_inputs(w, lengths=lengths)
    xc = cuda(x)
    o, S = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                             initial_state=xc["S0"], cu_seqlens=xc["cu_seqlens"], chunk=64)
    torch.cuda.synchronize()
    ro, rS = _oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "packed d=64 o")
    assert_parity(S, rS, torch.bfloat16, "packed d=64 final states")


def test_checkpoints_d64_dv96():
    dk, dv, every, slots = 64, 96, 128, 3
    w = replace(WORKLOADS[1], H=2, dk=dk, dv=dv, seed=62, initial_state=True)
    x = make_inputs(w, B=2, T=300)
    xc = cuda(x)
    ck = torch.full((2, 2, slots, dk, dv), float("nan"), device="cuda")
    kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                      initial_state=xc["S0"], chunk=64, checkpoints=ck, checkpoint_every=every)
    torch.cuda.synchronize()
    ck = ck.cpu()
    for n in range(2):
        for i in range(slots):
            p = (i + 1) * every
            if p <= 300:
                _, ref = oracle.recurrent(*(x[nm][n:n + 1, :p] for nm in NAMES), x["A"],
                                          S0=x["S0"][n:n + 1])
                assert_parity(ck[n, :, i], ref[0], torch.bfloat16, f"seq {n} checkpoint {i}")
            else:
                assert torch.isnan(ck[n, :, i]).all(), "slot past the sequence was written"


def test_from_host_d64_equals_device_call():
    w = replace(WORKLOADS[1], H=4, dk=64, dv=64, seed=63, initial_state=True)
    x = make_inputs(w, B=2, T=1000)
    xc = cuda(x)
    o_ref, S_ref = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                                     initial_state=xc["S0"], chunk=64)
    h = {n: x[n].contiguous().pin_memory() for n in NAMES}
    o_h, S = kda.chunk_prefill_from_host(h["q"], h["k"], h["v"], h["z"], h["beta"], xc["A"],
                                         initial_state=xc["S0"], segment_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu()), "o differs from the single device call"
    assert torch.equal(S.cpu(), S_ref.cpu()), "final state differs from the single device call"


def test_unsupported_narrow_shapes_take_the_recurrent_path():
    for dk, dv in [(48, 48), (40, 64), (64, 16), (8, 32), (64, 160)]:
        assert kda.prefill_path(dk, dv, 64, torch.bfloat16) == "recurrent", (dk, dv)
