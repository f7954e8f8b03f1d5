"""GPU parity of kda_gate and kda_decode_step against the fp64 oracle (through the C ABI)."""
import math

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(37, 3, 128), (5, 2, 16), (3, 1, 12), (1, 4, 7)])
def test_gate_matches_oracle(dtype, shape):
    g = torch.Generator().manual_seed(sum(shape))
    z = (torch.randn(shape, generator=g) * 4).to(dtype)
    A = torch.randn(shape[1], shape[2], generator=g) * 0.5
    out = kda.gate(z.cuda(), A.cuda())
    torch.cuda.synchronize()
    ref = oracle.gate(z, A)
    got = out.cpu().double().numpy()
    assert np.all(got >= -5.0) and np.all(got <= 0.0)
    assert np.abs(got - ref).max() <= 2e-6           # fp32 arithmetic on exact inputs


def test_gate_special_points():
    z = torch.tensor([[[0.0, float("inf"), float("-inf"), 1e30, -1e30, 8.0, math.log(3.0), 0.0]]])
    A = torch.tensor([[0.0, 0.0, 0.0, 0.0, 0.0, 30.0, 0.0, -50.0]])
    got = kda.gate(z.cuda(), A.cuda()).cpu().numpy()[0, 0]
    assert got[0] == -2.5 and got[1] == -5.0 and got[2] == 0.0
    assert got[3] == -5.0 and got[4] == 0.0 and got[5] == -5.0
    assert abs(got[6] - (-3.75)) < 1e-6 and got[7] == -2.5


def test_gate_empty():
    z = torch.empty(0, 2, 16, device="cuda")
    out = kda.gate(z, torch.zeros(2, 16, device="cuda"))
    assert out.shape == (0, 2, 16)


def _decode_case(B, H, d, dtype, seed):
    w = WORKLOADS[3]
    from dataclasses import replace
    w = replace(w, H=H, dk=d, dv=d, dtype=dtype, seed=seed)
    return make_inputs(w, B=B)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,d", [(4, 3, 128), (3, 2, 64), (2, 2, 20), (1, 1, 4)])
def test_decode_matches_oracle(B, H, d, dtype):
    x = _decode_case(B, H, d, dtype, seed=B * 100 + d)
    S0 = x["S0"].clone()
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.decode_step(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    torch.cuda.synchronize()
    # Decode = one token per sequence: the recurrence with B sequences of length 1.
    ro, rS = oracle.recurrent(x["q"][:, None], x["k"][:, None], x["v"][:, None],
                              x["z"][:, None], x["beta"][:, None], x["A"], S0=S0)
    assert_parity(o, ro[:, :, :].reshape(B, H, d), dtype, "decode o")
    assert_parity(state, rS, dtype, "decode state")
    # The state never passes through the input dtype: fp32 arithmetic throughout.
    assert rel_err(state, rS) < 1e-5


@pytest.mark.parametrize("dk,dv", [(128, 48), (96, 64), (48, 96), (24, 128)])
def test_decode_unequal_head_sizes(dk, dv):
    # CTAs of a warp per 16 columns of S, at least four warps (which load all d_k
    # channels): four warps for d_v <= 64, six for d_v = 96, eight for d_v = 128.
    from dataclasses import replace
    w = replace(WORKLOADS[3], H=3, dk=dk, dv=dv, dtype=torch.bfloat16, seed=dk + dv)
    x = make_inputs(w, B=5)
    S0 = x["S0"].clone()
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.decode_step(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(x["q"][:, None], x["k"][:, None], x["v"][:, None],
                              x["z"][:, None], x["beta"][:, None], x["A"], S0=S0)
    assert_parity(o, ro.reshape(5, 3, dv), torch.bfloat16, f"decode o dk={dk} dv={dv}")
    assert rel_err(state, rS) < 1e-5


def test_decode_full_workload():
    w = WORKLOADS[3]
    x = make_inputs(w)
    S0 = x["S0"].clone()
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.decode_step(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(x["q"][:, None], x["k"][:, None], x["v"][:, None],
                              x["z"][:, None], x["beta"][:, None], x["A"], S0=S0)
    assert_parity(o, ro.reshape(o.shape), torch.bfloat16, "decode o (256x32)")
    assert rel_err(state, rS) < 1e-5


def test_decode_repeated_steps_equal_prefill_recurrence():
    # n decode steps from S0 equal the recurrence over those n tokens.
    from dataclasses import replace
    w = replace(WORKLOADS[1], B=2, T=6, H=2, seed=31, initial_state=True)
    x = make_inputs(w)
    xc = cuda(x)
    state = xc["S0"].clone()
    outs = []
    for t in range(6):
        outs.append(kda.decode_step(xc["q"][:, t].contiguous(), xc["k"][:, t].contiguous(),
                                    xc["v"][:, t].contiguous(), xc["z"][:, t].contiguous(),
                                    xc["beta"][:, t].contiguous(), xc["A"], state))
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    assert_parity(torch.stack(outs, 1), ro.reshape(2, 6, 2, 128), torch.bfloat16, "decode x6")
    assert rel_err(state, rS) < 1e-5


def test_decode_empty_batch():
    e = torch.empty(0, 2, 128, device="cuda", dtype=torch.bfloat16)
    st = torch.empty(0, 2, 128, 128, device="cuda")
    o = kda.decode_step(e, e, e, e, torch.empty(0, 2, device="cuda", dtype=torch.bfloat16),
                        torch.zeros(2, 128, device="cuda"), st)
    assert o.shape == (0, 2, 128)
