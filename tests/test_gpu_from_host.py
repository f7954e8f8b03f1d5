"""kda_chunk_prefill_from_host: host inputs and output, copies overlapped with the kernels.

The segmented run continues each segment from the fp32 state the previous one
left, with chunk boundaries at the same tokens, so its o and final state must
equal one kda_chunk_prefill call on the whole batch bit for bit; the oracle
pins the result as well.
"""
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda

pytestmark = pytest.mark.gpu


def _pinned(x):
    return {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "z", "beta")}


@pytest.mark.parametrize("B,T,seg,with_s0", [(1, 4096, 1024, True), (2, 1000, 256, False),
                                             (1, 63, 64, True), (2, 3000, 8192, True)])
def test_from_host_equals_device_call(B, T, seg, with_s0):
    w = replace(WORKLOADS[2], H=4, seed=81 + T, initial_state=with_s0)
    x = make_inputs(w, B=B, T=T)
    xc = cuda(x)
    o_ref, S_ref = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                                     initial_state=xc["S0"], chunk=64)
    h = _pinned(x)
    o_h, S = kda.chunk_prefill_from_host(h["q"], h["k"], h["v"], h["z"], h["beta"], xc["A"],
                                         initial_state=xc["S0"], segment_tokens=seg)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_ref.cpu()), "o differs from the single device call"
    assert torch.equal(S.cpu(), S_ref.cpu()), "final state differs from the single device call"
    # and against the oracle on one sequence and all heads
    ro, rS = oracle.recurrent(*(x[n][B - 1:B] for n in ("q", "k", "v", "z", "beta")), x["A"],
                              S0=None if x["S0"] is None else x["S0"][B - 1:B])
    assert_parity(o_h[B - 1], ro, torch.bfloat16, "o vs oracle")
    assert_parity(S.cpu()[B - 1:B], rS, torch.bfloat16, "S vs oracle")


def test_from_host_state_in_place():
    """initial_state may be the final_state buffer itself."""
    w = replace(WORKLOADS[2], H=2, seed=88)
    x = make_inputs(w, B=1, T=700)
    xc = cuda(x)
    o_ref, S_ref = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                                     initial_state=xc["S0"], chunk=64)
    S = xc["S0"].clone()
    h = _pinned(x)
    o_h, S2 = kda.chunk_prefill_from_host(h["q"], h["k"], h["v"], h["z"], h["beta"], xc["A"],
                                          initial_state=S, final_state=S, segment_tokens=128)
    torch.cuda.synchronize()
    assert S2.data_ptr() == S.data_ptr()
    assert torch.equal(o_h, o_ref.cpu()) and torch.equal(S.cpu(), S_ref.cpu())
