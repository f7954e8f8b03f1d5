"""Failure detection without a GPU fault.

The tensor-core kernels bound every mbarrier wait (about 2 s), then record a
status and return.  kda_selftest_bounded_wait runs that same wait on a barrier
nothing arrives on: it must give up within its bound, say so, and leave the
context usable; the control case (the barrier completed by its own arrival)
must not give up.
"""
import time
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    kda.selftest_bounded_wait(status, arrive=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a completed barrier must not time out"

    status.fill_(7)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kda.selftest_bounded_wait(status, arrive=False)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == 1, "the wait on a barrier nothing completes must give up"
    assert 1.5 < dt < 30.0, f"the bounded wait gave up after {dt:.2f} s, not about 2 s"

    # the context still runs the layer correctly
    w = replace(WORKLOADS[1], H=2, seed=95)
    x = make_inputs(w, B=1, T=130)
    xc = cuda(x)
    o, S = kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], chunk=64)
    torch.cuda.synchronize()
    ro, rS = oracle.recurrent(*(x[n] for n in ("q", "k", "v", "z", "beta")), x["A"])
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "prefill after the timed-out wait")
    assert_parity(S, rS, torch.bfloat16, "final state after the timed-out wait")
