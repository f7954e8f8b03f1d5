"""kda_chunk_prefill_static_workspace: prefill without a caller workspace.

Some callers cannot allocate device memory when they run the layer (a plugin
whose host runtime owns every device allocation, or a serving loop with a
memory plan fixed at start-up).  For them the library keeps a fixed
__device__ scratch array and this entry point uses it in place of the
workspace kda_chunk_prefill takes.  These tests call it through the C ABI and
check it against kda_chunk_prefill on the same inputs, twice in a row.  Both
run the same kernels on the same inputs, so the results must agree bit for
bit: any difference would mean that a call depends on what an earlier call
left in the shared array.  After each call the array's device status word must
read 0 (no bounded wait gave up).  The file is named to be collected last.
"""
import ctypes
from dataclasses import replace

import pytest
import torch

import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300 import api
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs


def _static_status() -> int:
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    kda.static_workspace_status(st)
    torch.cuda.synchronize()
    return int(st.item())

pytestmark = pytest.mark.gpu

STATIC_BYTES = 64 * 1024 * 1024      # KDA_STATIC_WORKSPACE_BYTES in include/kda.h


def _call_static(x, o, S):
    """Direct C-ABI call of kda_chunk_prefill_static_workspace."""
    L = kda.lib()
    q = x["q"]
    B, T, H, dk = q.shape
    dv = x["v"].shape[-1]
    cu = x.get("cu_seqlens")
    n = B if cu is None else cu.numel() - 1
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return L.kda_chunk_prefill_static_workspace(
        p(q), p(x["k"]), p(x["v"]), p(x["z"]), p(x["beta"]), p(x["A"]), p(o), p(x["S0"]),
        p(S), p(cu), n, B, T, H, dk, dv, 64, 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs(seed, T, H=4, lengths=None):
    if lengths is not None:
        w = replace(WORKLOADS[4], H=H, seed=seed)
        x = make_inputs(w, lengths=lengths)
    else:
        w = replace(WORKLOADS[2], H=H, seed=seed)
        x = make_inputs(w, B=1, T=T)
    return {n: (t.cuda() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}


@pytest.mark.parametrize("case", ["fixed", "packed"])
def test_static_workspace_matches_caller_workspace_twice(case):
    # Two different inputs back to back through the static array.
    if case == "fixed":
        runs = [_inputs(seed=501, T=1000), _inputs(seed=502, T=777)]
    else:
        runs = [_inputs(seed=503, T=0, lengths=[300, 1, 64, 129]),
                _inputs(seed=504, T=0, lengths=[65, 700, 2])]
    assert kda.prefill_path(128, 128, 64, torch.bfloat16) == "chunked_tc"
    for x in runs:
        B, T, H, dk = x["q"].shape
        n = B if x.get("cu_seqlens") is None else x["cu_seqlens"].numel() - 1
        assert 0 < kda.workspace_size(n, B, T, H, dk, 128, 64, torch.bfloat16) <= STATIC_BYTES
        o = torch.full((B, T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        S = torch.full((n, H, dk, 128), float("nan"), device="cuda")
        assert _call_static(x, o, S) == 0, kda.lib().kda_last_error()
        torch.cuda.synchronize()
        assert _static_status() == 0
        ro, rS = kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                                   initial_state=x["S0"], cu_seqlens=x.get("cu_seqlens"),
                                   chunk=64)
        torch.cuda.synchronize()
        assert torch.equal(o, ro), "static-workspace o differs from kda_chunk_prefill"
        assert torch.equal(S, rS), "static-workspace state differs from kda_chunk_prefill"


def test_static_workspace_binding_and_size_limit():
    x = _inputs(seed=505, T=300, H=2)
    o, S = api.chunk_prefill_static_workspace(x["q"], x["k"], x["v"], x["z"], x["beta"],
                                              x["A"], initial_state=x["S0"])
    ro, rS = kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                               initial_state=x["S0"])
    torch.cuda.synchronize()
    assert _static_status() == 0
    assert torch.equal(o, ro) and torch.equal(S, rS)
    # A shape whose workspace exceeds the static array is rejected before any launch.
    L = kda.lib()
    T_big = 1 << 20
    need = L.kda_chunk_prefill_workspace_size(1, 1, T_big, 32, 128, 128, 64, 1)
    assert need > STATIC_BYTES
    f = ctypes.c_void_p(x["q"].data_ptr())
    rc = L.kda_chunk_prefill_static_workspace(f, f, f, f, f, f, f, None, None, None, 1, 1, T_big,
                                              32, 128, 128, 64, 1, None)
    assert rc == 2
    assert b"static workspace" in L.kda_last_error()
