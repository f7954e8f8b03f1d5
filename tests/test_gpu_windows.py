"""GPU parity of the 64-token path on calls longer than one window (262,144 tokens per
sequence of a fixed-length batch, or in all of a packed one), through the C ABI.

Such calls run window by window with the fp32 state carried between windows, so the
workspace holds one window's packages.  Packed windows cut sequences wherever the window
ends (mid-chunk included); the chunked form is exact for any chunk boundaries, so the
result must still match the oracle.  The heads are narrow (d = 32 or 64) so that the fp64
oracle walks these long sequences in seconds.
"""
from dataclasses import replace

import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda
from tests.test_gpu_prefill import _run_with_status, run_oracle

pytestmark = pytest.mark.gpu

WINDOW = 262144


def test_fixed_length_three_windows():
    w = replace(WORKLOADS[2], H=2, dk=32, dv=32, seed=800)
    x = make_inputs(w, device="cuda", B=1, T=2 * WINDOW + 8928)   # windows of W, W, 8928
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "3 windows o")
    assert_parity(S, rS, torch.bfloat16, "3 windows state")


def test_packed_windows_cut_sequences_mid_chunk():
    lengths = [200000, 120001, 1, 280000, 0, 5, 333]
    w = replace(WORKLOADS[4], H=2, dk=32, dv=32, seed=801)
    x = make_inputs(w, lengths=lengths)
    assert sum(lengths) > 2 * WINDOW
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle(x)
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "packed windows o")
    assert_parity(S, rS, torch.bfloat16, "packed windows state")


def test_windows_without_final_state():
    # The carried state then lives in the workspace.
    w = replace(WORKLOADS[2], H=1, dk=32, dv=32, seed=802)
    x = cuda(make_inputs(w, B=2, T=WINDOW + 4000))
    o, S = kda.chunk_prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"],
                             initial_state=x["S0"], output_final_state=False)
    torch.cuda.synchronize()
    assert S is None
    ro, _ = run_oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "windows, no final state, o")


def test_checkpoints_across_windows():
    w = replace(WORKLOADS[4], H=1, dk=32, dv=32, seed=803)
    lengths = [360003, 200000]
    x = make_inputs(w, lengths=lengths)
    xc = cuda(x)
    every = 32768
    slots = max(lengths) // every
    ck = torch.full((2, 1, slots, 32, 32), float("nan"), device="cuda")
    kda.chunk_prefill(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                      initial_state=xc["S0"], cu_seqlens=xc["cu_seqlens"], checkpoints=ck,
                      checkpoint_every=every)
    torch.cuda.synchronize()
    cu = x["cu_seqlens"].tolist()
    # sequence 1 starts at row 360003 and crosses the window edge at 524288 61 rows into a
    # chunk of its own 64-token grid; its checkpoint 4 lies before that edge, 5 after it
    for n, i in [(0, 0), (0, 7), (0, 8), (0, 9), (1, 1), (1, 4), (1, 5)]:
        m = (i + 1) * every
        rng = slice(cu[n], cu[n] + m)
        _, rS = oracle.recurrent(*(x[nm][0, rng] for nm in ("q", "k", "v", "z", "beta")), x["A"],
                                 S0=x["S0"][n:n + 1], cu_seqlens=torch.tensor([0, m]))
        assert_parity(ck[n, 0, i], rS[0, 0], torch.bfloat16, f"window checkpoint seq {n} #{i}")


def test_windowed_plain_pass_equals_host_segments_bit_for_bit():
    # One segment per window (no segment split) and host-buffer segments of 8,192 tokens
    # both hand the fp32 state on at 64-token-aligned points: the results are identical.
    w = replace(WORKLOADS[2], H=2, dk=32, dv=32, seed=804)
    x = make_inputs(w, B=1, T=2 * WINDOW + 640)
    xc = cuda(x)
    o1, S1 = kda.chunk_prefill_segmented(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"],
                                         1, initial_state=xc["S0"])
    h = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "z", "beta")}
    o2, S2 = kda.chunk_prefill_from_host(h["q"], h["k"], h["v"], h["z"], h["beta"], xc["A"],
                                         initial_state=xc["S0"], segment_tokens=8192)
    torch.cuda.synchronize()
    assert torch.equal(o1.cpu(), o2) and torch.equal(S1, S2)


def test_segmented_windows():
    # Few heads and two windows: each window is split into segments, and the second
    # window's first segment starts from the carried state.
    w = replace(WORKLOADS[2], H=1, dk=64, dv=64, seed=805)
    x = make_inputs(w, device="cuda", B=1, T=WINDOW + 40000)
    assert kda.auto_segments(1, WINDOW + 40000, 1, 64, 64) > 1
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "segmented windows o")
    assert_parity(S, rS, torch.bfloat16, "segmented windows state")


def test_fixed_length_batch_windows():
    # Eight sequences share a window: 262,144 / 8 = 32,768 positions each, so 40,000
    # tokens per sequence run in two windows.
    w = replace(WORKLOADS[2], H=2, dk=32, dv=32, seed=806)
    x = make_inputs(w, device="cuda", B=8, T=40000)
    o, S, status = _run_with_status(x)
    assert status == 0
    ro, rS = run_oracle({n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()})
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "batch windows o")
    assert_parity(S, rS, torch.bfloat16, "batch windows state")
