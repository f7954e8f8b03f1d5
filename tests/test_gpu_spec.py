"""kda_spec_verify / kda_spec_commit against the fp64 oracle (through the C ABI)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300.inputs import WORKLOADS, make_inputs
from tests.parity import assert_parity, cuda, rel_err

pytestmark = pytest.mark.gpu


def _draft(B, T, H, d, dtype, seed):
    """Draft tokens [B, T, H, d] and a start state [B, H, d, d]."""
    w = replace(WORKLOADS[1], H=H, dk=d, dv=d, dtype=dtype, seed=seed, initial_state=True)
    return make_inputs(w, B=B, T=T)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,T,H,d", [(3, 1, 2, 128), (3, 4, 2, 128), (2, 16, 3, 128), (2, 5, 2, 64),
                                     (2, 6, 2, 64)])
def test_verify_outputs_and_state_untouched(B, T, H, d, dtype):
    x = _draft(B, T, H, d, dtype, seed=B * 10 + T + d)
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.spec_verify(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    torch.cuda.synchronize()
    assert torch.equal(state, xc["S0"]), "verify must not modify the state"
    ro, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    # fp32 inputs, and up to 5 bf16 tokens: token by token in fp32.  More bf16 tokens: the
    # span as one 16-token chunk on the tensor cores, held to the layer's bf16 bound like
    # the tensor-core prefill.
    assert_parity(o.reshape(ro.shape), ro, dtype, f"verify B={B} T={T} d={d}")
    if dtype == torch.float32:
        assert rel_err(o.reshape(ro.shape), ro) < 1e-5
    if dtype == torch.bfloat16 and T <= 5:
        # fp32 arithmetic: only the bf16 rounding of o itself remains
        assert rel_err(o.reshape(ro.shape), ro) < 5e-3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_commit_accepted_prefix(dtype):
    B, T, H, d = 5, 6, 2, 128
    x = _draft(B, T, H, d, dtype, seed=91)
    xc = cuda(x)
    n_acc = torch.tensor([0, 1, 3, 6, 9], dtype=torch.int32)       # 9 is clamped to T
    state = xc["S0"].clone()
    kda.spec_commit(xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state, n_acc.cuda())
    torch.cuda.synchronize()
    got = state.cpu()
    assert torch.equal(got[0], x["S0"][0]), "n_accept = 0 leaves the state untouched"
    for b in range(1, B):
        n = min(int(n_acc[b]), T)
        _, rS = oracle.recurrent(*(x[nm][b:b + 1, :n] for nm in ("q", "k", "v", "z", "beta")),
                                 x["A"], S0=x["S0"][b:b + 1])
        assert_parity(got[b], rS[0], dtype, f"commit b={b} n={n}")
        assert rel_err(got[b], rS[0]) < 1e-5                          # fp32 state arithmetic


def test_verify_then_commit_equals_decode_steps():
    B, T, H, d = 4, 5, 2, 128
    x = cuda(_draft(B, T, H, d, torch.bfloat16, seed=92))
    st_spec = x["S0"].clone()
    o_spec = kda.spec_verify(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], st_spec)
    kda.spec_commit(x["k"], x["v"], x["z"], x["beta"], x["A"], st_spec,
                    torch.full((B,), T, dtype=torch.int32, device="cuda"))
    st_dec = x["S0"].clone()
    o_dec = [kda.decode_step(x["q"][:, t].contiguous(), x["k"][:, t].contiguous(),
                             x["v"][:, t].contiguous(), x["z"][:, t].contiguous(),
                             x["beta"][:, t].contiguous(), x["A"], st_dec) for t in range(T)]
    torch.cuda.synchronize()
    assert (o_spec.float() - torch.stack(o_dec, 1).float()).abs().max() <= 1e-2
    assert (st_spec - st_dec).abs().max() <= 1e-5 * st_dec.abs().max()


def test_full_size_verify_commit_b256_h32():
    B, T, H, d = 256, 4, 32, 128
    x = _draft(B, T, H, d, torch.bfloat16, seed=93)
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.spec_verify(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    n_acc = torch.randint(0, T + 1, (B,), generator=torch.Generator().manual_seed(5),
                          dtype=torch.int32)
    kda.spec_commit(xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state, n_acc.cuda())
    torch.cuda.synchronize()
    ro, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "verify B=256 H=32 T=4")
    got = state.cpu()
    for b in range(0, B, 37):
        n = int(n_acc[b])
        if n == 0:
            assert torch.equal(got[b], x["S0"][b])
            continue
        _, rS = oracle.recurrent(*(x[nm][b:b + 1, :n] for nm in ("q", "k", "v", "z", "beta")),
                                 x["A"], S0=x["S0"][b:b + 1])
        assert rel_err(got[b], rS[0]) < 1e-5


def test_verify_falls_back_to_fp32_for_other_head_sizes():
    # d_k = 40 is not a multiple of 16: bf16 verify runs token by token in fp32.
    w = replace(WORKLOADS[1], H=2, dk=40, dv=40, seed=94, initial_state=True)
    x = make_inputs(w, B=3, T=7)
    xc = cuda(x)
    o = kda.spec_verify(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], xc["S0"])
    torch.cuda.synchronize()
    ro, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "verify d=40 (fp32 path)")
    assert rel_err(o.reshape(ro.shape), ro) < 5e-3


def test_full_size_verify_t16_all_pairs():
    B, T, H, d = 256, 16, 32, 128
    x = _draft(B, T, H, d, torch.bfloat16, seed=95)
    xc = cuda(x)
    o = kda.spec_verify(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], xc["S0"])
    torch.cuda.synchronize()
    ro, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "verify B=256 H=32 T=16 (all pairs)")


def test_verify_tensor_cores_uneven_pairs_per_cta():
    # 640 (b, h) pairs: more than the two resident CTAs per SM, so the persistent
    # CTAs walk two or three pairs each and prefetch across pairs; T = 7 leaves
    # nine empty token rows of the 16-token chunk, d_k = 64 and d_v = 48 leave
    # channels of the 128-wide tiles empty.
    w = replace(WORKLOADS[1], H=2, dk=64, dv=48, seed=97, initial_state=True)
    x = make_inputs(w, B=320, T=7)
    xc = cuda(x)
    state = xc["S0"].clone()
    o = kda.spec_verify(xc["q"], xc["k"], xc["v"], xc["z"], xc["beta"], xc["A"], state)
    torch.cuda.synchronize()
    assert torch.equal(state, xc["S0"])
    ro, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], S0=x["S0"])
    assert_parity(o.reshape(ro.shape), ro, torch.bfloat16, "verify B=320 H=2 T=7 dk=64 dv=48")
