"""Seeded synthetic inputs for the KDA layer.

This module is the one piece of code that both the CUDA path and the fp64
oracle consume, so it holds none of the layer's arithmetic: it only draws
random tensors with the distributions of the workloads below.  Every tensor
comes from one torch.Generator seeded with the workload's seed, drawn in a
fixed order: sequence lengths (packed workloads only), A, q, k, v, z, beta,
initial state.

Distributions (N(m, s) means mean m, standard deviation s):
  q, k   N(0, 1), then divided by their L2 norm per (token, head)
  v, z   N(0, 1)
  beta   sigmoid(N(0, 1))            -- a write strength in (0, 1)
  A      N(0, 0.5) per (head, channel)
  S0     N(0, 0.02) fp32 where the workload has an initial state
  "z floor" workloads set z = +8 on channels [0, dk/2) of every token and
  head, which drives those channels' log-decay to its -5 floor.
Values are drawn in fp32 and then rounded once to the workload's input dtype;
both sides see the identical rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" | "decode"
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    seed: int
    B: int = 1
    T: int = 0
    chunk: int = 64
    initial_state: bool = False
    z_floor_half: bool = False
    n_seqs: int = 0           # > 0: packed variable-length batch
    max_len: int = 0          # lengths uniform in [1, max_len]
    note: str = field(default="")


# The five workloads of the layer's specification, indexed by seed.
WORKLOADS = {
    0: Workload("tiny-f32", "prefill", H=1, dk=16, dv=16, dtype=torch.float32, seed=0,
                B=1, T=64, chunk=16,
                note="B=1 H=1 T=64 d=16 fp32 chunk 16, S0=0"),
    1: Workload("prefill-b2-h8-t4096", "prefill", H=8, dk=128, dv=128, dtype=torch.bfloat16,
                seed=1, B=2, T=4096, chunk=64,
                note="B=2 H=8 T=4096 d=128 bf16 chunk 64, S0=0"),
    2: Workload("long-prefill-h32-t65536", "prefill", H=32, dk=128, dv=128,
                dtype=torch.bfloat16, seed=2, B=1, T=65536, chunk=64, initial_state=True,
                z_floor_half=True,
                note="B=1 H=32 T=65536 d=128 bf16 chunk 64, S0~N(0,0.02), z=+8 on half the channels"),
    3: Workload("decode-b256-h32", "decode", H=32, dk=128, dv=128, dtype=torch.bfloat16,
                seed=3, B=256, T=1, initial_state=True,
                note="B=256 H=32 d=128 one token, S~N(0,0.02) fp32 in place"),
    4: Workload("varlen-64seq-h16", "prefill", H=16, dk=128, dv=128, dtype=torch.bfloat16,
                seed=4, chunk=64, initial_state=True, n_seqs=64, max_len=32768,
                note="64 packed sequences, lengths U{1..32768}, H=16 d=128 bf16 chunk 64, "
                     "per-sequence S0~N(0,0.02)"),
}


def _normal(gen, shape, std=1.0, device="cpu"):
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device) * std


def _unit_rows(x):
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_lengths(n_seqs: int, max_len: int, gen) -> torch.Tensor:
    """Sequence lengths uniform on {1, ..., max_len} (int64, CPU)."""
    return torch.randint(1, max_len + 1, (n_seqs,), generator=gen, dtype=torch.int64)


def make_inputs(w: Workload, device: str = "cpu", T: int | None = None, B: int | None = None,
                lengths=None) -> dict:
    """Draws every input tensor of workload ``w``.

    ``T``/``B`` override the token count / batch of a fixed-length workload, and
    ``lengths`` the sequence lengths of a packed one (for scaled-down parity cases).
    Returns a dict with q, k, v, z, beta, A, S0 (or None) and, for packed
    workloads, cu_seqlens (int32, CPU) and lengths; prefill tensors are
    [B, T, H, d] (or packed [1, T_total, H, d]), decode tensors [B, H, d].
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    cpu_gen = gen if device == "cpu" else torch.Generator().manual_seed(w.seed)
    out = {}
    if w.kind == "prefill" and (w.n_seqs > 0 or lengths is not None):
        if lengths is None:
            lengths = make_lengths(w.n_seqs, w.max_len, cpu_gen)
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lengths, 0)
        out["lengths"] = lengths
        out["cu_seqlens"] = cu.to(torch.int32)
        lead = (1, int(cu[-1]))
        n_states = len(lengths)
    elif w.kind == "prefill":
        lead = (w.B if B is None else B, w.T if T is None else T)
        n_states = lead[0]
    else:
        lead = (w.B if B is None else B,)
        n_states = lead[0]
    H, dk, dv = w.H, w.dk, w.dv

    out["A"] = _normal(gen, (H, dk), 0.5, device)
    q = _unit_rows(_normal(gen, lead + (H, dk), 1.0, device))
    k = _unit_rows(_normal(gen, lead + (H, dk), 1.0, device))
    v = _normal(gen, lead + (H, dv), 1.0, device)
    z = _normal(gen, lead + (H, dk), 1.0, device)
    beta = torch.sigmoid(_normal(gen, lead + (H,), 1.0, device))
    if w.z_floor_half:
        z[..., : dk // 2] = 8.0
    for name, t in (("q", q), ("k", k), ("v", v), ("z", z), ("beta", beta)):
        out[name] = t.to(w.dtype)
    if w.initial_state:
        out["S0"] = _normal(gen, (n_states, H, dk, dv), 0.02, device)
    else:
        out["S0"] = None
    return out


def token_heads(w: Workload, inputs: dict) -> int:
    """Work units of one pass: tokens x heads (prefill) or sequences x heads (decode)."""
    if w.kind == "decode":
        return inputs["q"].shape[0] * w.H
    return inputs["q"].shape[0] * inputs["q"].shape[1] * w.H
