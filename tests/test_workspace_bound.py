"""Host-side check of the package-slot scheme of the tensor-core prefill.

Sequence n's packages start at slot floor(bos_n / 64) + n.  The workspace holds
floor(T / 64) + n_seqs + 1 slots per head, so every slot a sequence uses must
stay below that bound for valid and for malformed offsets (which the kernels
clamp into [0, T]).  The workspace-size query must match the bound.
"""
import random

import gated_delta_rule_34_gb300 as kda

PKG_BYTES = 99328
HEADER = 1024


def _clamped(cu, n, T):
    b, e = cu[n], cu[n + 1]
    b = min(max(b, 0), T)
    e = min(max(e, b), T)
    return b, e


def test_slots_stay_in_bounds():
    rng = random.Random(0)
    for _ in range(20000):
        N = rng.randint(1, 12)
        T = rng.randint(0, 700)
        if rng.random() < 0.5:
            cuts = sorted(rng.randint(0, T) for _ in range(N - 1))
            cu = [0] + cuts + [T]
        else:
            cu = [rng.randint(-100, T + 100) for _ in range(N + 1)]
        slots = T // 64 + N + 1
        used = set()
        for n in range(N):
            b, e = _clamped(cu, n, T)
            base = b // 64 + n
            nc = (e - b + 63) // 64
            assert nc == 0 or base + nc - 1 < slots
            if cu == sorted(cu) and cu[0] == 0 and cu[-1] == T:
                run = set(range(base, base + nc))
                assert not (run & used), "valid offsets must give disjoint slots"
                used |= run


def test_workspace_size_query_matches_bound():
    # Packages of the plain pass (the segment-parallel records come on top of them for
    # fixed-length batches that kda_chunk_prefill splits into segments).
    L = kda.lib()
    for n_seqs, B, T, H in [(1, 1, 4096, 8), (2, 2, 4096, 8), (64, 1, 1048576, 16), (3, 1, 1, 1),
                            (1, 1, 65536, 32)]:
        slots = (B * T) // 64 + n_seqs + 1
        packages = HEADER + slots * H * PKG_BYTES
        got = L.kda_chunk_prefill_workspace_size(n_seqs, B, T, H, 128, 128, 64, 1)
        if n_seqs != B:                       # packed: never segmented
            assert got == packages
            continue
        G = L.kda_chunk_prefill_auto_segments(B, T, H, 128, 128, 64, 1)
        assert got == packages + n_seqs * H * (G - 1) * (128 + 64) * 1024
        assert L.kda_chunk_prefill_segmented_workspace_size(B, T, H, 128, 128, 64, 1, 1) == packages
