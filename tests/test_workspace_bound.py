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


WINDOW = 262144         # tokens per launch of the 64-token path (per sequence when fixed)
CARRY = 128 * 128 * 4   # bytes of carried state per (sequence, head) between windows


def test_workspace_size_query_matches_bound():
    # Packages of one window (the segment-parallel records come on top of them for
    # fixed-length batches that kda_chunk_prefill splits into segments, and a carry area
    # for calls that run in several windows).
    L = kda.lib()
    for n_seqs, B, T, H in [(1, 1, 4096, 8), (2, 2, 4096, 8), (64, 1, 1048576, 16), (3, 1, 1, 1),
                            (1, 1, 65536, 32), (1, 1, 1 << 20, 32), (2, 2, 600000, 4),
                            (64, 64, 65536, 32), (3, 3, 100000, 2), (5000, 5000, 100, 1)]:
        fixed = n_seqs == B
        span = T if fixed else B * T
        W = max(64, WINDOW // B // 64 * 64) if fixed and B > 1 else WINDOW
        w = min(span, W)
        slots = (B * w if fixed else w) // 64 + n_seqs + 1
        packages = HEADER + slots * H * PKG_BYTES
        carry = n_seqs * H * CARRY if span > w else 0
        got = L.kda_chunk_prefill_workspace_size(n_seqs, B, T, H, 128, 128, 64, 1)
        if not fixed:                         # packed: never segmented
            assert got == packages + carry
            continue
        G = L.kda_chunk_prefill_auto_segments(B, T, H, 128, 128, 64, 1)
        seg = packages + n_seqs * H * (G - 1) * (128 + 64) * 1024 + carry
        if B == 1 and span > w:               # a single sequence may also come packed
            packed = HEADER + (w // 64 + 2) * H * PKG_BYTES + H * CARRY
            assert got == max(seg, packed)
        else:
            assert got == seg
        assert (L.kda_chunk_prefill_segmented_workspace_size(B, T, H, 128, 128, 64, 1, 1)
                == packages + carry)


def test_workspace_is_bounded_by_one_window():
    # A million-token, 32-head prefill needs one 262,144-token window of packages
    # (about 13 GB), not the ~52 GB its whole length would; four million tokens need no more.
    L = kda.lib()
    big = L.kda_chunk_prefill_workspace_size(1, 1, 1 << 20, 32, 128, 128, 64, 1)
    huge = L.kda_chunk_prefill_workspace_size(1, 1, 1 << 22, 32, 128, 128, 64, 1)
    one = L.kda_chunk_prefill_workspace_size(1, 1, WINDOW, 32, 128, 128, 64, 1)
    assert big < 14e9 and big == huge and big <= one + 32 * CARRY + 2 * 32 * PKG_BYTES
    packed = L.kda_chunk_prefill_workspace_size(64, 1, 1 << 22, 16, 128, 128, 64, 1)
    assert packed < 7e9
    # a large fixed-length batch is windowed over the batch's tokens, not per sequence
    batch = L.kda_chunk_prefill_workspace_size(64, 64, 65536, 32, 128, 128, 64, 1)
    assert batch < 14e9


def _window_part(b, e, w0, w1):
    """A sequence's chunks whose first row lies in [w0, w1), chunks counted from b."""
    def align(w):
        return b if w <= b else b + (w - b + 63) // 64 * 64
    lo, hi = align(w0), align(w1)
    bos, eos = min(lo, e), min(hi, e)
    return bos, max(eos, bos)


def test_packed_window_slots_stay_in_bounds_and_cover_every_chunk_once():
    rng = random.Random(1)
    for _ in range(3000):
        N = rng.randint(1, 9)
        lens = [rng.choice([0, 1, 63, 64, 65, rng.randint(0, 3000)]) for _ in range(N)]
        cu = [0]
        for ln in lens:
            cu.append(cu[-1] + ln)
        T = cu[-1]
        W = rng.choice([64, 128, 256, 1024])
        seen = {n: set() for n in range(N)}
        w0 = 0
        while True:
            w1 = min(T, w0 + W)
            slots = W // 64 + N + 1          # the workspace holds one full window
            used = set()
            last = -1
            for n in range(N):
                b, e = cu[n], cu[n + 1]
                bos, eos = _window_part(b, e, w0, w1)
                base = (max(bos, w0) - w0) // 64 + n
                assert base >= last, "slot bases rise with the sequence index"
                last = base
                nc = (eos - bos + 63) // 64
                run = set(range(base, base + nc))
                assert not (run & used) and all(0 <= s < slots for s in run)
                used |= run
                for c in range(nc):
                    start = bos + 64 * c
                    assert (start - b) % 64 == 0, "chunks stay on the sequence's own grid"
                    assert start not in seen[n], "a chunk runs in one window only"
                    seen[n].add(start)
            w0 = w1
            if w0 >= T:
                break
        for n in range(N):
            assert seen[n] == set(range(cu[n], cu[n + 1], 64)), "every chunk runs once"
