"""The C ABI without a GPU: exported symbols and host-side argument checks.

Every call here is rejected by validation before anything is launched, so the
tests run on a machine without a CUDA device.
"""
import ctypes
import os
import re
import subprocess

import pytest

import gated_delta_rule_34_gb300 as kda
from gated_delta_rule_34_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 4


@pytest.fixture(scope="module")
def L():
    from gated_delta_rule_34_gb300 import build
    build.build()
    return kda.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kda_gate", "kda_chunk_prefill", "kda_decode_step", "kda_status_string",
                 "kda_chunk_prefill_workspace_size", "kda_chunk_prefill_path", "kda_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", api.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(kda_\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(L, n)


def test_status_strings(L):
    for code, name in api.STATUS.items():
        assert L.kda_status_string(code).decode() == name
    assert L.kda_status_string(99).decode() == "KDA_ERR_UNKNOWN"


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def _prefill(L, **kw):
    a = dict(q=_fake(), k=_fake(), v=_fake(), z=_fake(), beta=_fake(), A=_fake(), o=_fake(),
             s0=None, s1=None, cu=None, n_seqs=1, B=1, T=8, H=2, dk=16, dv=16, chunk=16, dtype=0,
             ws=None, ws_bytes=0)
    a.update(kw)
    return L.kda_chunk_prefill(a["q"], a["k"], a["v"], a["z"], a["beta"], a["A"], a["o"],
                               a["s0"], a["s1"], a["cu"], a["n_seqs"], a["B"], a["T"], a["H"],
                               a["dk"], a["dv"], a["chunk"], a["dtype"], a["ws"], a["ws_bytes"],
                               None)


def test_prefill_rejects_bad_arguments(L):
    assert _prefill(L, q=None) == INVALID
    assert b"q is NULL" in L.kda_last_error()
    assert _prefill(L, k=_fake(0x10004)) == INVALID            # misaligned
    assert b"16-byte" in L.kda_last_error()
    assert _prefill(L, chunk=32) == INVALID
    assert _prefill(L, dtype=7) == INVALID
    assert _prefill(L, H=0) == INVALID
    assert _prefill(L, T=-1) == INVALID
    assert _prefill(L, n_seqs=2) == INVALID                     # != B without cu_seqlens
    assert _prefill(L, cu=_fake(), B=2, n_seqs=3) == INVALID    # packed needs B == 1
    assert _prefill(L, cu=_fake(0x10002)) == INVALID            # misaligned offsets
    assert _prefill(L, dk=256) == UNSUPPORTED
    assert _prefill(L, s0=_fake(0x10008)) == INVALID


def test_prefill_tc_path_requires_workspace(L):
    if L.kda_chunk_prefill_path(128, 128, 64, 1) != 1:
        pytest.skip("chunked tensor-core path not built")
    need = L.kda_chunk_prefill_workspace_size(1, 1, 4096, 2, 128, 128, 64, 1)
    assert need > 0
    rc = _prefill(L, dk=128, dv=128, chunk=64, dtype=1, T=4096, ws=None, ws_bytes=0)
    assert rc == WORKSPACE
    # The automatic segment split needs more than the plain pass and falls back to it
    # when the workspace only covers that; below the plain size the call is refused.
    plain = L.kda_chunk_prefill_segmented_workspace_size(1, 4096, 2, 128, 128, 64, 1, 1)
    assert 0 < plain <= need
    rc = _prefill(L, dk=128, dv=128, chunk=64, dtype=1, T=4096, ws=_fake(0x100000),
                  ws_bytes=plain - 1)
    assert rc == WORKSPACE
    rc = _prefill(L, dk=128, dv=128, chunk=64, dtype=1, T=4096, ws=_fake(0x100010),
                  ws_bytes=need)
    assert rc == INVALID                                        # not 256-byte aligned


def test_prefill_tc_path_rejects_token_counts_past_32_bit_coordinates(L):
    rc = _prefill(L, dk=128, dv=128, chunk=64, dtype=1, B=1, T=1 << 31, ws=_fake(0x100000),
                  ws_bytes=1 << 62)
    assert rc == UNSUPPORTED
    assert b"2^31" in L.kda_last_error()


def test_workspace_size_query(L):
    assert L.kda_chunk_prefill_workspace_size(1, 1, 64, 1, 16, 16, 16, 0) == 0   # SIMT path
    assert L.kda_chunk_prefill_workspace_size(0, 1, 64, 1, 128, 128, 64, 1) == 0


def test_path_query(L):
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(16, 16, 16, 0)] == "recurrent"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(128, 128, 64, 0)] == "recurrent"   # fp32
    # chunk 16, bf16: the 16-token tensor-core path (d_k, d_v multiples of 16)
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(128, 128, 16, 1)] == "chunk16_tc"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(48, 16, 16, 1)] == "chunk16_tc"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(40, 64, 16, 1)] == "recurrent"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(128, 128, 16, 0)] == "recurrent"   # fp32
    assert L.kda_chunk_prefill_workspace_size(1, 1, 4096, 8, 128, 128, 16, 1) == 1024
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(128, 128, 64, 1)] == "chunked_tc"
    # narrower bf16 heads: d_k a multiple of 16, d_v a multiple of 32
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(64, 64, 64, 1)] == "chunked_tc"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(16, 32, 64, 1)] == "chunked_tc"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(48, 64, 64, 1)] == "chunked_tc"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(40, 64, 64, 1)] == "recurrent"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(64, 48, 64, 1)] == "recurrent"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(8, 32, 64, 1)] == "recurrent"
    assert api.PATH_NAMES[L.kda_chunk_prefill_path(144, 128, 64, 1)] == "recurrent"


def test_gate_rejects_bad_arguments(L):
    assert L.kda_gate(None, _fake(), _fake(), 4, 2, 16, 0, None) == INVALID
    assert L.kda_gate(_fake(), _fake(), _fake(0x10004), 4, 2, 16, 0, None) == INVALID
    assert L.kda_gate(_fake(), _fake(), _fake(), -1, 2, 16, 0, None) == INVALID
    assert L.kda_gate(_fake(), _fake(), _fake(), 4, 2, 16, 5, None) == INVALID
    assert L.kda_gate(None, None, None, 0, 2, 16, 0, None) == 0           # empty: no launch


def test_decode_rejects_bad_arguments(L):
    f = _fake()
    assert L.kda_decode_step(None, f, f, f, f, f, f, f, 4, 2, 128, 128, 1, None) == INVALID
    assert L.kda_decode_step(f, f, f, f, f, f, _fake(0x10004), f, 4, 2, 128, 128, 1,
                             None) == INVALID
    assert L.kda_decode_step(f, f, f, f, f, f, f, f, 4, 2, 256, 128, 1, None) == UNSUPPORTED
    assert L.kda_decode_step(f, f, f, f, f, f, f, f, 4, 2, 128, 126, 1, None) == UNSUPPORTED
    assert L.kda_decode_step(f, f, f, f, f, f, f, f, -1, 2, 128, 128, 1, None) == INVALID
    assert L.kda_decode_step(None, None, None, None, None, None, None, None, 0, 2, 128, 128, 1,
                             None) == 0                                     # empty: no launch


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_LIB", None)
    monkeypatch.setattr(api, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        api.lib()


def test_spec_rejects_bad_arguments(L):
    f = _fake()
    assert L.kda_spec_verify(f, f, f, f, f, f, f, f, 2, 17, 2, 128, 128, 1, None) == UNSUPPORTED
    assert L.kda_spec_verify(f, f, f, f, f, f, f, f, 2, 0, 2, 128, 128, 1, None) == INVALID
    assert L.kda_spec_verify(None, f, f, f, f, f, f, f, 2, 4, 2, 128, 128, 1, None) == INVALID
    assert L.kda_spec_verify(f, f, f, f, f, f, f, f, 2, 4, 2, 256, 128, 1, None) == UNSUPPORTED
    assert L.kda_spec_commit(f, f, f, f, f, f, None, 2, 4, 2, 128, 128, 1, None) == INVALID
    assert L.kda_spec_commit(f, f, f, f, f, f, _fake(0x10002), 2, 4, 2, 128, 128, 1,
                             None) == INVALID
    assert L.kda_spec_commit(None, None, None, None, None, None, None, 0, 4, 2, 128, 128, 1,
                             None) == 0                                   # empty: no launch


def test_from_host_rejects_bad_arguments(L):
    f = _fake()
    s1, s2, s3 = ctypes.c_void_p(1), ctypes.c_void_p(2), ctypes.c_void_p(3)

    def call(**kw):
        a = dict(d=128, dtype=1, seg=1024, st=(s1, s2, s3), S1=f)
        a.update(kw)
        return L.kda_chunk_prefill_from_host(f, f, f, f, f, f, f, f, f, f, f, f, f, None, a["S1"],
                                             1, 4096, 2, a["d"], a["d"], a["dtype"], a["seg"], f,
                                             1 << 30, *a["st"])
    assert call(dtype=0) == UNSUPPORTED                       # fp32: not the tensor-core path
    assert call(d=40) == UNSUPPORTED                          # d_k not a multiple of 16
    assert call(seg=100) == INVALID                           # not a multiple of 64
    assert call(seg=0) == INVALID
    assert call(st=(s1, s1, s3)) == INVALID                   # streams must differ
    assert call(S1=None) == INVALID                           # the state carrier is required


def test_selftest_rejects_bad_status_pointer(L):
    assert L.kda_selftest_bounded_wait(None, 0, None) == INVALID
    assert L.kda_selftest_bounded_wait(_fake(0x10002), 0, None) == INVALID   # not 4-byte aligned


def test_static_workspace_status_rejects_bad_pointer(L):
    assert L.kda_static_workspace_status(None, None) == INVALID
    assert b"NULL" in L.kda_last_error()
    assert L.kda_static_workspace_status(_fake(0x10002), None) == INVALID
    assert b"aligned" in L.kda_last_error()


def test_segmented_rejects_bad_arguments(L):
    f = _fake()
    args = lambda **kw: dict(dict(B=1, T=128, H=2, dk=128, dv=128, chunk=64, dtype=1, G=2,  # noqa: E731
                                  ws=None, ws_bytes=0), **kw)

    def call(a):
        return L.kda_chunk_prefill_segmented(f, f, f, f, f, f, f, None, None, a["B"], a["T"],
                                             a["H"], a["dk"], a["dv"], a["chunk"], a["dtype"],
                                             a["G"], a["ws"], a["ws_bytes"], None)
    assert call(args(G=0)) == INVALID
    assert call(args(dtype=0)) == UNSUPPORTED           # fp32 stays on the recurrence
    assert call(args(chunk=16)) == UNSUPPORTED
    assert call(args()) == WORKSPACE                    # no workspace given
    assert L.kda_chunk_prefill_segmented_workspace_size(1, 128, 2, 128, 128, 64, 1, 0) == 0


def test_segment_policy_and_workspace(L):
    # The long-context workload (32 heads) keeps the plain pass; few heads are segmented.
    assert L.kda_chunk_prefill_auto_segments(1, 65536, 32, 128, 128, 64, 1) == 1
    assert L.kda_chunk_prefill_auto_segments(2, 4096, 8, 128, 128, 64, 1) == 1
    assert L.kda_chunk_prefill_auto_segments(1, 65536, 8, 128, 128, 64, 1) > 1
    assert L.kda_chunk_prefill_auto_segments(1, 65536, 1, 128, 128, 64, 1) > 1
    assert L.kda_chunk_prefill_auto_segments(1, 65536, 8, 128, 128, 64, 0) == 1   # fp32
    plain = L.kda_chunk_prefill_segmented_workspace_size(1, 65536, 8, 128, 128, 64, 1, 1)
    seg = L.kda_chunk_prefill_segmented_workspace_size(1, 65536, 8, 128, 128, 64, 1, 4)
    # four segments add three (pair, start state) records per head: 3 x 8 x (128 + 64) KiB
    assert seg - plain == 3 * 8 * (128 + 64) * 1024
    # segments shorter than one chunk collapse: 130 tokens make three chunks
    assert (L.kda_chunk_prefill_segmented_workspace_size(1, 130, 1, 128, 128, 64, 1, 50)
            == L.kda_chunk_prefill_segmented_workspace_size(1, 130, 1, 128, 128, 64, 1, 3))
    auto = L.kda_chunk_prefill_auto_segments(1, 65536, 8, 128, 128, 64, 1)
    assert (L.kda_chunk_prefill_workspace_size(1, 1, 65536, 8, 128, 128, 64, 1)
            == L.kda_chunk_prefill_segmented_workspace_size(1, 65536, 8, 128, 128, 64, 1, auto))
