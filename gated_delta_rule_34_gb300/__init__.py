"""GB300 (sm_103a) Kimi Delta Attention layer: a C-ABI CUDA library plus a thin binding.

    from gated_delta_rule_34_gb300 import chunk_prefill, decode_step, gate

The binding loads ``_build/libkda.so`` on first use (build it with
``python -m gated_delta_rule_34_gb300.build``); importing the package loads
nothing, so the seeded input generator (``.inputs``) can be used without a GPU.
"""
from .api import (KDAError, auto_segments, chunk_prefill, chunk_prefill_from_host,  # noqa: F401
                  chunk_prefill_segmented, chunk_prefill_static_workspace, decode_step, gate, lib, library_path,
                  prefill_path, selftest_bounded_wait, set_profile_events, spec_commit,
                  segmented_workspace_size, spec_verify, static_workspace_status,
                  workspace_size)

__all__ = ["KDAError", "auto_segments", "chunk_prefill", "chunk_prefill_segmented",
           "segmented_workspace_size", "chunk_prefill_from_host", "chunk_prefill_static_workspace",
           "decode_step", "gate", "lib", "library_path", "prefill_path", "selftest_bounded_wait",
           "set_profile_events", "spec_commit", "spec_verify", "static_workspace_status",
           "workspace_size"]
