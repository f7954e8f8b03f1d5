"""Plants plausible slips in a copy of the oracle and checks that the pins catch each.

The original oracle source is never modified: each mutant is a textual edit of
a temporary copy, compiled into its own library and swapped in for the
duration of one test.
"""
import os
import subprocess

import pytest
import torch

import oracle
from oracle import build as obuild
import tests.test_oracle_pins as pins

MUTANTS = {
    "no decay": ("D[c * dv + j] = alpha[c] * S[c * dv + j];", "D[c * dv + j] = S[c * dv + j];"),
    "erase sign": ("- b * kv[c] * kD[j]", "+ b * kv[c] * kD[j]"),
    "erase reads undecayed state": ("acc += kv[c] * D[c * dv + j];", "acc += kv[c] * S[c * dv + j];"),
    "output before update": ("acc += S[c * dv + j] * qv[c];", "acc += D[c * dv + j] * qv[c];"),
    "transposed state read": ("acc += S[c * dv + j] * qv[c];", "acc += S[(j * dv + c) % (dk * dv)] * qv[c];"),
    "write without beta": ("+ b * kv[c] * vv[j];", "+ kv[c] * vv[j];"),
    "gate complement": ("return KDA_REF_GMIN * sig;", "return KDA_REF_GMIN * (1.0 - sig);"),
    "gate without exp(A)": ("double x = exp(a) * z;", "double x = a * z;"),
    "A ignores head": ("(double)J->A[h * dk + c]", "(double)J->A[c]"),
    "beta from wrong head": ("ref_load(J->beta, row, J->dtype)", "ref_load(J->beta, t, J->dtype)"),
    "query is key": ("qv[c] = ref_load(J->q,", "qv[c] = ref_load(J->k,"),
}


def _pin_suite():
    """Returns the names of pins that fail against the currently loaded oracle."""
    checks = {
        "gate golden": pins.test_gate_golden_points,
        "gate indexing": pins.test_gate_array_matches_scalar_and_indexing,
        "hand no decay": pins.test_hand_example_no_decay,
        "hand channel decay": pins.test_hand_example_channel_decay,
        "closed form T3": lambda: pins.test_closed_form_three_tokens(0, torch.float32),
        "beta 0 keeps state": pins.test_beta_zero_no_decay_keeps_state,
        "beta 0 decay": pins.test_beta_zero_pure_decay_closed_form,
        "orthonormal recall": lambda: pins.test_orthonormal_keys_recall_values(4),
        "chunked agreement": lambda: pins.test_chunked_form_matches_recurrence(16),
    }
    failed = []
    for name, fn in checks.items():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def _build_variant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-ffp-contract=off", "-o", str(lib), str(path), "-lm"], check=True)
    return str(lib)


def test_unmutated_oracle_passes_every_pin():
    assert _pin_suite() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    lib = oracle.load_library(_build_variant(tmp_path, old, new))
    monkeypatch.setattr(oracle, "_LIB", lib)
    failed = _pin_suite()
    assert failed, f"mutant '{name}' passed every pin"
