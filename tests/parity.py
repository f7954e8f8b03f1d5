"""Shared helpers of the GPU parity tests (comparisons against the fp64 oracle)."""
import numpy as np
import pytest
import torch

# Bound on max |gpu - oracle| relative to max |oracle| over a whole tensor: 1e-4 for
# fp32 inputs and 2e-2 for bf16 inputs (the layer's stated parity tolerances).
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(got, ref) -> float:
    got = np.asarray(got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else got,
                     dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    scale = np.abs(ref).max() if ref.size else 0.0
    if scale == 0:
        return float(np.abs(got).max()) if got.size else 0.0
    return float(np.abs(got - ref).max() / scale)


def report(what: str, err: float, tol: float, extra: str = "") -> None:
    """Prints one margin line (visible with pytest -s): the measured relative error,
    the bound it is held to, and their ratio."""
    print(f"PARITY {what}: rel_err={err:.3e} tol={tol:.1e} used={err / tol:.1%}{extra}")


def assert_parity(got, ref, dtype, what="", tol=None):
    tol = TOL[dtype] if tol is None else tol
    e = rel_err(got, ref)
    report(what, e, tol)
    assert e <= tol, f"{what}: max|gpu-oracle|/max|oracle| = {e:.3e} > {tol:.1e}"
    return e


def cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")
