"""Helpers shared by the GPU parity tests (no arithmetic of the method)."""
from __future__ import annotations

import numpy as np
import pytest

TOL = 1e-5   # max|gpu - oracle| / max|oracle| per output tensor (f32 accumulate)


def cuda_or_skip():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_fmt1_gb300 as coli  # noqa: F401  (raises if the library is missing)
    return torch


def norm_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def upload(coli, m):
    return coli.tensor_upload(m.fmt, m.gs, m.O, m.I, m.data, m.scales)
