"""Helpers shared by the GPU parity tests: tolerance and error metric.

Error metric (the paper gives none; this is the reading used throughout): per
(b, h) slice, max_{t,j} |o - o_ref| / max_{t,j} |o_ref|; the reported error is
the maximum over slices.  The bar is 1e-4 for fp32 inputs and 2e-2 for bf16
inputs with fp32 accumulation.  Beside it the tests report the element-wise
max |o - o_ref| / (|o_ref| + 1e-3 max|o_ref|) (elem_rel_err), which is not a
gate.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact decode of the stored values (bf16 -> fp32 -> fp64 is exact)."""
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def slice_rel_err(o: np.ndarray, ref: np.ndarray) -> float:
    """o, ref: [..., T, dv] with leading slice axes, or [rows, dv] for one slice."""
    o = o.reshape(-1, o.shape[-2], o.shape[-1]) if o.ndim > 2 else o[None]
    ref = ref.reshape(o.shape)
    worst = 0.0
    for a, b in zip(o, ref):
        scale = np.max(np.abs(b))
        err = np.max(np.abs(a - b)) / scale if scale > 0 else np.max(np.abs(a))
        worst = max(worst, float(err))
    return worst


def elem_rel_err(o: np.ndarray, ref: np.ndarray) -> float:
    """Element-wise metric reported beside the slice metric (not a gate): per
    slice max_{t,j} |o - o_ref| / (|o_ref| + 1e-3 max|o_ref|), maximum over
    slices.  It exposes a large relative error on a small-magnitude output that
    the slice metric would average away."""
    o = o.reshape(-1, o.shape[-2], o.shape[-1]) if o.ndim > 2 else o[None]
    ref = ref.reshape(o.shape)
    worst = 0.0
    for a, b in zip(o, ref):
        floor = 1e-3 * np.max(np.abs(b))
        if floor == 0:
            continue
        worst = max(worst, float(np.max(np.abs(a - b) / (np.abs(b) + floor))))
    return worst


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import kernelized_causal_linear_gb300 as kg
    from kernelized_causal_linear_gb300 import build
    build.build()
    return kg
