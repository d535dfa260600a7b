"""Helpers shared by the GPU parity tests (host-side marshalling only)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

# Tolerances for bf16 inputs with fp32 accumulation against the fp64 oracle.
OUT_TOL = 1e-2
LSE_TOL = 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_softmax_sinks_gb300 as sa
    from attention_softmax_sinks_gb300 import _build
    _build.build()
    sa.load_library()
    return sa


def bf16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev(x, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def host(t):
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy().astype(np.float64)


def max_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    if np.isnan(diff).any():
        return float("nan")
    return float(diff.max()) if diff.size else 0.0


def assert_close(out, lse, ref_o, ref_l, what):
    eo = max_err(out, ref_o)
    el = max_err(lse, ref_l) if lse is not None else 0.0
    assert eo <= OUT_TOL, f"{what}: out max-abs error {eo} > {OUT_TOL}"
    assert el <= LSE_TOL, f"{what}: lse max-abs error {el} > {LSE_TOL}"
    return eo, el
