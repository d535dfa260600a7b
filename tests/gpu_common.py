"""Helpers shared by the GPU parity tests (host-side marshalling only)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

# Tolerances against the fp64 oracle: 1e-2 max-abs on the attention output and
# 1e-3 on the fp32 log-sum-exp.  A bf16 output is additionally rounded to the
# nearest bf16 when stored, which alone can move it by half an ulp, i.e. up to
# 2^-8 of its magnitude (0.0156 at |out| >= 4); that storage rounding is
# allowed on top of the 1e-2 budget (BF16_STORE_REL), nothing else is.
OUT_TOL = 1e-2
LSE_TOL = 1e-3
BF16_STORE_REL = 2.0 ** -8


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


def out_err_beyond_bf16_store(out, ref):
    """Max over elements of |out - ref| minus the bf16 storage rounding allowance."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    if not np.isfinite(out).all():
        return float("nan")
    excess = np.abs(out - ref) - BF16_STORE_REL * np.maximum(np.abs(out), np.abs(ref))
    return float(excess.max()) if excess.size else 0.0


def assert_close(out, lse, ref_o, ref_l, what, bf16_out=True):
    raw = max_err(out, ref_o)
    eo = out_err_beyond_bf16_store(out, ref_o) if bf16_out else raw
    el = max_err(lse, ref_l) if lse is not None else 0.0
    print(f"ERR {what}: out raw {raw:.3e} beyond-store {eo:.3e} lse {el:.3e}")
    assert eo <= OUT_TOL, f"{what}: out error {eo} (raw {raw}) > {OUT_TOL}"
    assert el <= LSE_TOL, f"{what}: lse max-abs error {el} > {LSE_TOL}"
    return eo, el
