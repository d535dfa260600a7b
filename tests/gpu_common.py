"""Helpers shared by the GPU parity tests (host-side marshalling only)."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

# Tolerances against the fp64 oracle: 1e-2 max-abs on the attention output and
# 1e-3 on the fp32 log-sum-exp.  A bf16 output is the round-to-nearest-even of
# the kernel's fp32 result, so what the 1e-2 budget can be checked against is
# the set of reals that round to the stored value: the interval between the
# midpoints to its two bf16 neighbours.  A stored value passes when that
# interval comes within 1e-2 of the fp64 oracle, i.e. when some pre-rounding
# value at most 1e-2 from the oracle stores as exactly this bf16 number.
# Equivalently (bf16 rounding is monotone):
#     round_bf16(oracle - 1e-2) <= stored <= round_bf16(oracle + 1e-2).
# This removes the storage rounding exactly.  Comparing the stored value with
# round_bf16(oracle) at 1e-2 would instead reject any value within 1e-2 of the
# oracle that lies on the other side of a rounding midpoint wherever a bf16 step
# exceeds 1e-2 (|out| >= 2), however small the arithmetic error.
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


def oracle_workers():
    """Threads for the oracle's independent (sequence, head) units: the host's cores."""
    return max(1, os.cpu_count() or 1)


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


def _bf16_neighbours(g):
    """The next bf16 values below and above each bf16 value g (float64 in, float64 out)."""
    bits = (np.asarray(g, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
    neg = (bits & 0x8000) != 0
    zero = (bits & 0x7FFF) == 0
    up = np.where(neg, bits - 1, bits + 1)
    down = np.where(neg, bits + 1, bits - 1)
    up = np.where(zero, 0x0001, up)          # +-0: the neighbours are +-2^-133
    down = np.where(zero, 0x8001, down)

    def widen(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return widen(down), widen(up)


def bf16_store_excess(out, ref):
    """Per element: the distance from the fp64 oracle value to the interval of reals
    that round to the stored bf16 value (0 where the oracle lies inside it)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    down, up = _bf16_neighbours(out)
    lo = 0.5 * (out + down)
    hi = 0.5 * (out + up)
    return np.maximum(0.0, np.maximum(lo - ref, ref - hi))


def out_err_beyond_bf16_store(out, ref):
    """Largest ``bf16_store_excess`` over the elements; NaN if any stored value is
    not finite or any oracle value is NaN."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    if not np.isfinite(out).all() or np.isnan(ref).any():
        return float("nan")
    if out.size == 0:
        return 0.0
    return float(bf16_store_excess(out, ref).max())


def out_err_vs_rounded_oracle(out, ref):
    """max |stored - round_bf16(oracle)|, for the log line only."""
    from oracle.moe import round_to_bf16
    out = np.asarray(out, dtype=np.float64)
    return float(np.abs(out - round_to_bf16(ref)).max()) if out.size else 0.0


def assert_close(out, lse, ref_o, ref_l, what, bf16_out=True):
    raw = max_err(out, ref_o)
    eo = out_err_beyond_bf16_store(out, ref_o) if bf16_out else raw
    el = max_err(lse, ref_l) if lse is not None else 0.0
    if bf16_out:
        rr = out_err_vs_rounded_oracle(out, ref_o)
        print(f"ERR {what}: out raw {raw:.3e} beyond-store {eo:.3e} vs-rounded {rr:.3e} lse {el:.3e}")
    else:
        print(f"ERR {what}: out {raw:.3e} lse {el:.3e}")
    assert eo <= OUT_TOL, f"{what}: out error {eo} beyond bf16 storage (raw {raw}) > {OUT_TOL}"
    assert el <= LSE_TOL, f"{what}: lse max-abs error {el} > {LSE_TOL}"
    return eo, el
