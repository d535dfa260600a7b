"""fp64 CPU oracle for the MoE-side steps around sink attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use this
module.  The library never calls it; it shares no code with the CUDA path.

Follows the page "GPT-OSS on day 0" (Perplexity, 2025):

* the model overview list: the output projection and the experts carry bias
  terms, and the expert weights are a softmax taken after the Top-K selection;
* section "Kernels for GPT-OSS / MoE": for GPT-OSS the router takes its softmax
  over the K selected experts only (not over all experts, as DeepSeek-style
  routers do), and computing the expert weights in bfloat16 is what keeps
  accuracy;
* same section: bias support was added to the expert GEMMs by starting the
  accumulator from the bias values, once per output (MN) tile.

Readings taken where the page is silent (each is also listed in the design notes):

R1. "expert weights in bfloat16": the router logits are bf16 values (the
    projection output is rounded to bf16 before anything is decided), the
    Top-K decision is taken on those bf16 values, the softmax over the K
    selected logits is exact here (fp64) and the stored weights are bf16;
R2. Top-K order: largest logit first; equal logits keep the lower expert index
    first (this also decides which of several equal logits is selected);
R3. a bias-seeded linear layer computes ``out = x W^T + b`` with the bias
    entering once per output element, exactly as if added after the sum;
R4. expert token counts (for dispatch) count every (token, selected expert)
    pair once.

Every number is fp64; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import numpy as np

from . import widen_bf16

__all__ = ["round_to_bf16", "linear_bias", "topk_indices", "router_topk_softmax",
           "expert_counts", "router"]


def round_to_bf16(x) -> np.ndarray:
    """fp64 values rounded to the nearest bf16 value (ties to even), returned as fp64.

    The rounding is taken on the fp64 value itself (no intermediate fp32, which
    would round twice): bf16 keeps 8 significant bits, and below the smallest
    normal number (2^-126) a fixed quantum of 2^-133.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x) & (x != 0.0)
    xs = np.where(finite, x, 1.0)
    _, e = np.frexp(xs)                       # |x| in [2^(e-1), 2^e)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    n = xs / q                                # exact: q is a power of two
    r = np.floor(n)
    frac = n - r
    r = r + ((frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2.0) == 1.0)))
    y = r * q
    y = np.where(np.abs(y) > 3.3895313892515355e38, np.copysign(np.inf, xs), y)
    return np.where(finite, y, x)


def bf16_bits(x) -> np.ndarray:
    """fp64 values that are exactly bf16 -> their uint16 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x, equal_nan=True):
        raise ValueError("values are not representable in fp32")
    bits = f.view(np.uint32)
    if np.any(bits & 0xFFFF):
        raise ValueError("values are not representable in bf16")
    return (bits >> 16).astype(np.uint16)


def linear_bias(x, w, bias) -> np.ndarray:
    """``out[m, n] = sum_k x[m, k] w[n, k] + bias[n]`` in fp64 (reading R3).

    x: [M, K], w: [N, K] (one row per output feature), bias: [N]; all bf16 bit
    patterns (uint16) or float arrays.
    """
    x = _f64(x)
    w = _f64(w)
    b = _f64(bias)
    return x @ w.T + b[None, :]


def topk_indices(row, k: int) -> np.ndarray:
    """Indices of the k largest values of one row, largest first, lower index first
    among equal values (reading R2): k rounds of "take the largest remaining"."""
    row = np.asarray(row, dtype=np.float64)
    taken = np.zeros(row.shape[0], dtype=bool)
    out = []
    for _ in range(k):
        best = -1
        for e in range(row.shape[0]):
            if taken[e]:
                continue
            if best < 0 or row[e] > row[best]:
                best = e
        taken[best] = True
        out.append(best)
    return np.array(out, dtype=np.int32)


def router_topk_softmax(logits, k: int):
    """Top-K then softmax over the K selected logits (section "Kernels for GPT-OSS / MoE").

    logits: [T, E] bf16 bit patterns (uint16) or fp64 values already on the bf16
    grid.  Returns (indices int32 [T, k], weights fp64 [T, k]); the weights are
    exact softmax values of the selected logits (the library stores them as bf16).
    """
    x = _f64(logits)
    t, e = x.shape
    if not 1 <= k <= e:
        raise ValueError("need 1 <= k <= num_experts")
    idx = np.zeros((t, k), dtype=np.int32)
    wts = np.zeros((t, k), dtype=np.float64)
    for i in range(t):
        sel = topk_indices(x[i], k)
        v = x[i, sel]
        mx = v.max()
        p = np.exp(v - mx)
        idx[i] = sel
        wts[i] = p / p.sum()
    return idx, wts


def expert_counts(indices, num_experts: int) -> np.ndarray:
    """Tokens routed to each expert (reading R4)."""
    c = np.zeros(num_experts, dtype=np.int64)
    for e in np.asarray(indices).ravel():
        c[int(e)] += 1
    return c


def router(x, w, bias, k: int):
    """Router projection with bias, rounded to bf16 (reading R1), then Top-K softmax.

    Returns (indices, weights, logits) with logits the bf16-rounded fp64 values.
    """
    logits = round_to_bf16(linear_bias(x, w, bias))
    idx, wts = router_topk_softmax(logits, k)
    return idx, wts, logits


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return widen_bf16(a)
    return a.astype(np.float64)
