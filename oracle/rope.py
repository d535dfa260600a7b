"""fp64 CPU oracle for the step that feeds sink attention: QKV bias, YaRN rotary
position encoding and the paged KV-cache append.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use this
module.  The library never calls it; it shares no code with the CUDA path.

The page "GPT-OSS on day 0" (Perplexity, 2025), model overview list, states that
the QKV projections carry biases (as in Qwen 2) and that positions are encoded
with YaRN (as in DeepSeek-V3).  It gives no constants or formulas, so this module
follows the YaRN paper (Peng, Quesnelle, Fan, Shippole, "YaRN: Efficient Context
Window Extension of Large Language Models", 2023), section 3:

* rotary encoding rotates each pair of a head's features by the angle
  ``p * theta_i`` (position p), ``theta_i = base^(-2 i / D)``, i < D/2;
* "NTK-by-parts": frequencies that turn many times over the original context
  length L keep ``theta_i`` (extrapolation), those that turn less than once are
  divided by the scale factor s (interpolation), with a linear ramp between;
* the attention temperature is applied by multiplying the rotation (cos and
  sin, for q and k alike) by ``0.1 ln(s) + 1``.

Readings taken where the pages are silent (each is also listed in the design notes):

Y1. the ramp is linear in the feature-pair index i between the two (fractional)
    indices at which the number of rotations over L equals beta_fast and
    beta_slow: ``c(n) = (D/2) ln(L / (2 pi n)) / ln(base)``,
    ``rho(i) = clamp((i - c(beta_fast)) / (c(beta_slow) - c(beta_fast)), 0, 1)``,
    ``theta'_i = theta_i (1 - rho(i)) + (theta_i / s) rho(i)``; the boundaries
    are not rounded to whole indices;
Y2. pairs are (x_i, x_{i + D/2}) ("half split"), rotated as the complex number
    ``(x_i + j x_{i+D/2}) e^{j p theta'_i}``;
Y3. the position of new token t of a sequence with q_len new tokens and a cache
    of kv_len tokens (the new ones included) is ``kv_len - q_len + t`` (the same
    bottom-right alignment as the causal mask);
Y4. the QKV projection output is laid out [T, (Hq + 2 Hkv) * D]: all query heads,
    then all key heads, then all value heads; the bias has the same layout and is
    added before the rotation; values are not rotated;
Y5. the appended K/V of token t lands in page ``page_table[b, pos // page_size]``,
    row ``pos % page_size`` of the paged cache ``[num_pages, Hkv, page_size, D]``.

Every number is fp64; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import math

import numpy as np

from . import widen_bf16

__all__ = ["rope_inv_freq", "yarn_correction_index", "yarn_inv_freq", "yarn_mscale", "rope_rotate",
           "token_positions", "qkv_bias_rope", "append_paged_kv"]


def rope_inv_freq(head_dim: int, base: float) -> np.ndarray:
    """Plain rotary frequencies ``theta_i = base^(-2 i / D)``, i < D/2."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return base ** (-2.0 * i / head_dim)


def yarn_correction_index(num_rotations: float, head_dim: int, base: float, orig_len: int) -> float:
    """Fractional pair index at which a frequency turns ``num_rotations`` times over
    ``orig_len`` positions (reading Y1)."""
    return (head_dim / 2.0) * math.log(orig_len / (2.0 * math.pi * num_rotations)) / math.log(base)


def yarn_inv_freq(head_dim: int, base: float, factor: float, orig_len: int,
                  beta_fast: float, beta_slow: float) -> np.ndarray:
    """YaRN frequencies ``theta'_i`` (paper section 3, "NTK-by-parts"; reading Y1)."""
    theta = rope_inv_freq(head_dim, base)
    if factor == 1.0:
        return theta
    lo = yarn_correction_index(beta_fast, head_dim, base, orig_len)
    hi = yarn_correction_index(beta_slow, head_dim, base, orig_len)
    i = np.arange(head_dim // 2, dtype=np.float64)
    rho = np.clip((i - lo) / (hi - lo), 0.0, 1.0)
    return theta * (1.0 - rho) + (theta / factor) * rho


def yarn_mscale(factor: float) -> float:
    """Attention-temperature factor on cos and sin (paper: sqrt(1/t) = 0.1 ln s + 1)."""
    return 1.0 if factor <= 1.0 else 0.1 * math.log(factor) + 1.0


def rope_rotate(x, positions, inv_freq, mscale: float = 1.0) -> np.ndarray:
    """Rotate the feature pairs (x_i, x_{i+D/2}) of x [N, H, D] by ``positions[n] * inv_freq[i]``
    and scale by mscale (reading Y2)."""
    x = np.asarray(x, dtype=np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(inv_freq)[None, :]
    c = (mscale * np.cos(ang))[:, None, :]
    s = (mscale * np.sin(ang))[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def token_positions(cu_seqlens_q, kv_lens=None) -> np.ndarray:
    """Position of every new token (reading Y3); kv_lens None means kv_len == q_len."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for b in range(len(cu) - 1):
        q_len = int(cu[b + 1] - cu[b])
        kv = q_len if kv_lens is None else int(kv_lens[b])
        pos[cu[b]:cu[b + 1]] = np.arange(kv - q_len, kv)
    return pos


def qkv_bias_rope(qkv, bias, cu_seqlens_q, kv_lens, num_qo_heads: int, num_kv_heads: int,
                  head_dim: int, inv_freq, mscale: float):
    """Bias add, then rotary encoding of q and k; returns exact (q, k, v) as fp64
    [T, H, D] arrays (readings Y3, Y4).  bias may be None."""
    x = _f64(qkv)
    t = x.shape[0]
    if bias is not None:
        x = x + _f64(bias)[None, :]
    hq, hkv, d = num_qo_heads, num_kv_heads, head_dim
    q = x[:, :hq * d].reshape(t, hq, d)
    k = x[:, hq * d:(hq + hkv) * d].reshape(t, hkv, d)
    v = x[:, (hq + hkv) * d:].reshape(t, hkv, d)
    pos = token_positions(cu_seqlens_q, kv_lens)
    return rope_rotate(q, pos, inv_freq, mscale), rope_rotate(k, pos, inv_freq, mscale), v.copy()


def append_paged_kv(k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, k_new, v_new):
    """The cache after writing every new token's K and V at its position (readings
    Y3, Y5).  Returns fp64 copies of the page arrays."""
    kp = _f64(k_pages).copy()
    vp = _f64(v_pages).copy()
    page_size = kp.shape[2]
    pos = token_positions(cu_seqlens_q, kv_lens)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    for b in range(len(cu) - 1):
        for t in range(int(cu[b]), int(cu[b + 1])):
            page = int(page_table[b][pos[t] // page_size])
            kp[page, :, pos[t] % page_size, :] = k_new[t]
            vp[page, :, pos[t] % page_size, :] = v_new[t]
    return kp, vp


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return widen_bf16(a)
    return a.astype(np.float64)
