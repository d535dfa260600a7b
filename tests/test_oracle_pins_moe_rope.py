"""The MoE-router, bias-linear and YaRN/QKV oracles against their pins, and
plausible mistakes planted in them (CPU only)."""
import math

import numpy as np
import pytest

from oracle import moe, rope
import oracle_pins_moe_rope as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


_router = moe.router_topk_softmax
_linear = moe.linear_bias
_topk = moe.topk_indices
_inv = rope.yarn_inv_freq
_rot = rope.rope_rotate
_pos = rope.token_positions
_qkv = rope.qkv_bias_rope


def _softmax_over_all_experts(logits, k):
    idx, _ = _router(logits, k)
    x = moe._f64(logits)
    p = np.exp(x - x.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return idx, np.take_along_axis(p, idx.astype(np.int64), axis=1)


def _ties_to_higher_index(row, k):
    row = np.asarray(row, dtype=np.float64)
    rev = _topk(row[::-1], k)
    return (len(row) - 1 - rev).astype(np.int32)


def _no_bf16_rounding(x, w, bias, k):
    logits = _linear(x, w, bias)
    idx, wts = _router(logits, k)
    return idx, wts, logits


def _truncating_bf16(x):
    x = np.asarray(x, dtype=np.float64).astype(np.float32)
    return ((x.view(np.uint32) >> 16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _transposed_weight(x, w, bias):
    # W read as [K, N] row-major instead of [N, K]
    w = moe._f64(w)
    return moe._f64(x) @ w.reshape(w.shape[1], w.shape[0]) + moe._f64(bias)[None, :]


def _bias_dropped(x, w, bias):
    return moe._f64(x) @ moe._f64(w).T


def _interleaved_pairs(x, positions, inv_freq, mscale=1.0):
    x = np.asarray(x, dtype=np.float64)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(inv_freq)[None, :]
    c = (mscale * np.cos(ang))[:, None, :]
    s = (mscale * np.sin(ang))[:, None, :]
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def _rotation_reversed(x, positions, inv_freq, mscale=1.0):
    return _rot(x, -np.asarray(positions, dtype=np.float64), inv_freq, mscale)


def _ramp_reversed(head_dim, base, factor, orig_len, beta_fast, beta_slow):
    return _inv(head_dim, base, factor, orig_len, beta_slow, beta_fast)


def _ln_ramp(head_dim, base, factor, orig_len, beta_fast, beta_slow):
    # ramp taken linearly in the number of rotations instead of the pair index
    theta = base ** (-np.arange(head_dim // 2) * 2.0 / head_dim)
    if factor == 1.0:
        return theta
    turns = orig_len * theta / (2 * math.pi)
    rho = np.clip((beta_fast - turns) / (beta_fast - beta_slow), 0.0, 1.0)
    return theta * (1 - rho) + theta / factor * rho


def _mscale_missing(factor):
    return 1.0


def _top_left_positions(cu_seqlens_q, kv_lens=None):
    return _pos(cu_seqlens_q, None)


def _values_rotated(qkv, bias, cu, kv, hq, hkv, d, inv, ms):
    q, k, v = _qkv(qkv, bias, cu, kv, hq, hkv, d, inv, ms)
    return q, k, rope.rope_rotate(v, rope.token_positions(cu, kv), inv, ms)


def _k_and_v_swapped(qkv, bias, cu, kv, hq, hkv, d, inv, ms):
    q, k, v = _qkv(qkv, bias, cu, kv, hq, hkv, d, inv, ms)
    return q, v, k


MUTANTS = {
    "softmax_over_all_experts": (moe, "router_topk_softmax", _softmax_over_all_experts),
    "ties_to_higher_index": (moe, "topk_indices", _ties_to_higher_index),
    "router_without_bf16_rounding": (moe, "router", _no_bf16_rounding),
    "bf16_truncation": (moe, "round_to_bf16", _truncating_bf16),
    "transposed_weight": (moe, "linear_bias", _transposed_weight),
    "bias_dropped": (moe, "linear_bias", _bias_dropped),
    "interleaved_rope_pairs": (rope, "rope_rotate", _interleaved_pairs),
    "rotation_reversed": (rope, "rope_rotate", _rotation_reversed),
    "yarn_ramp_reversed": (rope, "yarn_inv_freq", _ramp_reversed),
    "yarn_ramp_in_rotations": (rope, "yarn_inv_freq", _ln_ramp),
    "mscale_missing": (rope, "yarn_mscale", _mscale_missing),
    "top_left_positions": (rope, "token_positions", _top_left_positions),
    "values_rotated": (rope, "qkv_bias_rope", _values_rotated),
    "k_and_v_swapped": (rope, "qkv_bias_rope", _k_and_v_swapped),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    mod, attr, fn = MUTANTS[name]
    monkeypatch.setattr(mod, attr, fn)
    assert pins.failing_pins(), f"no pin catches the planted mistake {name}"


def test_pins_pass_unmutated():
    assert pins.failing_pins() == []
