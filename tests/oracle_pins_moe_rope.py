"""Pins that tie the MoE-router, bias-linear and YaRN/QKV oracles to facts outside
themselves: library routines on special cases (stable sort, argmax, softmax,
logistic, bincount, complex rotation, torch's linear and bf16 conversion),
closed forms worked by hand, and invariants of the definitions (rotary
relative-position property, ramp boundaries of YaRN's "NTK-by-parts").

Sources: the page "GPT-OSS on day 0" (model overview list; section "Kernels for
GPT-OSS / MoE") and the YaRN paper (Peng et al., 2023, section 3).

Functions look the oracle up at call time (``moe.<name>``, ``rope.<name>``) so
that the mutation tests can plant a mistake and check that a pin catches it.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

from oracle import moe, rope


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err} > {tol}"


def _bf16_grid(rng, shape, std=1.0):
    """Random fp64 values on the bf16 grid (rounded with the integer RNE trick on fp32)."""
    f = (rng.standard_normal(shape) * std).astype(np.float32)
    u = f.view(np.uint32)
    bits = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ bf16 rounding
def pin_round_to_bf16():
    rng = np.random.default_rng(11)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    u = f.view(np.uint32)
    ref = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32) << 16).view(np.float32)
    _close(moe.round_to_bf16(f.astype(np.float64)), ref.astype(np.float64), 0.0, "bf16 RNE vs integer trick")
    t = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    _close(moe.round_to_bf16(f.astype(np.float64)), t, 0.0, "bf16 RNE vs torch conversion")
    # ties go to the even neighbour: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    _close(moe.round_to_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)])),
           [1.0, 1 + 2 ** -6, -1.0], 0.0, "bf16 ties")


# ------------------------------------------------------------------ router
def pin_topk_is_stable_descending_sort():
    rng = np.random.default_rng(12)
    for e, k in ((32, 4), (128, 4), (7, 7), (5, 1)):
        x = rng.integers(-3, 4, (50, e)).astype(np.float64)      # many equal values
        for row in x:
            ref = np.argsort(-row, kind="stable")[:k]
            assert np.array_equal(moe.topk_indices(row, k), ref), "top-k order vs stable sort"


def pin_router_k1_is_argmax():
    rng = np.random.default_rng(13)
    x = rng.integers(-2, 3, (40, 32)).astype(np.float64)
    idx, w = moe.router_topk_softmax(x, 1)
    assert np.array_equal(idx[:, 0], np.argmax(x, axis=1)), "k=1 vs argmax (first maximum)"
    _close(w, np.ones((40, 1)), 0.0, "k=1 weight")


def pin_router_all_experts_is_softmax():
    rng = np.random.default_rng(14)
    x = _bf16_grid(rng, (20, 16), 3.0)
    idx, w = moe.router_topk_softmax(x, 16)
    full = scipy.special.softmax(x, axis=1)
    _close(w, np.take_along_axis(full, idx.astype(np.int64), axis=1), 1e-15, "k=E vs softmax")


def pin_router_renormalises_selected():
    """Softmax over the selected logits = full softmax restricted and renormalised,
    which differs from taking the full softmax's values (the all-experts variant)."""
    rng = np.random.default_rng(15)
    x = _bf16_grid(rng, (30, 128), 2.0)
    idx, w = moe.router_topk_softmax(x, 4)
    full = scipy.special.softmax(x, axis=1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    _close(w, sel / sel.sum(axis=1, keepdims=True), 1e-15, "renormalised softmax")
    _close(w.sum(axis=1), np.ones(30), 1e-15, "weights sum to one")
    assert np.max(np.abs(w - sel)) > 1e-3


def pin_router_equal_and_two_expert_closed_forms():
    idx, w = moe.router_topk_softmax(np.zeros((3, 8)), 4)
    assert np.array_equal(idx, np.tile(np.arange(4, dtype=np.int32), (3, 1))), "ties: lower index first"
    _close(w, np.full((3, 4), 0.25), 0.0, "equal logits")
    x = np.array([[0.5, -1.25, 2.0, 0.0]])
    idx, w = moe.router_topk_softmax(x, 2)
    assert idx.tolist() == [[2, 0]]
    _close(w[0], [scipy.special.expit(1.5), scipy.special.expit(-1.5)], 1e-15, "two-expert logistic")


def pin_router_decides_on_bf16_logits():
    """Two projections that differ below bf16 resolution round to one bf16 logit, so
    the lower expert index wins although its unrounded logit is smaller."""
    x = np.array([[1.0]])
    w = np.array([[1.0], [1.0], [0.0]])
    bias = np.array([0.0, 2 ** -10, 0.5])
    idx, wts, logits = moe.router(x, w, bias, 1)
    _close(logits, [[1.0, 1.0, 0.5]], 0.0, "router logits on the bf16 grid")
    assert idx.tolist() == [[0]]


def pin_expert_counts():
    rng = np.random.default_rng(16)
    idx = rng.integers(0, 32, (100, 4))
    assert np.array_equal(moe.expert_counts(idx, 32), np.bincount(idx.ravel(), minlength=32))


# ------------------------------------------------------------------ linear with bias
def pin_linear_bias_special_cases():
    rng = np.random.default_rng(17)
    m, n, k = 5, 7, 3
    x = _bf16_grid(rng, (m, k))
    w = _bf16_grid(rng, (n, k))
    b = _bf16_grid(rng, (n,))
    # unit-vector inputs pick one column of W (catches a transposed operand)
    for j in range(k):
        e = np.zeros((1, k))
        e[0, j] = 1.0
        _close(moe.linear_bias(e, w, b)[0], w[:, j] + b, 0.0, "unit row")
    _close(moe.linear_bias(np.zeros((m, k)), w, b), np.tile(b, (m, 1)), 0.0, "zero input is the bias")
    _close(moe.linear_bias(x, np.eye(k), np.zeros(k)), x, 0.0, "identity weight")
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w), torch.from_numpy(b)).numpy()
    _close(moe.linear_bias(x, w, b), ref, 1e-13, "vs torch linear in fp64")


# ------------------------------------------------------------------ YaRN rotary
def pin_yarn_factor_one_is_plain_rope():
    _close(rope.yarn_inv_freq(4, 10000.0, 1.0, 4096, 32.0, 1.0), [1.0, 0.01], 1e-16, "D=4 plain RoPE")
    assert rope.yarn_mscale(1.0) == 1.0


def pin_yarn_ramp_closed_form():
    """D=8, base 16: theta = 2^-i.  With L = 1024, beta_fast = 1024 / (4 pi) and
    beta_slow = 1024 / (16 pi) the ramp runs from pair index 1 to 3, so
    rho = (0, 0, 1/2, 1) and theta' = (1, 1/2, (1/4)(1/2 + 1/(2s)), 1/(8s))."""
    s = 4.0
    got = rope.yarn_inv_freq(8, 16.0, s, 1024, 1024 / (4 * math.pi), 1024 / (16 * math.pi))
    _close(got, [1.0, 0.5, 0.25 * (0.5 + 0.5 / s), 0.125 / s], 1e-15, "YaRN ramp")


def pin_yarn_boundaries():
    """Pairs turning more than beta_fast times over the original length keep theta;
    pairs turning less than beta_slow times are divided by s; the rest lie between."""
    d, base, s, L, bf, bs = 64, 150000.0, 32.0, 4096, 32.0, 1.0
    theta = base ** (-np.arange(d // 2) * 2.0 / d)
    turns = L * theta / (2 * math.pi)
    got = rope.yarn_inv_freq(d, base, s, L, bf, bs)
    fast, slow = turns >= bf, turns <= bs
    assert fast.any() and slow.any()
    _close(got[fast], theta[fast], 0.0, "fast pairs keep theta")
    _close(got[slow], theta[slow] / s, 1e-18, "slow pairs interpolate")
    mid = ~(fast | slow)
    assert np.all(got[mid] < theta[mid]) and np.all(got[mid] > theta[mid] / s)
    assert np.all(np.diff(got) < 0)
    _close(rope.yarn_mscale(math.exp(10.0)), 2.0, 1e-15, "mscale at s = e^10")


def pin_rotation_hand_worked():
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    got = rope.rope_rotate(x, [1], [1.0, 0.01])
    c1, s1, c2, s2 = math.cos(1), math.sin(1), math.cos(0.01), math.sin(0.01)
    _close(got[0, 0], [c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + s1, 4 * c2 + 2 * s2], 1e-15, "D=4 rotation")


def pin_rotation_is_complex_multiplication():
    rng = np.random.default_rng(18)
    x = rng.standard_normal((6, 3, 64))
    pos = rng.integers(0, 131072, 6)
    inv = rope.yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    ms = rope.yarn_mscale(32.0)
    got = rope.rope_rotate(x, pos, inv, ms)
    z = (x[..., :32] + 1j * x[..., 32:]) * (ms * np.exp(1j * pos[:, None, None] * inv[None, None, :]))
    _close(got, np.concatenate([z.real, z.imag], axis=-1), 1e-10, "complex rotation")


def pin_rotation_relative_position():
    """<R(p) q, R(p') k> depends on p - p' only, scaled by mscale^2; norms scale by mscale."""
    rng = np.random.default_rng(19)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    inv = rope.yarn_inv_freq(64, 150000.0, 32.0, 4096, 32.0, 1.0)
    ms = rope.yarn_mscale(32.0)

    def dot(p1, p2):
        return float(np.sum(rope.rope_rotate(q, [p1], inv, ms) * rope.rope_rotate(k, [p2], inv, ms)))
    _close(dot(100, 37), dot(5100, 5037), 1e-9, "relative position")
    _close(dot(0, 0), ms * ms * float(np.sum(q * k)), 1e-12, "position 0")
    n = np.linalg.norm(rope.rope_rotate(q, [777], inv, ms))
    _close(n, ms * np.linalg.norm(q), 1e-12, "norm")


def pin_positions_and_layout():
    assert rope.token_positions([0, 3, 3, 5], [10, 4, 2]).tolist() == [7, 8, 9, 0, 1]
    assert rope.token_positions([0, 2, 5]).tolist() == [0, 1, 0, 1, 2]
    hq, hkv, d, t = 4, 2, 4, 3
    qkv = np.repeat(np.arange(hq + 2 * hkv, dtype=np.float64), d)[None, :].repeat(t, 0)
    bias = np.full((hq + 2 * hkv) * d, 0.5)
    q, k, v = rope.qkv_bias_rope(qkv, bias, [0, t], None, hq, hkv, d, [0.0, 0.0], 1.0)
    assert np.all(q == np.arange(hq)[None, :, None] + 0.5)
    assert np.all(k == hq + np.arange(hkv)[None, :, None] + 0.5)
    assert np.all(v == hq + hkv + np.arange(hkv)[None, :, None] + 0.5)
    # values are never rotated; keys and queries are
    q, k, v = rope.qkv_bias_rope(qkv, None, [0, t], None, hq, hkv, d, [1.0, 0.5], 1.0)
    assert np.all(v == hq + hkv + np.arange(hkv)[None, :, None])
    assert not np.allclose(k[1:], hq + np.arange(hkv)[None, :, None])


def pin_append_paged_kv():
    kp = np.zeros((4, 1, 2, 1))
    vp = np.zeros((4, 1, 2, 1))
    # sequence 0: 1 new token at position 2 -> page_table[0][1] = 3, row 0
    # sequence 1: 2 new tokens at positions 0, 1 -> page 0 rows 0, 1
    pt = np.array([[2, 3], [0, 1]])
    kn = np.array([[[7.0]], [[8.0]], [[9.0]]])
    k2, v2 = rope.append_paged_kv(kp, vp, pt, [0, 1, 3], [3, 2], kn, -kn)
    want = np.zeros((4, 1, 2, 1))
    want[3, 0, 0, 0], want[0, 0, 0, 0], want[0, 0, 1, 0] = 7.0, 8.0, 9.0
    _close(k2, want, 0.0, "paged append K")
    _close(v2, -want, 0.0, "paged append V")


ALL_PINS = [pin_round_to_bf16, pin_topk_is_stable_descending_sort, pin_router_k1_is_argmax,
            pin_router_all_experts_is_softmax, pin_router_renormalises_selected,
            pin_router_equal_and_two_expert_closed_forms, pin_router_decides_on_bf16_logits,
            pin_expert_counts, pin_linear_bias_special_cases, pin_yarn_factor_one_is_plain_rope,
            pin_yarn_ramp_closed_form, pin_yarn_boundaries, pin_rotation_hand_worked,
            pin_rotation_is_complex_multiplication, pin_rotation_relative_position,
            pin_positions_and_layout, pin_append_paged_kv]


def failing_pins():
    bad = []
    for p in ALL_PINS:
        try:
            p()
        except Exception:          # noqa: BLE001 - any failure counts
            bad.append(p.__name__)
    return bad
