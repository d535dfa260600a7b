"""GPU parity: contiguous causal / full prefill against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close, bf16, dev, host, oracle_workers, require_gpu

pytestmark = pytest.mark.gpu


def _run(sa, data, max_len, scale, causal):
    return sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), max_len, scale, causal=causal)


def test_tiny_prefill_config_full():
    """1 x 128 tokens, causal, 4 query heads on 1 KV head, head_dim 64, sm_scale 1/8."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["tiny_prefill"]
    data = workloads.make_prefill(cfg["seed"], [cfg["seqlen"]], cfg["hq"], cfg["hkv"], cfg["d"],
                                  cfg["sink_std"])
    o, l = _run(sa, data, cfg["seqlen"], cfg["sm_scale"], True)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"],
                            cfg["sm_scale"], True)
    assert_close(host(o), host(l), ro, rl, "tiny prefill")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (64, 8), (3, 3), (16, 1)])
def test_ragged_prefill(causal, hq, hkv):
    """Lengths that span several 128-tiles plus ragged tails, single tokens included."""
    sa = require_gpu()
    lens = [1, 127, 128, 129, 300, 513]
    data = workloads.make_prefill(5, lens, hq, hkv, 64)
    o, l = _run(sa, data, max(lens), 0.125, causal)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"],
                            0.125, causal)
    assert_close(host(o), host(l), ro, rl, f"ragged prefill causal={causal} {hq}/{hkv}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens,hq,hkv", [([1024], 8, 1), ([640, 640, 640], 64, 8)])
def test_uniform_prefill_both_launch_forms(lens, hq, hkv, causal):
    """Equal-length contiguous batches: 32 items (one CTA per item, a single wave) and
    480 items (more than the SMs: the persistent grid)."""
    sa = require_gpu()
    data = workloads.make_prefill(8, lens, hq, hkv, 64)
    o, l = _run(sa, data, lens[0], 0.125, causal)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"],
                            0.125, causal)
    assert_close(host(o), host(l), ro, rl, f"uniform prefill {len(lens)}x{lens[0]} {hq}/{hkv} causal={causal}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("sink_fill", [-np.inf, 20.0, 1.0e4])
def test_prefill_sink_limits(sink_fill):
    sa = require_gpu()
    data = workloads.make_prefill(6, [200, 64], 8, 1, 64, sink_fill=sink_fill)
    o, l = _run(sa, data, 200, 0.125, True)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"],
                            0.125, True)
    assert_close(host(o), host(l), ro, rl, f"sink={sink_fill}")
    if sink_fill == 1.0e4:
        assert np.all(host(o) == 0.0)


def test_prefill_large_scores_rescale():
    """Scores that grow along the sequence force the running max to move many times."""
    sa = require_gpu()
    data = workloads.make_prefill(7, [1024], 8, 1, 64)
    scale = 1.0  # 8x the usual scale: logits of O(10), max jumps across tiles
    o, l = _run(sa, data, 1024, scale, True)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], scale, True)
    assert_close(host(o), host(l), ro, rl, "large logits")


def test_prefill_masked_keys_do_not_set_the_row_max():
    """Rows whose diagonal tile holds masked (future) keys that score over 150 log2 units
    above every visible key.  A full tile takes its row max from the reducing TMEM load;
    a diagonal tile must take it over the visible keys only, or every visible
    probability of these rows would underflow to zero."""
    sa = require_gpu()
    lens = [256, 200]
    data = workloads.make_prefill(9, lens, 8, 1, 64)
    q = data["q"] & np.uint16(0x7FFF)  # |q|: large positive scores against the keys below
    k = data["k"].copy()
    big = np.uint16(0x4180)  # bf16 16.0
    k[100:128] = big         # sequence 0: future of queries 0..99 inside their diagonal tile
    k[256 + 150:256 + 200] = big  # sequence 1: future of queries 128..149 in tile 1
    data = dict(data, q=q, k=k)
    o, l = _run(sa, data, max(lens), 0.125, True)
    assert sa.sink_attn_device_status(True) == 0
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True)
    assert np.isfinite(host(l)).all()
    assert_close(host(o), host(l), ro, rl, "masked large keys")


def test_causal_prefill_config_full():
    """4 x 8192 tokens, 64/8 heads, sinks with variance 2: every (token, head) row of
    every sequence against the oracle, element by element."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["causal_prefill"]
    lens = [cfg["seqlen"]] * cfg["batch"]
    data = workloads.make_prefill(cfg["seed"], lens, cfg["hq"], cfg["hkv"], cfg["d"], cfg["sink_std"])
    o, l = _run(sa, data, cfg["seqlen"], cfg["sm_scale"], True)
    assert sa.sink_attn_device_status(True) == 0
    go, gl = o.float().cpu().numpy(), l.cpu().numpy()
    del o, l
    cu = data["cu_seqlens"]
    for b in range(cfg["batch"]):
        lo, hi = int(cu[b]), int(cu[b + 1])
        ro, rl = oracle.prefill(data["q"][lo:hi], data["k"][lo:hi], data["v"][lo:hi], data["sinks"],
                                [0, hi - lo], cfg["sm_scale"], True, workers=oracle_workers())
        assert_close(go[lo:hi], gl[lo:hi], ro, rl, f"causal prefill 4x8192 sequence {b} (all rows)")
    assert np.isfinite(gl).all()
