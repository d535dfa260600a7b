"""GPU parity: attention with q taken from the QKV projection output and rotated on chip.

The page "GPT-OSS on day 0" (model overview list) gives the QKV projections biases
and encodes positions with YaRN; the *_qkv attention calls apply the query bias
and the rotation inside the attention kernels (prefill: in shared memory before
the first score MMA; decode: in the registers that hold q), after
qkv_bias_rope_kv / qkv_bias_rope_append_paged_kv wrote the rotated keys and the
per-token (cos, sin) table.  Each case is checked two ways:

* against the unfused path (qkv_bias_rope writing rotated q, then the plain
  call): the on-chip arithmetic is the same, so outputs must be bit-identical;
* end to end against the oracle: the q, k, v the GPU stores (k, v in the cache;
  q as the unfused kernel writes it, which the bitwise check ties to the on-chip
  q) must each be a bf16 rounding of the oracle's fp64 bias + YaRN value to
  within fp32 arithmetic error, and the attention oracle run on those bytes must
  match the fused output.  The bf16 rounding of q and k is a decision taken in
  the kernel's precision: near a rounding midpoint the fp32 and fp64 rotations
  can round to neighbouring bf16 values, and one such step moves a logit by up to
  about 2^-8 |q_d k_d| sm_scale (4e-3 here), more than the 1e-3 lse budget of the
  attention itself, so the oracle attends over the stored values.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close, bf16, bf16_store_excess, dev, host, oracle_workers, require_gpu
from oracle import rope as orope

pytestmark = pytest.mark.gpu

HQ, HKV, D = 64, 8, 64


def _yarn(sa):
    p = sa.GPT_OSS_YARN
    inv = orope.yarn_inv_freq(D, p["rope_base"], p["factor"], p["orig_len"], p["beta_fast"], p["beta_slow"])
    return inv, orope.yarn_mscale(p["factor"])


def _oracle_qkv(sa, qkv, bias, cu, kv_lens, hq=HQ, hkv=HKV):
    """Oracle bias + rotation in fp64: (q, k, v) [T, H, D]."""
    inv, ms = _yarn(sa)
    return orope.qkv_bias_rope(qkv, bias, cu, kv_lens, hq, hkv, D, inv, ms)


def _assert_valid_rounding(stored, exact, what):
    """Every stored bf16 value is the rounding of a real within fp32 arithmetic error
    (2e-6 relative, floor 2e-6) of the oracle's fp64 value."""
    g = np.asarray(stored, dtype=np.float64)
    y = np.asarray(exact, dtype=np.float64)
    excess = bf16_store_excess(g, y)
    bound = 2e-6 * np.maximum(1.0, np.abs(y))
    worst = float((excess - bound).max()) if excess.size else 0.0
    print(f"ROUND {what}: max excess {float(excess.max()):.3e}")
    assert worst <= 0.0, f"{what}: stored bf16 value not a rounding of the oracle value (excess {worst:.3e})"


@pytest.mark.parametrize("lens,with_bias", [([1, 127, 128, 129, 300, 513], True),
                                            ([700, 5, 64], False)])
def test_fused_prefill_equals_unfused_and_oracle(lens, with_bias):
    sa = require_gpu()
    cu = workloads.cu_seqlens_from(lens)
    t = int(cu[-1])
    inp = workloads.make_qkv(51, t, HQ, HKV)
    qkv, cu_d = bf16(inp["qkv"]), dev(cu)
    bias = bf16(inp["bias"]) if with_bias else None
    sinks = dev(workloads.sinks_f32(51, HQ))
    # unfused: rotated q, k, v from the rope kernel, then the plain prefill
    q, k, v = sa.qkv_bias_rope(qkv, bias, cu_d, HQ, HKV)
    o_ref, l_ref = sa.sink_attn_prefill(q, k, v, sinks, cu_d, max(lens), 0.125)
    # fused: k, v and the table from the K/V pass; q rotated inside the prefill
    k2, v2, table = sa.qkv_bias_rope_kv(qkv, bias, cu_d, HQ, HKV)
    assert torch.equal(k2, k) and torch.equal(v2, v)
    o, l = sa.sink_attn_prefill_qkv(qkv, bias, table, k2, v2, sinks, cu_d, max(lens), 0.125, HQ)
    assert sa.sink_attn_device_status(True) == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref), "fused prefill differs from the unfused path"
    # end to end against the oracle
    rq, rk, rv = _oracle_qkv(sa, inp["qkv"], inp["bias"] if with_bias else None, cu, None)
    for name, g, y in (("q", q, rq), ("k", k2, rk), ("v", v2, rv)):
        _assert_valid_rounding(host(g), y, f"prefill {name}")
    ro, rl = oracle.prefill(host(q), host(k2), host(v2), host(sinks), cu, 0.125, True, workers=oracle_workers())
    assert_close(host(o), host(l), ro, rl, f"fused prefill lens={lens} bias={with_bias}")


def test_fused_prefill_causal_4x8192_equals_unfused():
    """The causal-prefill shape (4 x 8192 tokens, 64/8 heads): fused and unfused agree bit for bit."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["causal_prefill"]
    lens = [cfg["seqlen"]] * cfg["batch"]
    cu = workloads.cu_seqlens_from(lens)
    inp = workloads.make_qkv(52, int(cu[-1]), HQ, HKV)
    qkv, bias, cu_d = bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu)
    sinks = dev(workloads.sinks_f32(52, HQ, cfg["sink_std"]))
    q, k, v = sa.qkv_bias_rope(qkv, bias, cu_d, HQ, HKV)
    o_ref, l_ref = sa.sink_attn_prefill(q, k, v, sinks, cu_d, cfg["seqlen"], cfg["sm_scale"])
    del q
    k2, v2, table = sa.qkv_bias_rope_kv(qkv, bias, cu_d, HQ, HKV)
    o, l = sa.sink_attn_prefill_qkv(qkv, bias, table, k2, v2, sinks, cu_d, cfg["seqlen"], cfg["sm_scale"], HQ)
    assert sa.sink_attn_device_status(True) == 0
    assert torch.equal(k2, k) and torch.equal(v2, v)
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def _paged_case(seed, q_lens, kv_lens, hq=HQ, hkv=HKV):
    """A paged cache holding each sequence's earlier tokens, plus the projection output of
    its q_len new tokens (the last q_len positions)."""
    base = workloads.make_mixed(seed, q_lens, kv_lens, hq, hkv, D)
    cu = base["cu_seqlens_q"]
    inp = workloads.make_qkv(seed + 100, int(cu[-1]), hq, hkv)
    return base, inp


@pytest.mark.parametrize("q_lens,kv_lens", [([1, 5, 128, 129, 300, 1], [1, 40, 128, 700, 300, 2000]),
                                            ([1, 1, 1, 3, 17], [4096, 33, 900, 3, 17])])
def test_fused_paged_prefill_equals_unfused_and_oracle(q_lens, kv_lens):
    sa = require_gpu()
    base, inp = _paged_case(61, q_lens, kv_lens)
    cu, kvl, table_d = base["cu_seqlens_q"], base["kv_lens"], dev(base["page_table"])
    qkv, bias = bf16(inp["qkv"]), bf16(inp["bias"])
    cu_d, kvl_d = dev(cu), dev(kvl)
    sinks = dev(base["sinks"])
    # unfused: append k, v and write rotated q; then the plain paged prefill
    kp1, vp1 = bf16(base["k_pages"]), bf16(base["v_pages"])
    q = sa.qkv_bias_rope_append_paged(qkv, bias, cu_d, kvl_d, kp1, vp1, table_d, HQ)
    o_ref, l_ref = sa.sink_attn_prefill_paged(q, kp1, vp1, table_d, cu_d, kvl_d, sinks, max(q_lens), 0.125)
    # fused
    kp2, vp2 = bf16(base["k_pages"]), bf16(base["v_pages"])
    rt = sa.qkv_bias_rope_append_paged_kv(qkv, bias, cu_d, kvl_d, kp2, vp2, table_d, HQ)
    assert torch.equal(kp1, kp2) and torch.equal(vp1, vp2)
    o, l = sa.sink_attn_prefill_paged_qkv(qkv, bias, rt, kp2, vp2, table_d, cu_d, kvl_d, sinks, max(q_lens),
                                          0.125, HQ)
    assert sa.sink_attn_device_status(True) == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref), "fused paged prefill differs from the unfused path"
    # oracle: the appended cache holds roundings of the oracle's k, v at the new positions
    # and the old contents elsewhere; q likewise; then attend over the stored bytes
    rq, rk, rv = _oracle_qkv(sa, inp["qkv"], inp["bias"], cu, kvl)
    kp, vp = orope.append_paged_kv(base["k_pages"], base["v_pages"], base["page_table"], cu, kvl, rk, rv)
    _assert_valid_rounding(host(q), rq, "paged q")
    _assert_valid_rounding(host(kp2), kp, "paged k cache")
    _assert_valid_rounding(host(vp2), vp, "paged v cache")
    ro, rl = oracle.prefill_paged(host(q), host(kp2), host(vp2), base["page_table"], cu, kvl, base["sinks"],
                                  0.125, True, workers=oracle_workers())
    assert_close(host(o), host(l), ro, rl, f"fused paged prefill q_lens={q_lens}")


@pytest.mark.parametrize("splits", [1, 4])
@pytest.mark.parametrize("hq,hkv", [(64, 8), (24, 2)])
def test_fused_decode_equals_unfused_and_oracle(splits, hq, hkv):
    sa = require_gpu()
    kv_lens = [1, 17, 600, 4096, 2049]
    q_lens = [1] * len(kv_lens)
    base, inp = _paged_case(71, q_lens, kv_lens, hq, hkv)
    cu, kvl, table_d = base["cu_seqlens_q"], base["kv_lens"], dev(base["page_table"])
    qkv, bias = bf16(inp["qkv"]), bf16(inp["bias"])
    cu_d, kvl_d = dev(cu), dev(kvl)
    sinks = dev(base["sinks"])
    kp1, vp1 = bf16(base["k_pages"]), bf16(base["v_pages"])
    q = sa.qkv_bias_rope_append_paged(qkv, bias, cu_d, kvl_d, kp1, vp1, table_d, hq)
    kp2, vp2 = bf16(base["k_pages"]), bf16(base["v_pages"])
    rt = sa.qkv_bias_rope_append_paged_kv(qkv, bias, cu_d, kvl_d, kp2, vp2, table_d, hq)
    assert torch.equal(kp1, kp2) and torch.equal(vp1, vp2)
    o_ref, l_ref = sa.sink_attn_decode(q, kp1, vp1, table_d, kvl_d, sinks, 0.125, num_splits=splits)
    o, l = sa.sink_attn_decode_qkv(qkv, bias, rt, kp2, vp2, table_d, kvl_d, sinks, 0.125, hq,
                                   num_splits=splits)
    assert sa.sink_attn_device_status(True) == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref), "fused decode differs from the unfused path"
    if splits > 1:
        o, l = sa.sink_attn_merge(o, l)
    rq, rk, rv = _oracle_qkv(sa, inp["qkv"], inp["bias"], cu, kvl, hq, hkv)
    kp, vp = orope.append_paged_kv(base["k_pages"], base["v_pages"], base["page_table"], cu, kvl, rk, rv)
    _assert_valid_rounding(host(q), rq, "decode q")
    _assert_valid_rounding(host(kp2), kp, "decode k cache")
    _assert_valid_rounding(host(vp2), vp, "decode v cache")
    ro, rl = oracle.decode(host(q), host(kp2), host(vp2), base["page_table"], kvl, base["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, f"fused decode {hq}/{hkv} splits={splits}")


def test_fused_calls_reject_bad_arguments():
    sa = require_gpu()
    inp = workloads.make_qkv(81, 16, HQ, HKV)
    qkv = bf16(inp["qkv"])
    cu = dev(workloads.cu_seqlens_from([16]))
    k, v, table = sa.qkv_bias_rope_kv(qkv, None, cu, HQ, HKV)
    lib = sa.load_library()
    st = lib.sink_attn_prefill_qkv(qkv.data_ptr(), None, None, k.data_ptr(), v.data_ptr(),
                                   dev(np.zeros(HQ, np.float32)).data_ptr(), cu.data_ptr(), 1, 16, 16, HQ, HKV, 64,
                                   0.125, 1, qkv.data_ptr(), None, None)
    assert st == 1  # SA_ERR_NULL: the table is required
    st = lib.sink_attn_prefill_qkv(qkv.data_ptr(), None, table.data_ptr() + 8, k.data_ptr(), v.data_ptr(),
                                   dev(np.zeros(HQ, np.float32)).data_ptr(), cu.data_ptr(), 1, 16, 16, HQ, HKV, 64,
                                   0.125, 1, qkv.data_ptr(), None, None)
    assert st == 7  # SA_ERR_ALIGNMENT
