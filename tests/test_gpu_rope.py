"""GPU parity: QKV bias + YaRN rotary encoding (+ paged K/V append) against the
fp64 oracle.

Tolerance, from the arithmetic: the kernel adds the bias in fp32, rotates with
fp32 cos/sin of an angle reduced in fp64 (error below 3e-7 rad after rounding
the reduced angle to fp32), and rounds once to bf16.  So an output may differ
from the exact value by the bf16 storage rounding (at most 2^-8 of its
magnitude) plus 1e-6 * mscale * (|a| + |b|), where (a, b) is the biased pair
it was rotated from.  Values (not rotated) get the storage term only.  Cache
slots that no new token maps to must keep their bytes exactly."""
import numpy as np
import pytest
import torch

import workloads
from gpu_common import bf16, dev, host, require_gpu
from oracle import rope as orope
from oracle import widen_bf16

pytestmark = pytest.mark.gpu

STORE = 2.0 ** -8
FP32 = 1e-6


def _params(sa, plain=False):
    if plain:
        return dict(rope_base=10000.0, factor=1.0, orig_len=4096, beta_fast=32.0, beta_slow=1.0)
    return dict(sa.GPT_OSS_YARN)


def _oracle_tables(p):
    inv = orope.yarn_inv_freq(64, p["rope_base"], p["factor"], p["orig_len"], p["beta_fast"],
                              p["beta_slow"])
    return inv, orope.yarn_mscale(p["factor"])


def _pair_scale(x):
    """|a| + |b| for every feature, with (a, b) its rotation pair."""
    half = x.shape[-1] // 2
    s = np.abs(x[..., :half]) + np.abs(x[..., half:])
    return np.concatenate([s, s], axis=-1)


def _assert_rot(got, ref, pre, ms, what):
    bound = STORE * np.abs(ref) + FP32 * ms * _pair_scale(pre) + 1e-30
    excess = np.abs(got - ref) - bound
    print(f"ERR {what}: raw {np.abs(got - ref).max():.3e} beyond-bound {excess.max():.3e}")
    assert excess.max() <= 0.0, f"{what}: {excess.max()}"


def _biased(qkv, bias, hq, hkv):
    x = widen_bf16(qkv) + (0.0 if bias is None else widen_bf16(bias)[None, :])
    t = x.shape[0]
    return (x[:, :hq * 64].reshape(t, hq, 64), x[:, hq * 64:(hq + hkv) * 64].reshape(t, hkv, 64),
            x[:, (hq + hkv) * 64:].reshape(t, hkv, 64))


@pytest.mark.parametrize("plain", [False, True])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("hq,hkv", [(64, 8), (4, 1), (120, 4), (48, 8)])
def test_qkv_bias_rope_contiguous(plain, with_bias, hq, hkv):
    # A CTA takes the whole tokens that fit 64 KB of qkv rows: 6 at 64/8 heads, 16 (the cap)
    # at 4/1, 4 at 120/4 (128 head rows, the largest supported), 8 at 48/8; the 323 tokens
    # leave a partial last CTA in every case.
    sa = require_gpu()
    q_lens = [5, 0, 300, 1, 17]
    kv_lens = np.array([10, 3, 300, 131072, 4000], dtype=np.int32)
    cu = workloads.cu_seqlens_from(q_lens)
    t = int(cu[-1])
    inp = workloads.make_qkv(31, t, hq, hkv)
    bias = inp["bias"] if with_bias else None
    p = _params(sa, plain)
    q, k, v = sa.qkv_bias_rope(bf16(inp["qkv"]), None if bias is None else bf16(bias), dev(cu), hq, hkv,
                               kv_lens=dev(kv_lens), rope=p)
    inv, ms = _oracle_tables(p)
    rq, rk, rv = orope.qkv_bias_rope(inp["qkv"], bias, cu, kv_lens, hq, hkv, 64, inv, ms)
    pq, pk, pv = _biased(inp["qkv"], bias, hq, hkv)
    _assert_rot(host(q), rq, pq, ms, "q")
    _assert_rot(host(k), rk, pk, ms, "k")
    _assert_rot(host(v), rv, np.zeros_like(pv), 0.0, "v")
    assert sa.sink_attn_device_status(True) == 0


def test_qkv_rope_positions_default_to_zero_based():
    sa = require_gpu()
    cu = workloads.cu_seqlens_from([7, 9])
    inp = workloads.make_qkv(32, 16, 8, 2)
    p = _params(sa)
    q, k, v = sa.qkv_bias_rope(bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu), 8, 2, rope=p)
    inv, ms = _oracle_tables(p)
    rq, rk, rv = orope.qkv_bias_rope(inp["qkv"], inp["bias"], cu, None, 8, 2, 64, inv, ms)
    pq, pk, _ = _biased(inp["qkv"], inp["bias"], 8, 2)
    _assert_rot(host(q), rq, pq, ms, "q zero-based")
    _assert_rot(host(k), rk, pk, ms, "k zero-based")


def test_append_paged_kv_mixed_batch():
    """Ragged mixed batch: decode rows (1 new token) and chunks, permuted pages, a
    cache pre-filled with random bytes; only the new tokens' slots may change."""
    sa = require_gpu()
    hq, hkv = 64, 8
    q_lens = np.array([1, 40, 0, 1, 129, 16], dtype=np.int32)
    kv_lens = np.array([1, 700, 33, 17, 129, 48], dtype=np.int32)
    cu = workloads.cu_seqlens_from(q_lens)
    t = int(cu[-1])
    table, num_pages = workloads.page_layout(33, kv_lens, 16, permute=True, extra_pages=3)
    kp = workloads.normal_bf16(34, 1, (num_pages, hkv, 16, 64))
    vp = workloads.normal_bf16(34, 2, (num_pages, hkv, 16, 64))
    inp = workloads.make_qkv(35, t, hq, hkv)
    p = _params(sa)
    gk, gv = bf16(kp), bf16(vp)
    q = sa.qkv_bias_rope_append_paged(bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu), dev(kv_lens), gk, gv,
                                      dev(table), hq, rope=p)
    inv, ms = _oracle_tables(p)
    rq, rk, rv = orope.qkv_bias_rope(inp["qkv"], inp["bias"], cu, kv_lens, hq, hkv, 64, inv, ms)
    ek, ev = orope.append_paged_kv(kp, vp, table, cu, kv_lens, rk, rv)
    pq, pk, pv = _biased(inp["qkv"], inp["bias"], hq, hkv)
    _assert_rot(host(q), rq, pq, ms, "q paged")
    # the slots written, and the untouched remainder byte for byte
    written = np.zeros((num_pages, 16), dtype=bool)
    pos = orope.token_positions(cu, kv_lens)
    pre_k = np.zeros_like(ek)
    for b in range(len(q_lens)):
        for tok in range(int(cu[b]), int(cu[b + 1])):
            pg, row = int(table[b, pos[tok] // 16]), int(pos[tok] % 16)
            written[pg, row] = True
            pre_k[pg, :, row, :] = pk[tok]
    gkn = gk.view(torch.int16).cpu().numpy().view(np.uint16)
    gvn = gv.view(torch.int16).cpu().numpy().view(np.uint16)
    mask = np.broadcast_to(written[:, None, :, None], gkn.shape)
    assert np.array_equal(gkn[~mask], kp[~mask]) and np.array_equal(gvn[~mask], vp[~mask])
    gkf, gvf = widen_bf16(gkn), widen_bf16(gvn)
    sel = written
    _assert_rot(gkf.transpose(0, 2, 1, 3)[sel], ek.transpose(0, 2, 1, 3)[sel],
                pre_k.transpose(0, 2, 1, 3)[sel], ms, "k appended")
    _assert_rot(gvf.transpose(0, 2, 1, 3)[sel], ev.transpose(0, 2, 1, 3)[sel],
                np.zeros_like(ev.transpose(0, 2, 1, 3)[sel]), 0.0, "v appended")
    assert sa.sink_attn_device_status(True) == 0


def test_append_rejects_positions_outside_the_table():
    """kv_len beyond the page table: the token's K/V is skipped and the status word
    reports it; nothing else is written."""
    sa = require_gpu()
    cu = workloads.cu_seqlens_from([2])
    kv = np.array([40], dtype=np.int32)            # positions 38, 39 -> page index 2
    table = np.array([[0, 1]], dtype=np.int32)     # only two pages mapped
    kp = workloads.normal_bf16(36, 1, (2, 1, 16, 64))
    vp = workloads.normal_bf16(36, 2, (2, 1, 16, 64))
    inp = workloads.make_qkv(37, 2, 4, 1)
    gk, gv = bf16(kp), bf16(vp)
    sa.qkv_bias_rope_append_paged(bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu), dev(kv), gk, gv,
                                  dev(table), 4)
    assert sa.sink_attn_device_status(True) == 5          # SA_ERR_BOUNDS
    assert np.array_equal(gk.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(gv.view(torch.int16).cpu().numpy().view(np.uint16), vp)


def test_qkv_rope_prefill_sized_sampled():
    """32768 tokens (4 x 8192 causal-prefill batch), 64/8 heads, GPT-OSS YaRN; 256
    sampled tokens against the oracle."""
    sa = require_gpu()
    cu = workloads.cu_seqlens_from([8192] * 4)
    inp = workloads.make_qkv(38, 32768, 64, 8)
    p = _params(sa)
    q, k, v = sa.qkv_bias_rope(bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu), 64, 8, rope=p)
    rows = np.sort(np.random.default_rng(6).choice(32768, 256, replace=False))
    inv, ms = _oracle_tables(p)
    pos = orope.token_positions(cu)[rows]
    sub_cu = np.arange(len(rows) + 1, dtype=np.int32)
    sub_kv = (pos + 1).astype(np.int32)                  # one token per row at its own position
    rq, rk, rv = orope.qkv_bias_rope(inp["qkv"][rows], inp["bias"], sub_cu, sub_kv, 64, 8, 64, inv, ms)
    pq, pk, _ = _biased(inp["qkv"][rows], inp["bias"], 64, 8)
    _assert_rot(host(q)[rows], rq, pq, ms, "q 32k")
    _assert_rot(host(k)[rows], rk, pk, ms, "k 32k")
    _assert_rot(host(v)[rows], rv, np.zeros_like(rv), 0.0, "v 32k")


def test_append_then_decode_step():
    """One decode step as a serving loop runs it: the new token's QKV gets its bias and
    YaRN rotation and its K/V are appended to the paged cache (qkv_bias_rope_append_paged),
    then attention with sinks reads the cache (split decode + merge).  The oracle builds
    its own cache: fp64 rotation rounded to bf16, appended by the oracle, then its decode."""
    from oracle import moe
    import oracle
    sa = require_gpu()
    hq, hkv = 64, 8
    kv_lens = np.array([1, 17, 300, 4096], dtype=np.int32)     # including the new token
    b = len(kv_lens)
    base = workloads.make_decode(94, list(kv_lens), hq, hkv, 64)
    cu = np.arange(b + 1, dtype=np.int32)                        # one new token per sequence
    inp = workloads.make_qkv(95, b, hq, hkv)
    p = _params(sa)
    gk, gv = bf16(base["k_pages"]), bf16(base["v_pages"])
    q = sa.qkv_bias_rope_append_paged(bf16(inp["qkv"]), bf16(inp["bias"]), dev(cu), dev(kv_lens), gk, gv,
                                      dev(base["page_table"]), hq, rope=p)
    po, pl = sa.sink_attn_decode(q, gk, gv, dev(base["page_table"]), dev(kv_lens), dev(base["sinks"]), 0.125,
                                 num_splits=3)
    out, lse = sa.sink_attn_merge(po, pl)
    inv, ms = _oracle_tables(p)
    rq, rk, rv = orope.qkv_bias_rope(inp["qkv"], inp["bias"], cu, kv_lens, hq, hkv, 64, inv, ms)
    bits = lambda x: moe.bf16_bits(moe.round_to_bf16(x))
    kp, vp = orope.append_paged_kv(base["k_pages"], base["v_pages"], base["page_table"], cu, kv_lens,
                                   moe.round_to_bf16(rk), moe.round_to_bf16(rv))
    ro, rl = oracle.decode(bits(rq), bits(kp), bits(vp), base["page_table"], kv_lens, base["sinks"], 0.125)
    from gpu_common import assert_close
    assert_close(host(out), host(lse), ro, rl, "append then decode")
    assert sa.sink_attn_device_status(True) == 0
