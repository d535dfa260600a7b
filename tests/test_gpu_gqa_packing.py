"""GPU parity of GQA packing in the persistent prefill schedule: sequences with at
most 2 * 128 / G new tokens (G = query heads per KV head >= 4) are computed as one
item per KV head whose tiles hold 128 / G tokens x the G heads.  Lengths straddle
the packing limit and the tile boundary inside a packed item; paged and contiguous
KV, causal and not, G = 4, 8, 16."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_common import assert_close, bf16, dev, host, require_gpu

pytestmark = pytest.mark.gpu


def _lens(g):
    tpt = 128 // g          # tokens per packed tile
    lim = 2 * tpt           # packing limit
    q = [1, tpt - 1, tpt, tpt + 1, lim - 1, lim, lim + 1, 1, 3, 200]
    return [x for x in q if x >= 1]


@pytest.mark.parametrize("hq,hkv", [(64, 16), (64, 8), (32, 2)])
@pytest.mark.parametrize("causal", [True, False])
def test_packed_paged(hq, hkv, causal):
    sa = require_gpu()
    q_lens = _lens(hq // hkv)
    kv_lens = [max(q, 1) + extra for q, extra in zip(q_lens, [0, 17, 300, 5, 128, 1000, 33, 4095, 2, 64])]
    d = workloads.make_mixed(71, q_lens, kv_lens, hq, hkv, 64)
    o, l = sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), max(q_lens), 0.125, causal=causal)
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"],
                                  d["cu_seqlens_q"], d["kv_lens"], d["sinks"], 0.125, causal)
    assert_close(host(o), host(l), ro, rl, f"packed paged hq={hq} hkv={hkv} causal={causal}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("hq,hkv", [(64, 8), (16, 4)])
def test_packed_contiguous(hq, hkv):
    sa = require_gpu()
    lens = _lens(hq // hkv)
    d = workloads.make_prefill(72, lens, hq, hkv, 64)
    o, l = sa.sink_attn_prefill(bf16(d["q"]), bf16(d["k"]), bf16(d["v"]), dev(d["sinks"]),
                                dev(d["cu_seqlens"]), max(lens), 0.125, causal=True)
    ro, rl = oracle.prefill(d["q"], d["k"], d["v"], d["sinks"], d["cu_seqlens"], 0.125, True)
    assert_close(host(o), host(l), ro, rl, f"packed contiguous hq={hq} hkv={hkv}")
    assert sa.sink_attn_device_status(True) == 0


def test_many_decode_rows_in_one_call():
    """300 single-token rows (KV 1..5000) plus two chunks: most items are packed."""
    sa = require_gpu()
    rng = np.random.default_rng(73)
    q_lens = [1] * 300 + [500, 31]
    kv_lens = list(rng.integers(1, 5000, 300)) + [1500, 31]
    d = workloads.make_mixed(74, q_lens, kv_lens, 64, 8, 64)
    o, l = sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), 500, 0.125, causal=True)
    cu = d["cu_seqlens_q"]
    rows = [(int(cu[b]), int(h)) for b, h in zip(range(0, 300, 7), rng.integers(0, 64, 43))]
    rows += [(int(cu[300]) + 499, 5), (int(cu[301]) + 30, 63), (int(cu[301]), 0)]
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"], cu,
                                  d["kv_lens"], d["sinks"], 0.125, True, rows=rows)
    go = host(o)[[r[0] for r in rows], [r[1] for r in rows]]
    gl = host(l)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_close(go, gl, ro, rl, "many decode rows")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("hq,hkv", [(24, 2), (6, 2), (40, 8), (12, 1)])
def test_groups_that_do_not_divide_the_tile(hq, hkv):
    """Group sizes 12, 3, 5 and 12 (odd, or not dividing 128): short sequences are not
    packed and take the head-pair (or single-head) items; results match the oracle."""
    sa = require_gpu()
    q_lens = [1, 3, 9, 20, 40, 130]
    kv_lens = [1, 100, 9, 700, 40, 200]
    d = workloads.make_mixed(75, q_lens, kv_lens, hq, hkv, 64)
    o, l = sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), max(q_lens), 0.125, causal=True)
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"],
                                  d["cu_seqlens_q"], d["kv_lens"], d["sinks"], 0.125, True)
    assert_close(host(o), host(l), ro, rl, f"group {hq // hkv} paged")
    c = workloads.make_prefill(76, q_lens, hq, hkv, 64)
    o2, l2 = sa.sink_attn_prefill(bf16(c["q"]), bf16(c["k"]), bf16(c["v"]), dev(c["sinks"]),
                                  dev(c["cu_seqlens"]), max(q_lens), 0.125)
    ro2, rl2 = oracle.prefill(c["q"], c["k"], c["v"], c["sinks"], c["cu_seqlens"], 0.125, True)
    assert_close(host(o2), host(l2), ro2, rl2, f"group {hq // hkv} contiguous")
    assert sa.sink_attn_device_status(True) == 0
