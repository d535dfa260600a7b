"""GPU parity on edge cases: empty rows and sequences, large batches, long sequences."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_common import assert_close, bf16, dev, host, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_zero_length_rows(splits):
    """kv_len == 0: only the sink remains, so out = 0 and lse = sink (-inf without sink)."""
    sa = require_gpu()
    kv = [0, 5, 0, 300]
    d = workloads.make_decode(41, [max(1, x) for x in kv], 64, 8, 64)
    d["kv_lens"] = np.array(kv, dtype=np.int32)
    d["sinks"][3] = -np.inf
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]
    o, l = sa.sink_attn_decode(*args, 0.125, num_splits=splits)
    if splits > 1:
        o, l = sa.sink_attn_merge(o, l)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125)
    assert np.all(host(o)[[0, 2]] == 0.0)
    assert np.isneginf(host(l)[0, 3]) and host(l)[0, 0] == pytest.approx(float(d["sinks"][0]), abs=1e-6)
    assert_close(host(o), host(l), ro, rl, f"zero-length decode splits={splits}")
    assert sa.sink_attn_device_status(True) == 0


def test_prefill_with_empty_sequences():
    sa = require_gpu()
    lens = [0, 200, 0, 1, 0, 129]
    data = workloads.make_prefill(42, lens, 16, 2, 64)
    o, l = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), 200, 0.125)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True)
    assert_close(host(o), host(l), ro, rl, "prefill with empty sequences")
    assert sa.sink_attn_device_status(True) == 0


def test_paged_prefill_with_empty_and_decode_rows():
    sa = require_gpu()
    q_lens = [0, 1, 1, 0, 40, 1]
    kv_lens = [10, 1, 700, 3, 40, 129]
    d = workloads.make_mixed(43, q_lens, kv_lens, 64, 8, 64)
    o, l = sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), 40, 0.125)
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["cu_seqlens_q"],
                                  d["kv_lens"], d["sinks"], 0.125, True)
    assert_close(host(o), host(l), ro, rl, "paged prefill with empty and decode rows")
    assert sa.sink_attn_device_status(True) == 0


def test_large_decode_batch():
    """1024 sequences of short, ragged KV: many CTAs, every row checked on a sample."""
    sa = require_gpu()
    rng = np.random.default_rng(44)
    kv = rng.integers(1, 600, 1024).tolist()
    d = workloads.make_decode(44, kv, 64, 8, 64)
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]
    o, l = sa.sink_attn_decode(*args, 0.125)
    pick = list(range(0, 1024, 37)) + [1023]
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"], d["sinks"],
                           0.125, batches=pick)
    assert_close(host(o)[pick], host(l)[pick], ro[pick], rl[pick], "decode batch 1024")
    assert sa.sink_attn_device_status(True) == 0


def test_long_single_sequence_prefill():
    """One 32768-token causal sequence, 64/8 heads: sampled rows across the whole range."""
    sa = require_gpu()
    n = 32768
    data = workloads.make_prefill(45, [n], 64, 8, 64)
    o, l = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), n, 0.125)
    rng = np.random.default_rng(46)
    rows = [(int(t), int(h)) for t, h in zip(rng.integers(0, n, 24), rng.integers(0, 64, 24))]
    rows += [(0, 0), (n - 1, 63), (16383, 7)]
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True,
                            rows=rows)
    go = host(o)[[r[0] for r in rows], [r[1] for r in rows]]
    gl = host(l)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_close(go, gl, ro, rl, "32k prefill sampled")
    assert sa.sink_attn_device_status(True) == 0


def test_positive_infinite_sink_everywhere():
    """sink = +inf takes all the probability: out = 0 and lse = +inf on every path
    (prefill, paged prefill, unsplit decode, split decode + merge), as the oracle says."""
    sa = require_gpu()
    data = workloads.make_prefill(91, [130, 7], 8, 1, 64, sink_fill=np.inf)
    o, l = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), 130, 0.125)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True)
    assert np.all(ro == 0) and np.all(np.isposinf(rl))
    assert np.all(host(o) == 0) and np.all(np.isposinf(host(l)))
    d = workloads.make_decode(92, [1, 40, 3000], 64, 8, 64, sink_fill=np.inf)
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]), dev(d["kv_lens"]),
            dev(d["sinks"])]
    o1, l1 = sa.sink_attn_decode(*args, 0.125, num_splits=1)
    po, pl = sa.sink_attn_decode(*args, 0.125, num_splits=4)
    mo, ml = sa.sink_attn_merge(po, pl)
    for out, lse in ((o1, l1), (mo, ml)):
        assert np.all(host(out) == 0) and np.all(np.isposinf(host(lse)))
    m = workloads.make_mixed(93, [1, 20], [50, 300], 64, 8, 64, sink_fill=np.inf)
    o2, l2 = sa.sink_attn_prefill_paged(bf16(m["q"]), bf16(m["k_pages"]), bf16(m["v_pages"]),
                                        dev(m["page_table"]), dev(m["cu_seqlens_q"]), dev(m["kv_lens"]),
                                        dev(m["sinks"]), 20, 0.125)
    assert np.all(host(o2) == 0) and np.all(np.isposinf(host(l2)))
    assert sa.sink_attn_device_status(True) == 0


def _sample_rows(cu, hq, seed):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(len(cu) - 1):
        if cu[b + 1] == cu[b]:
            continue
        for tok in {int(cu[b]), int(cu[b + 1]) - 1, int(rng.integers(cu[b], cu[b + 1]))}:
            rows.append((tok, int(rng.integers(0, hq))))
    return rows


def test_paged_prefill_beyond_the_on_chip_schedule():
    """300 sequences of up to 600 new tokens (1500 sequence x query-block pairs, more than
    the 1024 the persistent schedule sorts on chip): the CTAs fall back to reverse
    query-block order; decode rows, short chunks and empty sequences mixed, sampled rows
    of every sequence against the oracle."""
    sa = require_gpu()
    rng = np.random.default_rng(47)
    q_lens = rng.choice([0, 1, 1, 5, 129, 300, 600], 300).tolist()
    q_lens[7] = 600
    kv_lens = [q + int(rng.integers(0, 900)) for q in q_lens]
    kv_lens = [max(k, 1) for k in kv_lens]
    d = workloads.make_mixed(47, q_lens, kv_lens, 64, 8, 64)
    o, l = sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), 600, 0.125)
    rows = _sample_rows(d["cu_seqlens_q"], 64, 48)
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["cu_seqlens_q"],
                                  d["kv_lens"], d["sinks"], 0.125, True, rows=rows)
    go = host(o)[[r[0] for r in rows], [r[1] for r in rows]]
    gl = host(l)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_close(go, gl, ro, rl, "paged prefill, 1500 pairs")
    assert sa.sink_attn_device_status(True) == 0


def test_contiguous_prefill_beyond_the_on_chip_schedule():
    """The same fallback for a ragged contiguous batch: 300 sequences of 1..600 tokens."""
    sa = require_gpu()
    rng = np.random.default_rng(49)
    lens = rng.integers(1, 601, 300).tolist()
    lens[3] = 600
    data = workloads.make_prefill(49, lens, 64, 8, 64)
    o, l = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), 600, 0.125)
    rows = _sample_rows(data["cu_seqlens"], 64, 50)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True,
                            rows=rows)
    go = host(o)[[r[0] for r in rows], [r[1] for r in rows]]
    gl = host(l)[[r[0] for r in rows], [r[1] for r in rows]]
    assert_close(go, gl, ro, rl, "contiguous prefill, 1500 pairs")
    assert sa.sink_attn_device_status(True) == 0


def test_decode_with_the_largest_split_count():
    """num_splits = 256 (the largest the interface takes) on a 65536-token sequence: 16
    pages per split, merged; two sequences (one shorter, leaving splits empty) checked."""
    sa = require_gpu()
    d = workloads.make_decode(51, [65536, 3000], 64, 8, 64)
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]
    po, pl = sa.sink_attn_decode(*args, 0.125, num_splits=256)
    o, l = sa.sink_attn_merge(po, pl)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"], d["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, "decode, 256 splits")
    assert sa.sink_attn_device_status(True) == 0
