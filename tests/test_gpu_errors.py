"""Device-side error reporting without faulting the GPU.

Bad page ids and lengths are caught by the kernels' own bounds checks (the
access is skipped, a status bit is set); a wait that runs out stops its CTA
and sets a status bit.  Each case is followed by a normal call to show that
the context is still usable.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_common import assert_close, bf16, dev, host, require_gpu

pytestmark = pytest.mark.gpu

SA_OK, SA_ERR_BOUNDS, SA_ERR_TIMEOUT = 0, 5, 6


def _decode_ok(sa):
    d = workloads.make_decode(2, [50, 700], 64, 8, 64)
    o, l = sa.sink_attn_decode(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
                               dev(d["kv_lens"]), dev(d["sinks"]), 0.125)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"], d["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, "decode after error")
    assert sa.sink_attn_device_status(True) == SA_OK


def test_bad_page_id_decode_is_reported():
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    d = workloads.make_decode(3, [100, 300], 64, 8, 64)
    table = d["page_table"].copy()
    table[1, 3] = d["num_pages"] + 5        # outside the cache: must be skipped, not read
    table[0, 0] = -7
    sa.sink_attn_decode(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(table),
                        dev(d["kv_lens"]), dev(d["sinks"]), 0.125, num_splits=2)
    assert sa.sink_attn_device_status(True) == SA_ERR_BOUNDS
    _decode_ok(sa)


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_skips_a_bad_page_and_keeps_the_rest(splits):
    """A page id outside the cache is skipped and flagged; every other key still counts.
    Decode attention does not depend on the order of the keys, so the result must equal
    the oracle over the same cache with that page removed.  Odd page counts (37, 22) leave
    a warp's last pair with a single page; the bad page sits inside a pair."""
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    kv = np.array([16 * 37, 16 * 21 + 5], dtype=np.int32)
    d = workloads.make_decode(8, kv.tolist(), 64, 8, 64)
    table = d["page_table"].copy()
    table[0, 10] = d["num_pages"] + 3
    args = (bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(table), dev(d["kv_lens"]),
            dev(d["sinks"]), 0.125)
    if splits > 1:
        po, pl = sa.sink_attn_decode(*args, num_splits=splits)
        o, l = sa.sink_attn_merge(po, pl)
    else:
        o, l = sa.sink_attn_decode(*args)
    assert sa.sink_attn_device_status(True) == SA_ERR_BOUNDS
    ref_table = d["page_table"].copy()
    kept = np.delete(ref_table[0], 10)
    ref_table[0, :kept.shape[0]] = kept
    ref_kv = d["kv_lens"].copy()
    ref_kv[0] -= 16
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], ref_table, ref_kv, d["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, f"decode with a skipped page, {splits} split(s)")


def test_bad_lengths_are_reported():
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    d = workloads.make_decode(4, [100, 300], 64, 8, 64)
    kv = d["kv_lens"].copy()
    kv[0] = d["page_table"].shape[1] * 16 + 1   # more tokens than the page table holds
    sa.sink_attn_decode(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
                        dev(kv), dev(d["sinks"]), 0.125)
    assert sa.sink_attn_device_status(True) == SA_ERR_BOUNDS
    data = workloads.make_prefill(5, [64, 64], 8, 1, 64)
    cu = data["cu_seqlens"].copy()
    cu[1] = 100                                 # a length above max_seqlen
    sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                         dev(cu), 64, 0.125)
    assert sa.sink_attn_device_status(True) == SA_ERR_BOUNDS
    _decode_ok(sa)


def test_bad_page_id_paged_prefill_is_reported():
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    d = workloads.make_mixed(6, [20, 1], [300, 40], 16, 2, 64)
    table = d["page_table"].copy()
    table[0, 2] = 1 << 20
    sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(table),
                               dev(d["cu_seqlens_q"]), dev(d["kv_lens"]), dev(d["sinks"]), 20, 0.125)
    assert sa.sink_attn_device_status(True) == SA_ERR_BOUNDS
    _decode_ok(sa)


def test_wait_that_never_completes_times_out():
    """A barrier nothing releases: the bounded wait gives up and reports."""
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    sa.sink_attn_selftest_wait_timeout(2_000_000)  # 2 ms
    assert sa.sink_attn_device_status(True) == SA_ERR_TIMEOUT
    _decode_ok(sa)


def test_zero_wait_budget_unwinds_cleanly():
    """With a zero wait budget the kernels may give up at their first wait; they
    must then unwind (drain their copies and MMAs, free TMEM) and report, and
    the next call with the normal budget must be correct."""
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    d = workloads.make_decode(7, [3000, 5000], 64, 8, 64)
    data = workloads.make_prefill(8, [700, 129], 16, 2, 64)
    try:
        sa.sink_attn_set_wait_timeout_ns(0)
        sa.sink_attn_decode(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
                            dev(d["kv_lens"]), dev(d["sinks"]), 0.125)
        sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                             dev(data["cu_seqlens"]), 700, 0.125)
        assert sa.sink_attn_device_status(True) in (SA_OK, SA_ERR_TIMEOUT)
    finally:
        sa.sink_attn_set_wait_timeout_ns(2_000_000_000)
    o, l = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]), dev(data["sinks"]),
                                dev(data["cu_seqlens"]), 700, 0.125)
    ro, rl = oracle.prefill(data["q"], data["k"], data["v"], data["sinks"], data["cu_seqlens"], 0.125, True)
    assert_close(host(o), host(l), ro, rl, "prefill after zero budget")
    _decode_ok(sa)


def test_zero_wait_budget_linear_unwinds_cleanly():
    """The linear layer's waits give up at once under a zero budget; its drains (MMAs
    before TMEM is freed, copies before shared memory is released) still wait, so the
    kernel ends cleanly and the next call with the normal budget is correct."""
    from oracle import moe
    sa = require_gpu()
    sa.sink_attn_device_status(True)
    d = workloads.make_linear(81, 1024, 2880, 1024)
    x, w, b = bf16(d["x"]), bf16(d["w"]), bf16(d["bias"])
    try:
        sa.sink_attn_set_wait_timeout_ns(0)
        sa.linear_bias(x, w, b)
        assert sa.sink_attn_device_status(True) in (SA_OK, SA_ERR_TIMEOUT)
    finally:
        sa.sink_attn_set_wait_timeout_ns(2_000_000_000)
    out = sa.linear_bias(x, w, b)
    rows = [0, 1, 511, 1023]
    ref = moe.linear_bias(d["x"][rows], d["w"], d["bias"])
    got = host(out)[rows]
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-2)
    assert sa.sink_attn_device_status(True) == SA_OK
