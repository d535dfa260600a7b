"""Several host threads and streams using the library at once.

The calls keep no state between launches apart from per-device lookups (status word,
SM count, shared-memory opt-ins, the 16-CTA cluster capacity), which are filled once
under a lock or through atomics.  Four host threads, each on its own CUDA stream, run
split decode + merge, on-chip cluster decode and prefill on their own inputs at the same
time; every result must equal, bit for bit, the same call made alone.
"""
import threading

import pytest
import torch

import workloads
from gpu_common import bf16, dev, require_gpu

pytestmark = pytest.mark.gpu


def _inputs(seed):
    d = workloads.make_decode(seed, [4096, 1000 + 37 * seed, 17, 2500], 64, 8, 64)
    dec = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
           dev(d["kv_lens"]), dev(d["sinks"])]
    p = workloads.make_prefill(seed + 100, [300 + seed, 129, 640], 64, 8, 64)
    pre = [bf16(p["q"]), bf16(p["k"]), bf16(p["v"]), dev(p["sinks"]), dev(p["cu_seqlens"])]
    return dec, pre


def _work(sa, dec, pre, stream):
    """The calls of one thread, on `stream`; returns their outputs."""
    with torch.cuda.stream(stream):
        po, pl = sa.sink_attn_decode(*dec, 0.125, num_splits=5, stream=stream)
        mo, ml = sa.sink_attn_merge(po, pl, stream=stream)
        co, cl = sa.sink_attn_decode(*dec, 0.125, num_splits=1, stream=stream)
        one = [t[0:1] for t in (dec[0], dec[3], dec[4])]
        so, sl = sa.sink_attn_decode(one[0], dec[1], dec[2], one[1], one[2], dec[5], 0.125, num_splits=1,
                                     stream=stream)
        fo, fl = sa.sink_attn_prefill(*pre, 640, 0.125, stream=stream)
    return [mo, ml, co, cl, so, sl, fo, fl]


def test_threads_on_their_own_streams_match_single_calls():
    sa = require_gpu()
    n = 4
    data = [_inputs(70 + i) for i in range(n)]
    # each thread's calls made alone first (results compared later)
    alone = []
    for dec, pre in data:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        alone.append([t.clone() for t in _work(sa, dec, pre, s)])
        torch.cuda.synchronize()
    assert sa.sink_attn_device_status(True) == 0

    results = [None] * n
    errors = []
    start = threading.Barrier(n)

    def run(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            start.wait()
            outs = []
            for _ in range(5):  # several rounds, so the threads' launches interleave
                outs = _work(sa, data[i][0], data[i][1], s)
            s.synchronize()
            results[i] = outs
        except Exception as e:  # reported after the join
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    torch.cuda.synchronize()
    for i in range(n):
        assert results[i] is not None, f"thread {i} did not finish"
        for a, b in zip(alone[i], results[i]):
            assert torch.equal(a, b), f"thread {i}: result differs from the call made alone"
    assert sa.sink_attn_device_status(True) == 0
