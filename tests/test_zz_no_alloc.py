"""sink_attn_decode_noalloc: split decode + merge with no device allocation.

Some callers cannot allocate device memory when they enqueue work (a plugin
that is only given its input and output buffers, a serving loop that forbids
cudaMalloc on its hot path because it may synchronise or fail).  For them the
library keeps the split partials in a fixed device array of its own.  This
file checks, through the C ABI, that the allocation-free call returns what the
allocating pair sink_attn_decode + sink_attn_merge returns, on two calls in a
row with different inputs (the second call must not see the first's leftovers
in the shared array), and that a request larger than the array is refused.

It is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_common import LSE_TOL, OUT_TOL, bf16, dev, host, max_err, out_err_beyond_bf16_store, require_gpu

pytestmark = pytest.mark.gpu

SA_ERR_CAPACITY = 9


def _inputs(seed, kv):
    d = workloads.make_decode(seed, kv, 64, 8, 64)
    return [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]


def test_noalloc_matches_decode_and_merge_twice_in_a_row():
    sa = require_gpu()
    cases = [(31, [4096] * 12 + [1, 17, 999], 8), (32, [300, 8000, 2, 5000], 32)]
    for seed, kv, splits in cases:
        args = _inputs(seed, kv)
        po, pl = sa.sink_attn_decode(*args, 0.125, num_splits=splits)
        ref_o, ref_l = sa.sink_attn_merge(po, pl)
        b = args[0].shape[0]
        out = torch.full((b, 64, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((b, 64), float("nan"), dtype=torch.float32, device="cuda")
        sa.sink_attn_decode_noalloc(*args, 0.125, num_splits=splits, out=out, lse=lse)
        torch.cuda.synchronize()
        assert out_err_beyond_bf16_store(host(out), host(ref_o)) <= OUT_TOL
        assert max_err(host(lse), host(ref_l)) <= LSE_TOL
        assert sa.sink_attn_device_status(True) == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    sa = require_gpu()
    lib = sa.load_library()
    fake = ctypes.c_void_p(0x10000)
    # 64 sequences x 256 splits x 64 heads x 65 floats > 2,097,152: refused before any launch
    st = lib.sink_attn_decode_noalloc(fake, fake, fake, fake, fake, fake, 64, 64, 8, 64, 16, 256, 16384,
                                      0.125, 256, fake, None, None)
    assert st == SA_ERR_CAPACITY
    assert "scratch" in sa.sink_attn_status_string(st)
