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


def _pair_and_noalloc(sa, args, splits, b, hq):
    po, pl = sa.sink_attn_decode(*args, 0.125, num_splits=splits)
    ref_o, ref_l = sa.sink_attn_merge(po, pl)
    out = torch.full((b, hq, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b, hq), float("nan"), dtype=torch.float32, device="cuda")
    sa.sink_attn_decode_noalloc(*args, 0.125, num_splits=splits, out=out, lse=lse)
    torch.cuda.synchronize()
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("hq,hkv,kv,splits", [
    (64, 8, [4096] * 6 + [1, 17, 0, 999], 4),      # group 8; an empty sequence
    (64, 4, [3000, 64, 2049], 3),                  # group 16 (two 8-wide query tiles)
    (32, 8, [5000, 333], 2),                       # group 4
    (64, 8, [8192, 1000, 16], 33),                 # more splits than a warp's lanes; empty splits
    (16, 16, [700, 4096], 16),                     # no grouping
])
def test_noalloc_is_decode_then_merge_bit_for_bit(hq, hkv, kv, splits):
    """The allocation-free call runs the same split decode and merge kernels on the
    library's scratch, so its result equals sink_attn_decode + sink_attn_merge exactly,
    lse included, across group sizes, split counts above a warp's lanes, empty
    sequences and splits, and -inf / large sinks."""
    sa = require_gpu()
    d = workloads.make_decode(40 + splits, kv, hq, hkv, 64)
    sinks = d["sinks"].copy()
    sinks[0] = -np.inf  # ordinary softmax for head 0
    sinks[1] = 20.0     # a sink that takes almost all the weight
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(sinks)]
    out, lse, ref_o, ref_l = _pair_and_noalloc(sa, args, splits, len(kv), hq)
    assert torch.equal(out, ref_o)
    assert torch.equal(lse, ref_l)
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
