"""Capture of the hot path into a CUDA graph (decode + merge, on-chip split
decode, prefill) and replay: the launches take no host synchronisation, so a
captured step reproduces the eager results exactly."""
import numpy as np
import pytest
import torch

import workloads
from gpu_common import bf16, dev, require_gpu

pytestmark = pytest.mark.gpu


def test_decode_merge_and_prefill_in_one_graph():
    sa = require_gpu()
    d = workloads.make_decode(51, [4096] * 16 + [77, 1000], 64, 8, 64)
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]
    b = args[0].shape[0]
    po = torch.empty((b, 4, 64, 64), dtype=torch.float32, device="cuda")
    pl = torch.empty((b, 4, 64), dtype=torch.float32, device="cuda")
    out_split = torch.empty((b, 64, 64), dtype=torch.bfloat16, device="cuda")
    lse_split = torch.empty((b, 64), dtype=torch.float32, device="cuda")
    out_one = torch.empty_like(out_split)
    lse_one = torch.empty_like(lse_split)
    pf = workloads.make_prefill(52, [300, 129], 16, 2, 64)
    pq, pk, pv, ps, pcu = (bf16(pf["q"]), bf16(pf["k"]), bf16(pf["v"]), dev(pf["sinks"]),
                           dev(pf["cu_seqlens"]))
    pout = torch.empty_like(pq)
    plse = torch.empty((pq.shape[0], 16), dtype=torch.float32, device="cuda")

    def step():
        sa.sink_attn_decode(*args, 0.125, num_splits=4, out=po, lse=pl)
        sa.sink_attn_merge(po, pl, out=out_split, lse=lse_split)
        sa.sink_attn_decode(*args, 0.125, num_splits=1, out=out_one, lse=lse_one)
        sa.sink_attn_prefill(pq, pk, pv, ps, pcu, 300, 0.125, out=pout, lse=plse)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up: per-device lookups happen here
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out_split, lse_split, out_one, lse_one, pout, plse)]
    for t in (out_split, lse_split, out_one, lse_one, pout, plse):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in (out_split, lse_split, out_one, lse_one, pout, plse):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for e, t in zip(eager, (out_split, lse_split, out_one, lse_one, pout, plse)):
            assert torch.equal(e, t)
    assert sa.sink_attn_device_status(True) == 0


def test_single_sequence_cluster_decode_in_a_graph():
    """One sequence of 4096 tokens per step: the unsplit call splits each (sequence, KV head)
    across a 16-CTA cluster (8 where 16 cannot be resident) and merges on chip; 8 such steps
    over 8 sequences captured in one graph replay the eager results exactly."""
    sa = require_gpu()
    d = workloads.make_decode(53, [4096] * 8, 64, 8, 64)
    q, kp, vp, pt, kl, sk = (bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
                             dev(d["kv_lens"]), dev(d["sinks"]))
    assert sa.sink_attn_decode_splits(1, 8, 4096, 16, 152) == 1
    out = torch.empty((8, 64, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, 64), dtype=torch.float32, device="cuda")

    def steps():
        for i in range(8):
            sl = slice(i, i + 1)
            sa.sink_attn_decode(q[sl], kp, vp, pt[sl], kl[sl], sk, 0.125, num_splits=1, out=out[sl], lse=lse[sl])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        steps()                                  # eager first: the cluster-size query happens here
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = (out.clone(), lse.clone())
    # the whole batch in one call (clusters of 4) is the same attention
    o_all, l_all = sa.sink_attn_decode(q, kp, vp, pt, kl, sk, 0.125, num_splits=1)
    assert (o_all.float() - eager[0].float()).abs().max().item() <= 2e-2
    assert (l_all - eager[1]).abs().max().item() <= 1e-4
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        steps()
    for _ in range(2):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[0]) and torch.equal(lse, eager[1])
    assert sa.sink_attn_device_status(True) == 0
