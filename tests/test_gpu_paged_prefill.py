"""GPU parity: mixed batches of new tokens over a paged KV cache."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close, bf16, dev, host, oracle_workers, require_gpu

pytestmark = pytest.mark.gpu


def _run(sa, d, max_q, scale, causal=True):
    return sa.sink_attn_prefill_paged(bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]),
                                      dev(d["page_table"]), dev(d["cu_seqlens_q"]), dev(d["kv_lens"]),
                                      dev(d["sinks"]), max_q, scale, causal=causal)


@pytest.mark.parametrize("causal", [True, False])
def test_paged_prefill_small(causal):
    sa = require_gpu()
    q_lens = [1, 5, 128, 129, 300, 1]
    kv_lens = [1, 40, 128, 700, 300, 2000]
    d = workloads.make_mixed(3, q_lens, kv_lens, 64, 8, 64)
    o, l = _run(sa, d, max(q_lens), 0.125, causal)
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"],
                                  d["cu_seqlens_q"], d["kv_lens"], d["sinks"], 0.125, causal)
    assert_close(host(o), host(l), ro, rl, f"paged prefill causal={causal}")
    assert sa.sink_attn_device_status(True) == 0


def test_ragged_mixed_config():
    """32 sequences, KV log-uniform in [1, 32768], decode rows and 128-2048 token chunks:
    every new token of every sequence, every head, against the oracle."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["ragged_mixed"]
    q_lens, kv_lens = workloads.ragged_mixed_lengths(cfg["seed"] + 2, cfg["num_seqs"], cfg["max_kv"])
    d = workloads.make_mixed(cfg["seed"], q_lens, kv_lens, cfg["hq"], cfg["hkv"], cfg["d"],
                             cfg["page_size"], cfg["sink_std"])
    o, l = _run(sa, d, int(q_lens.max()), cfg["sm_scale"])
    assert sa.sink_attn_device_status(True) == 0
    ro, rl = oracle.prefill_paged(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["cu_seqlens_q"],
                                  d["kv_lens"], d["sinks"], cfg["sm_scale"], True, workers=oracle_workers())
    assert_close(host(o), host(l), ro, rl, "ragged mixed (all rows)")


def test_paged_prefill_matches_contiguous_prefill_bitwise():
    """With kv_len == q_len and an identity page table the paged kernel sees the same
    keys in the same order as the contiguous one, so the outputs are bit-identical."""
    sa = require_gpu()
    lens = [300, 64]
    data = workloads.make_prefill(11, lens, 16, 2, 64)
    o1, l1 = sa.sink_attn_prefill(bf16(data["q"]), bf16(data["k"]), bf16(data["v"]),
                                  dev(data["sinks"]), dev(data["cu_seqlens"]), 300, 0.125)
    table, num_pages = workloads.page_layout(0, lens, 16, permute=True)
    kp = np.zeros((num_pages, 2, 16, 64), dtype=np.uint16)
    vp = np.zeros_like(kp)
    cu = data["cu_seqlens"]
    for b, n in enumerate(lens):
        for j in range(n):
            kp[table[b, j // 16], :, j % 16] = data["k"][cu[b] + j]
            vp[table[b, j // 16], :, j % 16] = data["v"][cu[b] + j]
    d = dict(q=data["q"], k_pages=kp, v_pages=vp, page_table=table, cu_seqlens_q=cu,
             kv_lens=np.array(lens, dtype=np.int32), sinks=data["sinks"])
    o2, l2 = _run(sa, d, 300, 0.125)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
