"""GPU parity: Top-K-then-softmax router against the fp64 oracle.

The Top-K decision is taken on the same bf16 logits on both sides, so expert
indices (and counts) must match bit for bit.  The weights are softmax values
computed in fp32 and stored as bf16: they may differ from the exact fp64 value
by the bf16 storage rounding (at most 2^-8 of the value) plus fp32 rounding
(below 1e-6 of the value)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_common import bf16, host, require_gpu
from oracle import moe

pytestmark = pytest.mark.gpu

W_REL = 2.0 ** -8 + 1e-6


def _check(sa, bits, k, rows=None):
    lg = bf16(bits)
    idx, w, counts = sa.moe_router_topk_softmax(lg, k, return_counts=True)
    torch.cuda.synchronize()
    ref_bits = bits if rows is None else bits[rows]
    ridx, rw = moe.router_topk_softmax(ref_bits, k)
    gidx = idx.cpu().numpy()
    gw = host(w)
    if rows is not None:
        gidx, gw = gidx[rows], gw[rows]
    assert np.array_equal(gidx, ridx), "expert indices differ"
    err = np.abs(gw - rw) - W_REL * np.abs(rw)
    print(f"ERR router k={k}: weight raw {np.abs(gw - rw).max():.3e} beyond-store {err.max():.3e}")
    assert err.max() <= 1e-12
    if rows is None:
        assert np.array_equal(counts.cpu().numpy(), moe.expert_counts(ridx, bits.shape[1]))
    else:
        assert int(counts.sum()) == bits.shape[0] * k
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("t,e,k", [(1000, 128, 4), (777, 32, 4), (300, 7, 3), (257, 256, 8),
                                   (64, 1, 1), (100, 33, 8), (5, 64, 1)])
def test_router_normal_logits(t, e, k):
    sa = require_gpu()
    _check(sa, workloads.make_router_logits(21, t, e, std=2.0), k)


@pytest.mark.parametrize("e,k", [(128, 4), (32, 4), (8, 8)])
def test_router_ties_lower_index_first(e, k):
    sa = require_gpu()
    _check(sa, workloads.make_router_logits(22, 600, e, levels=2), k)


def test_router_negative_zero_and_infinities():
    sa = require_gpu()
    bits = workloads.make_router_logits(23, 50, 16, levels=1)
    bits[:, 3] = 0x8000          # -0 ties with +0: the lower index wins
    bits[:, 5] = 0xFF80          # -inf never wins while a finite logit remains
    bits[0, :] = 0xFF80
    bits[0, 9] = 0x3F80          # one finite logit among -inf: weight 1, the rest 0
    _check(sa, bits, 4)


def test_router_empty_batch_clears_counts():
    sa = require_gpu()
    lg = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    counts = torch.full((32,), 7, dtype=torch.int32, device="cuda")
    sa.moe_router_topk_softmax(lg, 4, expert_counts=counts)
    assert int(counts.abs().sum()) == 0


def test_router_prefill_sized_batch_sampled():
    """32768 tokens x 128 experts, top 4 (one token per row of the causal-prefill
    workload); 512 sampled rows against the oracle, counts must total T * k."""
    sa = require_gpu()
    bits = workloads.make_router_logits(24, 32768, 128, std=2.0)
    rows = np.random.default_rng(5).choice(32768, 512, replace=False)
    _check(sa, bits, 4, rows=np.sort(rows))


def test_router_unaligned_logits_take_the_scalar_path():
    """Logits that start 2 bytes past a 16-byte boundary (a column slice of a wider
    tensor) are read element by element; the result is the same."""
    sa = require_gpu()
    bits = workloads.make_router_logits(25, 300, 129, std=2.0)
    lg = bf16(bits)[:, 1:]                       # [300, 128] view, row stride 129
    rows = lg.contiguous()                         # reference: aligned copy
    idx_a, w_a = sa.moe_router_topk_softmax(rows, 4)
    off = torch.empty(300 * 128 + 1, dtype=torch.bfloat16, device="cuda")
    shifted = off[1:].view(300, 128)               # 2-byte offset from the allocation
    shifted.copy_(rows)
    idx_b, w_b = sa.moe_router_topk_softmax(shifted, 4)
    assert torch.equal(idx_a, idx_b) and torch.equal(w_a, w_b)
    ridx, _ = moe.router_topk_softmax(bits[:, 1:], 4)
    assert np.array_equal(idx_b.cpu().numpy(), ridx)
