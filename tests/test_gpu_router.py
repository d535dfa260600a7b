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
from oracle import widen_bf16
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


def test_router_with_projection_against_the_oracle_router():
    """The whole router: bias-seeded linear layer (router projection, bf16 logits) then
    Top-K softmax, against the oracle's composite (fp64 projection rounded to bf16).

    The decision rides on bf16 logits rounded from an fp32 (GPU) or fp64 (oracle) sum,
    which may land on different sides of a rounding boundary: the unique part is every
    row whose K-th and (K+1)-th oracle logits differ by more than twice the bound on
    the GPU logit error; there the experts and weights must match.  On the other rows
    the selection must be valid: no unselected expert beats a selected one by more than
    that bound, and the weights still form a descending softmax."""
    sa = require_gpu()
    t, e, hidden, k = 2048, 128, 2880, 4
    d = workloads.make_linear(26, t, e, hidden, std=1.0, w_std=0.05, bias_std=0.5)
    logits = sa.linear_bias(bf16(d["x"]), bf16(d["w"]), bf16(d["bias"]))
    idx, w = sa.moe_router_topk_softmax(logits, k)
    gidx, gw = idx.cpu().numpy(), host(w)
    ridx, rw, rlog = moe.router(d["x"], d["w"], d["bias"], k)
    exact = moe.linear_bias(d["x"], d["w"], d["bias"])
    mag = np.abs(widen_bf16(d["x"])) @ np.abs(widen_bf16(d["w"])).T
    # GPU logit error: fp32 accumulation (K 2^-23 sum|x w|) plus the bf16 rounding (2^-8 |l|)
    eb = (hidden * 2.0 ** -23 * mag + 2.0 ** -8 * np.abs(exact)).max(axis=1)
    srt = -np.sort(-rlog, axis=1)
    # unique rows: the K+1 largest logits (and so the selection and its order) are
    # separated by more than the logit error on both sides
    unique = np.all(-np.diff(srt[:, :k + 1], axis=1) > 2 * eb[:, None], axis=1)
    assert unique.sum() >= 256, "too few unambiguous rows to test"
    assert np.array_equal(gidx[unique], ridx[unique])
    # a logit error of up to eb moves a softmax weight by at most (e^(2 eb) - 1) of itself
    tol = (np.expm1(2 * eb[unique])[:, None] + W_REL) * np.abs(rw[unique]) + 1e-12
    assert np.all(np.abs(gw[unique] - rw[unique]) <= tol)
    for row in np.where(~unique)[0]:
        sel = set(gidx[row].tolist())
        assert len(sel) == k
        worst_sel = min(exact[row, list(sel)])
        best_unsel = max(exact[row, [c for c in range(e) if c not in sel]])
        assert best_unsel <= worst_sel + 2 * eb[row]
        assert np.all(np.diff(gw[row]) <= 0) and abs(gw[row].sum() - 1.0) <= k * 2.0 ** -8
    print(f"router end to end: {int(unique.sum())} of {t} rows unambiguous, all match")


@pytest.mark.parametrize("t,e,hidden,k", [(2048, 128, 2880, 4), (1000, 32, 2880, 4), (129, 64, 512, 2),
                                          (300, 256, 256, 8), (1, 128, 2880, 1), (777, 104, 640, 3),
                                          # more 128-row blocks than SMs: 256-row tiles (two sub-tiles)
                                          (24037, 128, 640, 4), (20000, 32, 256, 4), (19500, 64, 512, 2),
                                          (32768, 128, 2880, 4), (20000, 256, 256, 8),
                                          # eight slots, six selected
                                          (1000, 128, 512, 6), (24037, 104, 256, 5)])
def test_fused_router_is_projection_then_topk(t, e, hidden, k):
    """moe_router (projection with bias seeded in TMEM, bf16 logits, Top-K softmax in the
    epilogue) equals linear_bias followed by moe_router_topk_softmax bit for bit, counts
    included; the two-kernel path is tied to the oracle by the tests above."""
    sa = require_gpu()
    d = workloads.make_linear(27, t, e, hidden, std=1.0, w_std=0.05, bias_std=0.5)
    x, w, b = bf16(d["x"]), bf16(d["w"]), bf16(d["bias"])
    idx_f, w_f, c_f = sa.moe_router(x, w, b, k, return_counts=True)
    logits = sa.linear_bias(x, w, b)
    idx_u, w_u, c_u = sa.moe_router_topk_softmax(logits, k, return_counts=True)
    assert torch.equal(idx_f, idx_u) and torch.equal(w_f, w_u) and torch.equal(c_f, c_u)
    assert int(c_f.sum()) == t * k
    assert sa.sink_attn_device_status(True) == 0
