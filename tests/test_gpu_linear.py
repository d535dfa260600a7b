"""GPU parity: bias-seeded tcgen05 linear layer against the fp64 oracle.

Error bound, from the arithmetic: bf16 x bf16 products are exact in fp32; the
tensor core accumulates K of them in fp32 starting from the bias, which (for
recursive summation, allowing truncation instead of rounding) errs by at most
K * 2^-23 * sum_k |x_k w_k|; the result is rounded once to bf16 (at most 2^-8
of its magnitude).  Each output must lie within that bound, and the RMS error
must stay below 2^-8 of the RMS output (a systematic mistake such as a dropped
K step or a shifted tile fails it even where the worst-case bound is loose)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_common import bf16, host, require_gpu
from oracle import moe, widen_bf16

pytestmark = pytest.mark.gpu


def _check(got, x, w, bias, rows=None, what=""):
    xs = x if rows is None else x[rows]
    ref = moe.linear_bias(xs, w, bias if bias is not None else np.zeros(w.shape[0], np.uint16))
    g = got if rows is None else got[rows]
    k = x.shape[1]
    mag = np.abs(widen_bf16(xs)) @ np.abs(widen_bf16(w)).T
    bound = 2.0 ** -8 * np.abs(ref) + k * 2.0 ** -23 * mag
    err = np.abs(g - ref)
    rms_err = float(np.sqrt(np.mean(err ** 2)))
    rms_ref = float(np.sqrt(np.mean(ref ** 2)))
    print(f"ERR linear {what}: max {err.max():.3e} rms {rms_err:.3e} (rms out {rms_ref:.3e})")
    assert np.all(err <= bound), f"{what}: {np.max(err - bound)} beyond the bound"
    assert rms_err <= 2.0 ** -8 * rms_ref


@pytest.mark.parametrize("m,n,k", [(128, 128, 64), (300, 200, 136), (1, 2880, 4096), (64, 128, 2880),
                                   (257, 5120, 2880), (129, 192, 8)])
@pytest.mark.parametrize("with_bias", [True, False])
def test_linear_bias_shapes(m, n, k, with_bias):
    sa = require_gpu()
    d = workloads.make_linear(51, m, n, k)
    bias = d["bias"] if with_bias else None
    out = sa.linear_bias(bf16(d["x"]), bf16(d["w"]), None if bias is None else bf16(bias))
    _check(host(out), d["x"], d["w"], bias, what=f"{m}x{n}x{k} bias={with_bias}")
    assert sa.sink_attn_device_status(True) == 0


def test_linear_many_tiles_per_cta_sampled():
    """Output projection shape, 4096 tokens x 2880 features x 4096 inputs: 480 tiles over
    the SMs, so every CTA reuses both accumulators several times; 96 sampled rows
    checked against the oracle, every row checked against cuBLAS within the same bound."""
    sa = require_gpu()
    m, n, k = 4096, 2880, 4096
    d = workloads.make_linear(52, m, n, k)
    x, w, b = bf16(d["x"]), bf16(d["w"]), bf16(d["bias"])
    out = sa.linear_bias(x, w, b)
    rows = np.sort(np.random.default_rng(7).choice(m, 96, replace=False))
    _check(host(out), d["x"], d["w"], d["bias"], rows=rows, what="4096x2880x4096")
    # the rest: against an fp32 library product of the same bf16 inputs
    ref = (x.float() @ w.float().T + b.float()).double()
    mag = x.float().abs() @ w.float().abs().T
    bound = 2.0 ** -8 * ref.abs() + 2 * k * 2.0 ** -23 * mag.double()
    assert bool(((out.double() - ref).abs() <= bound).all())
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("m,n,k", [(24037, 128, 640), (19500, 104, 2880), (20000, 64, 136)])
def test_linear_skinny_two_subtiles_sampled(m, n, k):
    """Skinny outputs (one column tile, N <= 128) with more 128-row blocks than SMs take
    256-row tiles: two 128-row sub-tiles read each W stage.  Rows sampled from both
    sub-tiles of many tiles and the ragged last tile are checked against the oracle,
    every row against cuBLAS within the same bound."""
    sa = require_gpu()
    d = workloads.make_linear(54, m, n, k)
    x, w, b = bf16(d["x"]), bf16(d["w"]), bf16(d["bias"])
    out = sa.linear_bias(x, w, b)
    rng = np.random.default_rng(8)
    edge = [0, 127, 128, 255, 256, 383, 384, m - 257, m - 129, m - 128, m - 2, m - 1]
    rows = np.unique(np.concatenate([rng.choice(m, 80, replace=False), np.array(edge)]))
    _check(host(out), d["x"], d["w"], d["bias"], rows=rows, what=f"{m}x{n}x{k} two sub-tiles")
    ref = (x.float() @ w.float().T + b.float()).double()
    mag = x.float().abs() @ w.float().abs().T
    bound = 2.0 ** -8 * ref.abs() + 2 * k * 2.0 ** -23 * mag.double()
    assert bool(((out.double() - ref).abs() <= bound).all())
    assert sa.sink_attn_device_status(True) == 0


def test_linear_bias_is_the_seed():
    """x = 0: every output is exactly the bias (the accumulator starts from it)."""
    sa = require_gpu()
    d = workloads.make_linear(53, 200, 384, 128)
    x = torch.zeros((200, 128), dtype=torch.bfloat16, device="cuda")
    out = sa.linear_bias(x, bf16(d["w"]), bf16(d["bias"]))
    assert torch.equal(out, bf16(d["bias"]).unsqueeze(0).expand(200, 384))


def test_linear_empty_rows():
    sa = require_gpu()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((64, 64), dtype=torch.bfloat16, device="cuda")
    assert sa.linear_bias(x, w).shape == (0, 64)
