"""GPU parity: paged split-KV decode and merge against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import LSE_TOL, OUT_TOL, assert_close, bf16, dev, host, max_err, oracle_workers, require_gpu

pytestmark = pytest.mark.gpu


def _run(sa, d, scale, splits):
    args = [bf16(d["q"]), bf16(d["k_pages"]), bf16(d["v_pages"]), dev(d["page_table"]),
            dev(d["kv_lens"]), dev(d["sinks"])]
    o, l = sa.sink_attn_decode(*args, scale, num_splits=splits)
    return o, l, args


@pytest.mark.parametrize("hq,hkv", [(64, 8), (8, 8), (32, 8), (64, 4), (4, 1)])
@pytest.mark.parametrize("sink_fill", [None, -np.inf, 20.0])
def test_decode_small(hq, hkv, sink_fill):
    sa = require_gpu()
    kv = [1, 15, 16, 17, 129, 300, 1000, 2049]
    d = workloads.make_decode(7, kv, hq, hkv, 64, sink_fill=sink_fill)
    o, l, _ = _run(sa, d, 0.125, 1)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, f"decode hq={hq} hkv={hkv} sink={sink_fill}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("batch,kv,hq,hkv", [(1, 3000, 64, 8), (2, 777, 64, 8), (16, 2048, 64, 8),
                                             (64, 4096, 64, 8), (256, 600, 64, 8),
                                             # one wave: clusters of 16 (8 where 16 cannot be resident)
                                             (1, 4096, 64, 8), (3, 8192, 64, 8), (1, 4096, 64, 4),
                                             (2, 5000, 32, 8)])
def test_unsplit_decode_with_on_chip_cluster_split(batch, kv, hq, hkv):
    """num_splits == 1: each sequence's KV range may be split across a CTA cluster
    (sizes 1..16 depending on the shape) and merged on chip; parity with the oracle
    and with the explicit split + merge path."""
    sa = require_gpu()
    lens = [kv - (7 * b) % 50 for b in range(batch)]
    d = workloads.make_decode(17, lens, hq, hkv, 64)
    o, l, args = _run(sa, d, 0.125, 1)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125, batches=range(min(batch, 16)))
    n = min(batch, 16)
    assert_close(host(o)[:n], host(l)[:n], ro[:n], rl[:n], f"cluster decode batch={batch}")
    po, pl = sa.sink_attn_decode(*args, 0.125, num_splits=5)
    mo, ml = sa.sink_attn_merge(po, pl)
    assert_close(host(o), host(l), host(mo), host(ml), f"cluster vs split+merge batch={batch}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("splits", [2, 3, 7, 32, 200])
def test_decode_split_partials_and_merge(splits):
    sa = require_gpu()
    kv = [1, 16, 33, 500, 1777, 4096]
    d = workloads.make_decode(8, kv, 64, 8, 64)
    po, pl, _ = _run(sa, d, 0.125, splits)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125, num_splits=splits)
    # partials: same tolerance on o (fp32 output) and lse; empty splits are exactly (0, -inf)
    assert max_err(host(po), ro) <= OUT_TOL
    assert max_err(host(pl), rl) <= LSE_TOL
    empty = np.isneginf(rl)
    assert np.all(np.isneginf(host(pl)[empty])) and np.all(host(po)[empty] == 0)
    mo, ml = sa.sink_attn_merge(po, pl)
    fo, fl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125)
    assert_close(host(mo), host(ml), fo, fl, f"merged splits={splits}")


def test_merge_against_oracle_merge():
    sa = require_gpu()
    rng = np.random.default_rng(3)
    b, s, h = 5, 9, 16
    po = rng.standard_normal((b, s, h, 64)).astype(np.float32)
    pl = (rng.standard_normal((b, s, h)) * 3).astype(np.float32)
    pl[0, :, 0] = -np.inf                      # all splits empty: out 0, lse -inf
    pl[1, 3:, 2] = -np.inf                     # some empty
    pl[2, 4, 5] = np.inf                       # an infinite sink dominates
    mo, ml = sa.sink_attn_merge(dev(po), dev(pl))
    ro, rl = oracle.merge(po, pl)
    assert_close(host(mo), host(ml), ro, rl, "merge")


def test_paged_decode_config_full():
    """Paged decode at full size: 64 sequences x 4096 tokens, 64/8 heads, every row checked."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["paged_decode"]
    d = workloads.make_decode(cfg["seed"], [cfg["kv_len"]] * cfg["batch"], cfg["hq"], cfg["hkv"],
                              cfg["d"], cfg["page_size"], cfg["sink_std"])
    splits = sa.sink_attn_decode_splits(cfg["batch"], cfg["hkv"], cfg["kv_len"])
    po, pl, args = _run(sa, d, cfg["sm_scale"], splits)
    if splits > 1:
        o, l = sa.sink_attn_merge(po, pl)
    else:
        o, l = po, pl
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], cfg["sm_scale"])
    assert_close(host(o), host(l), ro, rl, "paged decode full")
    # the unsplit path gives the same answer within tolerance
    o1, l1 = sa.sink_attn_decode(*args, cfg["sm_scale"], num_splits=1)
    assert_close(host(o1), host(l1), ro, rl, "paged decode unsplit")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("sink_fill", [None, -np.inf, 20.0])
def test_long_decode_config_full(sink_fill):
    """Long-context split decode: 8 x 131072 tokens, 64/8 heads, 32 splits, merged; every
    sequence and head against the oracle, partials (split 0 alone carries the sink) too."""
    sa = require_gpu()
    cfg = workloads.WORKLOADS["long_decode"]
    d = workloads.make_decode(cfg["seed"], [cfg["kv_len"]] * cfg["batch"], cfg["hq"], cfg["hkv"],
                              cfg["d"], cfg["page_size"], cfg["sink_std"], sink_fill=sink_fill)
    po, pl, _ = _run(sa, d, cfg["sm_scale"], cfg["num_splits"])
    o, l = sa.sink_attn_merge(po, pl)
    assert sa.sink_attn_device_status(True) == 0
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], cfg["sm_scale"], num_splits=cfg["num_splits"],
                           workers=min(4, oracle_workers()))
    fo, fl = oracle.merge(ro, rl)
    assert_close(host(o), host(l), fo, fl, f"long decode 8x131072 sink={sink_fill} (all rows)")
    assert max_err(host(po), ro) <= OUT_TOL
    assert max_err(host(pl), rl) <= LSE_TOL
    del d, po, pl
    torch.cuda.empty_cache()


def test_page_permutation_is_bit_exact():
    """The same logical KV under two page permutations gives bitwise-identical output."""
    sa = require_gpu()
    kv = [5, 16, 100, 999, 2500]
    d1 = workloads.make_decode(9, kv, 64, 8, 64, permute=False)
    t2, _ = workloads.page_layout(1234, kv, 16, permute=True)
    k2 = np.zeros_like(d1["k_pages"])
    v2 = np.zeros_like(d1["v_pages"])
    for b, n in enumerate(kv):
        for j in range((n + 15) // 16):
            k2[t2[b, j]] = d1["k_pages"][d1["page_table"][b, j]]
            v2[t2[b, j]] = d1["v_pages"][d1["page_table"][b, j]]
    d2 = dict(d1, k_pages=k2, v_pages=v2, page_table=t2)
    for splits in (1, 4):
        o1, l1, _ = _run(sa, d1, 0.125, splits)
        o2, l2, _ = _run(sa, d2, 0.125, splits)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("hq,hkv", [(6, 2), (24, 2), (40, 8), (12, 1)])
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_odd_groups(hq, hkv, splits):
    """Group sizes 3, 12, 5, 12: the 8-wide MMA tiles are partly masked (two tiles above 8)."""
    sa = require_gpu()
    kv = [1, 17, 600, 2049]
    d = workloads.make_decode(19, kv, hq, hkv, 64)
    o, l, _ = _run(sa, d, 0.125, splits)
    if splits > 1:
        o, l = sa.sink_attn_merge(o, l)
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125)
    assert_close(host(o), host(l), ro, rl, f"decode group {hq // hkv} splits={splits}")
    assert sa.sink_attn_device_status(True) == 0


@pytest.mark.parametrize("batch,kv,splits", [(1, 131072, 32), (2, 65536, 16), (1, 20000, 8), (3, 9999, 3),
                                             (1, 4096, 2)])
def test_decode_small_grid_long_walks(batch, kv, splits):
    """Small grids whose warps walk long page ranges (64 pages per warp for one 131072-token
    sequence in 32 splits): every sequence against the oracle, partials included, and
    against the merged result of a different split count."""
    sa = require_gpu()
    lens = [kv - 13 * b for b in range(batch)]
    d = workloads.make_decode(23, lens, 64, 8, 64)
    po, pl, args = _run(sa, d, 0.125, splits)
    assert sa.sink_attn_device_status(True) == 0
    ro, rl = oracle.decode(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["kv_lens"],
                           d["sinks"], 0.125, num_splits=splits, workers=min(4, oracle_workers()))
    assert max_err(host(po), ro) <= OUT_TOL
    assert max_err(host(pl), rl) <= LSE_TOL
    mo, ml = sa.sink_attn_merge(po, pl)
    fo, fl = oracle.merge(ro, rl)
    assert_close(host(mo), host(ml), fo, fl, f"long walks batch={batch} kv={kv} splits={splits}")
    po2, pl2 = sa.sink_attn_decode(*args, 0.125, num_splits=splits + 1)
    mo2, ml2 = sa.sink_attn_merge(po2, pl2)
    assert_close(host(mo), host(ml), host(mo2), host(ml2), "long walks vs another split count")
