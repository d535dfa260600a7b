"""The fp64 oracle against its pins, and plausible mistakes planted in it.

CPU only.  The pins are in ``oracle_pins.py``; each must pass on the oracle as
written, and each planted mistake (a mutant of the oracle, made on the CPU)
must make at least one pin fail.
"""
import math

import numpy as np
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def _mut_attention(transform):
    orig = oracle.attention_with_sink

    def mutant(q, k, v, sink, sm_scale, visible=None, with_sink=True, return_probs=False):
        return transform(orig, q, k, v, sink, sm_scale, visible, with_sink, return_probs)
    return mutant


def _sink_scaled(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    return orig(q, k, v, sink * sm_scale, sm_scale, visible, with_sink, rp)


def _sink_dropped(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    return orig(q, k, v, sink, sm_scale, visible, False, rp)


def _sink_in_every_split(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    return orig(q, k, v, sink, sm_scale, visible, True, rp)


def _sink_has_value_row(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    out, lse, p, ps = orig(q, k, v, sink, sm_scale, visible, with_sink, True)
    out = out + ps[:, None]
    return (out, lse, p, ps) if rp else (out, lse)


def _lse_log2(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    res = orig(q, k, v, sink, sm_scale, visible, with_sink, rp)
    return (res[0], res[1] / math.log(2)) + tuple(res[2:])


def _top_left_causal(q_len, kv_len, causal, rows=None):
    i = np.arange(q_len) if rows is None else np.asarray(rows)
    vis = np.ones((len(i), kv_len), dtype=bool)
    if causal:
        vis = np.arange(kv_len)[None, :] <= i[:, None]
    return vis


def _max_over_masked(orig, q, k, v, sink, sm_scale, visible, with_sink, rp):
    # the row max taken over the masked scores as well (the mask applied to the
    # exponentials afterwards): equal in exact arithmetic, but visible terms underflow
    # when a masked score is far above them
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, L = q.shape[0], k.shape[0]
    scores = sm_scale * (q @ k.T)
    x = np.concatenate([scores, np.full((n, 1), float(sink) if with_sink else -np.inf)], axis=1)
    m = x.max(axis=1, keepdims=True)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        e = np.exp(x - m)
    if visible is not None:
        e[:, :L] = np.where(visible, e[:, :L], 0.0)
    z = e.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        p_all = np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)
        lse = (m + np.log(np.where(z > 0, z, 1.0)))[:, 0]
    out = p_all[:, :L] @ v
    return (out, lse, p_all[:, :L], p_all[:, L]) if rp else (out, lse)


_ORIG_VISIBLE = oracle.visible_keys


def _visibility_of_first_row(q_len, kv_len, causal, rows=None):
    # every row of a block takes the mask of the block's first query
    vis = _ORIG_VISIBLE(q_len, kv_len, causal, rows)
    return np.broadcast_to(vis[:1], vis.shape).copy() if len(vis) else vis


_ORIG_LOCATE = oracle.locate_token


def _locate_left(cu, tok):
    # searchsorted to the left: a token that starts a sequence goes to the one before
    cu = np.asarray(cu, dtype=np.int64)
    b = max(0, int(np.searchsorted(cu, tok, side="left")) - 1)
    return b, int(tok - cu[b])


def _locate_global_index(cu, tok):
    b, _ = _ORIG_LOCATE(cu, tok)
    return b, int(tok)


_ORIG_DECODE = oracle.decode


def _decode_batches_by_position(*args, batches=None, **kw):
    # the restricted decode writes its n-th picked sequence to row n
    po, pl = _ORIG_DECODE(*args, batches=batches, **kw)
    if batches is None:
        return po, pl
    po2, pl2 = np.zeros_like(po), np.zeros_like(pl)
    for n, b in enumerate(batches):
        po2[n], pl2[n] = po[b], pl[b]
    return po2, pl2


def _gqa_modulo(h, hq, hkv):
    return h % hkv


def _split_drops_last_token(kv_len, page_size, num_splits):
    return [(a, max(a, b - 1) if b == kv_len and b > a else b)
            for a, b in _ORIG_SPLITS(kv_len, page_size, num_splits)]


_ORIG_SPLITS = oracle.split_token_ranges


def _online_d_starts_at_zero(q, k, v, sink, sm_scale, block):
    # the page's running denominator starts at 1 for the sink; this mutant forgets it
    q = np.asarray(q, dtype=np.float64)
    m, d, acc = float(sink), 0.0, np.zeros(np.asarray(v).shape[1])
    for start in range(0, len(k), block):
        s = sm_scale * (np.asarray(k[start:start + block]) @ q)
        m_new = max(m, float(s.max()))
        c = math.exp(m - m_new) if m != -math.inf else 0.0
        w = np.exp(s - m_new)
        d, acc, m = d * c + w.sum(), acc * c + w @ v[start:start + block], m_new
    return acc / d, m + math.log(d)


_ORIG_MERGE = oracle.merge


def _merge_posinf_as_finite(partial_o, partial_lse):
    # forgets the +inf case: weights e^(lse - max) with max = +inf
    po = np.asarray(partial_o, dtype=np.float64)
    pl = np.asarray(partial_lse, dtype=np.float64)
    m = pl.max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", over="ignore"):
        w = np.where(np.isneginf(pl), 0.0, np.exp(pl - np.where(np.isneginf(m), 0.0, m)))
        z = w.sum(axis=1, keepdims=True)
        lse = np.where(np.isneginf(m), -np.inf, m + np.log(np.where(z > 0, z, 1.0)))[:, 0]
        out = np.einsum("bsh,bshd->bhd", np.where(z > 0, w / np.where(z > 0, z, 1.0), 0.0), po)
    return out, lse


def _merge_empty_row_lse_zero(partial_o, partial_lse):
    # an all-empty row reports lse = 0 (log of the guard value) instead of -inf
    out, lse = _ORIG_MERGE(partial_o, partial_lse)
    return out, np.where(np.isneginf(lse), 0.0, lse)


MUTANTS = {
    "sink_scaled_by_sm_scale": ("attention_with_sink", _mut_attention(_sink_scaled)),
    "sink_dropped": ("attention_with_sink", _mut_attention(_sink_dropped)),
    "sink_in_every_split": ("attention_with_sink", _mut_attention(_sink_in_every_split)),
    "sink_has_value_row": ("attention_with_sink", _mut_attention(_sink_has_value_row)),
    "lse_in_log2": ("attention_with_sink", _mut_attention(_lse_log2)),
    "top_left_causal": ("visible_keys", _top_left_causal),
    "row_max_over_masked_scores": ("attention_with_sink", _mut_attention(_max_over_masked)),
    "gqa_modulo": ("kv_head_of", _gqa_modulo),
    "split_drops_last_token": ("split_token_ranges", _split_drops_last_token),
    "online_d_starts_at_zero": ("online_sink_attention", _online_d_starts_at_zero),
    "visibility_of_first_row": ("visible_keys", _visibility_of_first_row),
    "sequence_lookup_left": ("locate_token", _locate_left),
    "row_index_not_local": ("locate_token", _locate_global_index),
    "decode_batches_by_position": ("decode", _decode_batches_by_position),
    "merge_posinf_as_finite": ("merge", _merge_posinf_as_finite),
    "merge_empty_row_lse_zero": ("merge", _merge_empty_row_lse_zero),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oracle, attr, fn)
    failing = oracle_pins.failing_pins()
    assert failing, f"no pin catches the planted mistake {name}"


def test_pins_pass_unmutated():
    assert oracle_pins.failing_pins() == []
