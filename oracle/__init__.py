"""fp64 CPU oracle for attention with softmax sinks.  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use this
package.  The library never calls it; it shares no code with the CUDA path.

What it computes follows the page "GPT-OSS on day 0" (Perplexity, 2025),
section "Kernels for GPT-OSS / Sink Attention":

* the operation is ``attn = softmax(q k^T * sm_scale + sink) V`` where each
  attention head owns one pretrained sink value that enters the softmax
  (the same page, model overview: "each attention head has a pretrained sink
  parameter factored into the softmax");
* the online algorithm on that page starts the running max ``m`` at the head's
  sink and the running denominator ``d`` at 1, i.e. the state after seeing one
  extra logit equal to the sink that carries no value row; when the KV range is
  split into blocks, that seed belongs to the first block only.

Readings taken where the page is silent (each is also listed in the design notes):

1. the sink is one extra logit column per (query row, head): it adds
   ``exp(sink - M)`` to the denominator and no row of V;
2. ``sm_scale`` multiplies ``q . k`` only, never the sink;
3. query head ``h`` reads KV head ``h // (Hq / Hkv)`` (contiguous groups);
4. causal masking is bottom-right aligned: with ``q_len`` new tokens at the
   end of a ``kv_len`` cache, query ``i`` sees keys ``j <= i + kv_len - q_len``;
5. ``lse`` is the natural log of the denominator in scaled-logit units,
   including the sink term: ``lse = M + ln Z``;
6. a split-KV partial covers pages ``[s c, min((s+1) c, n_pages))`` with
   ``c = ceil(n_pages / S)``; only split 0 holds the sink column; an empty
   split without sink is ``(o, lse) = (0, -inf)``;
7. splits are combined with the log-sum-exp merge
   ``lse = log sum_s exp(lse_s)``, ``o = sum_s exp(lse_s - lse) o_s``;
8. a row with no visible key and sink = -inf has ``o = 0, lse = -inf``;
   a sink of +inf gives ``o = 0, lse = +inf``.

Every number is fp64; bf16 inputs are widened exactly.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "widen_bf16", "kv_head_of", "visible_keys", "locate_token", "sequence_head",
    "attention_with_sink", "online_sink_attention", "prefill", "gather_pages", "prefill_paged",
    "split_token_ranges", "decode", "merge",
]


# ---------------------------------------------------------------- inputs
def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("expected uint16 bf16 bit patterns")
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    return widen_bf16(x) if x.dtype == np.uint16 else x.astype(np.float64)


# ---------------------------------------------------------------- readings 3 and 4
def kv_head_of(h: int, num_qo_heads: int, num_kv_heads: int) -> int:
    """Query head h reads KV head h // (Hq / Hkv) (reading 3)."""
    return h // (num_qo_heads // num_kv_heads)


def visible_keys(q_len: int, kv_len: int, causal: bool, rows=None) -> np.ndarray:
    """Boolean [q_len, kv_len]: key j visible to query i (reading 4, bottom-right).

    With ``rows`` (query indices within the sequence) only those rows are built:
    [len(rows), kv_len].
    """
    i = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    j = np.arange(kv_len)[None, :]
    if not causal:
        return np.ones((len(i), kv_len), dtype=bool)
    return j <= i[:, None] + (kv_len - q_len)


def locate_token(cu_seqlens, tok: int):
    """(sequence b, index i of the token within b) for a flat token index.

    Sequence b owns tokens [cu[b], cu[b+1]); an empty sequence owns none, so the
    owner is the last b whose start is <= tok.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    b = int(np.searchsorted(cu, tok, side="right") - 1)
    return b, int(tok - cu[b])


def _rows_per_block(kv_len: int) -> int:
    """Query rows per block, so that a block's score matrix holds about 2^22 entries."""
    return max(1, (1 << 22) // max(1, kv_len))


def sequence_head(q, k, v, sink, sm_scale, q_len: int, kv_len: int, causal: bool, rows=None):
    """Rows of one (sequence, head): q [n, D] holds the query rows ``rows`` (indices
    within the sequence, all of them when None); k, v [kv_len, D].

    Rows are independent, so they are taken a block of rows at a time; a block's
    score matrix stops after the last key any of its rows can see (the keys after
    it are masked for every row of the block and would add exact zeros).
    """
    idx = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    d = np.asarray(v).shape[-1]
    out = np.zeros((len(idx), d))
    lse = np.zeros(len(idx))
    step = _rows_per_block(kv_len)
    for r0 in range(0, len(idx), step):
        sel = idx[r0:r0 + step]
        last = kv_len
        if causal and len(sel):
            last = max(0, min(kv_len, int(sel.max()) + kv_len - q_len + 1))
        vis = visible_keys(q_len, kv_len, causal, rows=sel)[:, :last]
        o, l = attention_with_sink(q[r0:r0 + step], k[:last], v[:last], sink, sm_scale, vis)
        out[r0:r0 + len(sel)], lse[r0:r0 + len(sel)] = o, l
    return out, lse


def _run_units(fn, units, workers: int):
    """fn over independent units, on ``workers`` threads (numpy releases the GIL)."""
    units = list(units)
    if workers <= 1 or len(units) <= 1:
        return [fn(u) for u in units]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, units))


# ---------------------------------------------------------------- the definition
def attention_with_sink(q, k, v, sink, sm_scale, visible=None, with_sink=True,
                        return_probs=False):
    """Sink attention for a block of query rows of one head, by definition.

    q [n, D], k [L, D], v [L, D] (float64), sink a scalar, visible [n, L] bool.
    The full score matrix is built with one extra column holding the sink
    (readings 1, 2); the softmax runs over each row of that matrix; the sink
    column has no value row.  Returns out [n, D], lse [n] (and, if asked,
    p [n, L] and p_sink [n]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, L = q.shape[0], k.shape[0]
    scores = sm_scale * (q @ k.T)                                     # [n, L]
    if visible is not None:
        scores = np.where(visible, scores, -np.inf)
    sink_col = np.full((n, 1), float(sink) if with_sink else -np.inf)
    x = np.concatenate([scores, sink_col], axis=1)                   # [n, L + 1]
    m = x.max(axis=1, keepdims=True)                                  # [n, 1]
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(x - m_safe)
    # rows whose max is +inf: only +inf entries carry weight (reading 8)
    e = np.where(np.isposinf(m) & ~np.isposinf(x), 0.0, e)
    e = np.where(np.isposinf(m) & np.isposinf(x), 1.0, e)
    z = e.sum(axis=1, keepdims=True)                                  # [n, 1]
    with np.errstate(invalid="ignore", divide="ignore"):
        p_all = np.where(z > 0, e / np.where(z > 0, z, 1.0), 0.0)
        lse = np.where(finite, m + np.log(np.where(z > 0, z, 1.0)), m)[:, 0]
    p = p_all[:, :L]
    p_sink = p_all[:, L]
    out = p @ v if L else np.zeros((n, v.shape[1] if v.ndim == 2 else q.shape[1]))
    if return_probs:
        return out, lse, p, p_sink
    return out, lse


def online_sink_attention(q, k, v, sink, sm_scale, block: int):
    """The page's online algorithm for one query row, in its order.

    The running max ``m`` starts at the sink and the running denominator ``d``
    at 1 (0 when the sink is -inf, the limit of exp(sink - sink)); keys are
    visited in blocks of ``block``; for each block the max is updated, the old
    state is rescaled by ``exp(m_old - m_new)`` and the block's terms are added.
    Used by the tests to show the page's algorithm reaches the definition.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m = float(sink)
    d = 0.0 if m == -math.inf else 1.0
    acc = np.zeros(v.shape[1])
    for start in range(0, k.shape[0], block):
        s = sm_scale * (k[start:start + block] @ q)
        m_new = max(m, float(s.max()))
        if m_new == -math.inf:
            continue
        scale_old = math.exp(m - m_new) if m != -math.inf else 0.0
        w = np.exp(s - m_new)
        d = d * scale_old + float(w.sum())
        acc = acc * scale_old + w @ v[start:start + block]
        m = m_new
    if d == 0.0:
        return np.zeros_like(acc), -math.inf
    return acc / d, m + math.log(d)


# ---------------------------------------------------------------- contiguous prefill
def prefill(q, k, v, sinks, cu_seqlens, sm_scale, causal=True, rows=None, workers=1):
    """Ragged contiguous prefill (q_len == kv_len per sequence).

    q [T, Hq, D], k/v [T, Hkv, D] (bf16 bits or floats), sinks [Hq],
    cu_seqlens [B+1].  Returns out [T, Hq, D], lse [T, Hq] in fp64.  With
    ``rows`` (a list of (token, head)), only those rows are computed and the
    results come back as arrays [len(rows), D] and [len(rows)].  ``workers``
    threads share the (sequence, head) units.
    """
    qf, kf, vf = _as_f64(q), _as_f64(k), _as_f64(v)
    sinks = np.asarray(sinks, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    t, hq, d = qf.shape
    hkv = kf.shape[1]
    if rows is not None:
        groups = {}
        for r, (tok, h) in enumerate(rows):
            b, i = locate_token(cu, int(tok))
            groups.setdefault((b, int(h)), []).append((r, i))
        out = np.zeros((len(rows), d))
        lse = np.zeros(len(rows))
    else:
        groups = {(b, h): None for b in range(len(cu) - 1) if cu[b + 1] > cu[b] for h in range(hq)}
        out = np.zeros((t, hq, d))
        lse = np.zeros((t, hq))

    def unit(key):
        b, h = key
        lo, hi = int(cu[b]), int(cu[b + 1])
        g = kv_head_of(h, hq, hkv)
        sel = None if groups[key] is None else [i for _, i in groups[key]]
        qrows = qf[lo:hi, h] if sel is None else qf[lo + np.asarray(sel, dtype=np.int64), h]
        return sequence_head(qrows, kf[lo:hi, g], vf[lo:hi, g], sinks[h], sm_scale,
                             hi - lo, hi - lo, causal, sel)

    for key, (o, l) in zip(groups, _run_units(unit, groups, workers)):
        b, h = key
        if groups[key] is None:
            lo, hi = int(cu[b]), int(cu[b + 1])
            out[lo:hi, h], lse[lo:hi, h] = o, l
        else:
            for n, (r, _) in enumerate(groups[key]):
                out[r], lse[r] = o[n], l[n]
    return out, lse


# ---------------------------------------------------------------- paged KV
def gather_pages(pages, page_table_row, kv_len, page_size=None):
    """Logical [kv_len, Hkv, D] view of one sequence from pages [P, Hkv, page, D]."""
    pages = np.asarray(pages)
    ps = pages.shape[2] if page_size is None else page_size
    idx = np.arange(kv_len)
    phys = np.asarray(page_table_row)[idx // ps]
    if kv_len and (phys.min() < 0 or phys.max() >= pages.shape[0]):
        raise IndexError("page id out of range")
    return pages[phys, :, idx % ps, :]                 # [kv_len, Hkv, D]


def prefill_paged(q, k_pages, v_pages, page_table, cu_seqlens_q, kv_lens, sinks, sm_scale,
                  causal=True, rows=None, workers=1):
    """Mixed batch over a paged cache: sequence b has q_len new tokens, the last
    q_len of its kv_len cached tokens (reading 4).  q [Tq, Hq, D].  ``rows`` and
    ``workers`` as for ``prefill``."""
    qf = _as_f64(q)
    sinks = np.asarray(sinks, dtype=np.float64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    t, hq, d = qf.shape
    hkv = np.asarray(k_pages).shape[1]
    if rows is not None:
        groups = {}
        for r, (tok, h) in enumerate(rows):
            b, i = locate_token(cu, int(tok))
            groups.setdefault((b, int(h)), []).append((r, i))
        out = np.zeros((len(rows), d))
        lse = np.zeros(len(rows))
    else:
        groups = {(b, h): None for b in range(len(cu) - 1) if cu[b + 1] > cu[b] for h in range(hq)}
        out = np.zeros((t, hq, d))
        lse = np.zeros((t, hq))
    cache = {}

    def kv_of(b):
        if b not in cache:
            kv_len = int(kv_lens[b])
            cache[b] = (_as_f64(gather_pages(k_pages, page_table[b], kv_len)),
                        _as_f64(gather_pages(v_pages, page_table[b], kv_len)))
        return cache[b]

    for b in sorted({b for b, _ in groups}):
        kv_of(b)

    def unit(key):
        b, h = key
        lo, hi = int(cu[b]), int(cu[b + 1])
        kb, vb = kv_of(b)
        g = kv_head_of(h, hq, hkv)
        sel = None if groups[key] is None else [i for _, i in groups[key]]
        qrows = qf[lo:hi, h] if sel is None else qf[lo + np.asarray(sel, dtype=np.int64), h]
        return sequence_head(qrows, kb[:, g], vb[:, g], sinks[h], sm_scale,
                             hi - lo, int(kv_lens[b]), causal, sel)

    for key, (o, l) in zip(groups, _run_units(unit, groups, workers)):
        b, h = key
        if groups[key] is None:
            lo, hi = int(cu[b]), int(cu[b + 1])
            out[lo:hi, h], lse[lo:hi, h] = o, l
        else:
            for n, (r, _) in enumerate(groups[key]):
                out[r], lse[r] = o[n], l[n]
    return out, lse


# ---------------------------------------------------------------- split-KV decode and merge
def split_token_ranges(kv_len: int, page_size: int, num_splits: int):
    """Token range of each split (reading 6): pages [s c, min((s+1) c, n)), c = ceil(n / S)."""
    n_pages = (kv_len + page_size - 1) // page_size
    c = (n_pages + num_splits - 1) // num_splits if n_pages else 0
    ranges = []
    for s in range(num_splits):
        p0, p1 = min(s * c, n_pages), min((s + 1) * c, n_pages)
        ranges.append((min(p0 * page_size, kv_len), min(p1 * page_size, kv_len)))
    return ranges


def decode(q, k_pages, v_pages, page_table, kv_lens, sinks, sm_scale, num_splits=1, batches=None,
           workers=1):
    """One new token per sequence over a paged cache.

    q [B, Hq, D].  With num_splits == 1 returns out [B, Hq, D], lse [B, Hq].
    With num_splits > 1 returns the partials o [B, S, Hq, D], lse [B, S, Hq]:
    split s attends to its own token range, and only split 0 has the sink
    column (the page's rule that the seeded max belongs to the first block).
    ``batches`` restricts the work to some sequences (other rows stay 0);
    ``workers`` threads share the sequences.
    """
    qf = _as_f64(q)
    sinks = np.asarray(sinks, dtype=np.float64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    bsz, hq, d = qf.shape
    hkv = np.asarray(k_pages).shape[1]
    ps = np.asarray(k_pages).shape[2]
    po = np.zeros((bsz, num_splits, hq, d))
    pl = np.zeros((bsz, num_splits, hq))

    def unit(b):
        kv_len = int(kv_lens[b])
        kb = _as_f64(gather_pages(k_pages, page_table[b], kv_len))
        vb = _as_f64(gather_pages(v_pages, page_table[b], kv_len))
        for s, (t0, t1) in enumerate(split_token_ranges(kv_len, ps, num_splits)):
            for h in range(hq):
                g = kv_head_of(h, hq, hkv)
                o, l = attention_with_sink(qf[b, h][None], kb[t0:t1, g], vb[t0:t1, g], sinks[h],
                                           sm_scale, None, with_sink=(s == 0))
                po[b, s, h], pl[b, s, h] = o[0], l[0]

    _run_units(unit, range(bsz) if batches is None else batches, workers)
    if num_splits == 1:
        return po[:, 0], pl[:, 0]
    return po, pl


def merge(partial_o, partial_lse):
    """Combine split partials (reading 7).  partial_o [B, S, H, D], partial_lse [B, S, H]."""
    po = np.asarray(partial_o, dtype=np.float64)
    pl = np.asarray(partial_lse, dtype=np.float64)
    m = pl.max(axis=1, keepdims=True)                                 # [B, 1, H]
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isneginf(pl), 0.0, np.exp(pl - m_safe))
    w = np.where(np.isposinf(m), np.where(np.isposinf(pl), 1.0, 0.0), w)
    z = w.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = np.where(finite, m_safe + np.log(np.where(z > 0, z, 1.0)), m)[:, 0]
        lse = np.where(finite[:, 0] & (z[:, 0] == 0), -np.inf, lse)
        wn = np.where(z > 0, w / np.where(z > 0, z, 1.0), 0.0)
    out = np.einsum("bsh,bshd->bhd", wn, po)
    return out, lse
