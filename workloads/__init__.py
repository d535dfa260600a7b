"""Seeded synthetic inputs for the sink-attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the fp64 oracle and the GPU path consume the exact
bytes produced here, so a parity test compares the two on identical inputs.

Shapes follow the GPT-OSS attention layout described on the page "GPT-OSS on
day 0" (Perplexity, 2025), section "Kernels for GPT-OSS / Sink Attention":
grouped-query attention with one pretrained sink logit per query head.  Sizes
of the five workloads (query/KV head counts, head_dim 64, page size 16, batch
and lengths) are listed in ``WORKLOADS``.

Conventions
-----------
* bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
  from float32 normal draws).  Whoever consumes them widens them exactly.
* Normal draws are made in independent chunks of ``CHUNK`` elements, chunk
  ``c`` of stream ``s`` coming from ``numpy.random.default_rng([seed, s, c])``.
  The result therefore does not depend on how many threads generate it.
* Paged KV caches use the layout ``[num_pages, num_kv_heads, page_size,
  head_dim]``; ``page_table[b, j]`` is the physical page holding logical tokens
  ``[16 j, 16 j + 16)`` of sequence ``b``; unused entries are ``-1``.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22

# stream ids: one per tensor role, so tensors never share random numbers
STREAM_Q, STREAM_K, STREAM_V, STREAM_SINK, STREAM_PERM, STREAM_LENS = 1, 2, 3, 4, 5, 6
STREAM_LOGITS, STREAM_QKV, STREAM_BIAS, STREAM_X, STREAM_W = 7, 8, 9, 10, 11


def _round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    u = x.view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def _normal_chunk(seed: int, stream: int, chunk: int, count: int, std: float) -> np.ndarray:
    rng = np.random.default_rng([seed, stream, chunk])
    x = rng.standard_normal(count, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return _round_to_bf16_bits(x)


def normal_bf16(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws with the given shape (chunked, thread-parallel)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        out[lo:hi] = _normal_chunk(seed, stream, c, hi - lo, std)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (used by harness code to build tensors)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def sinks_f32(seed: int, num_heads: int, std: float = 1.0, fill: float | None = None) -> np.ndarray:
    """Per-head sink logits, fp32.  ``fill`` overrides the draw (e.g. -inf or +20)."""
    if fill is not None:
        return np.full(num_heads, fill, dtype=np.float32)
    rng = np.random.default_rng([seed, STREAM_SINK])
    return (rng.standard_normal(num_heads, dtype=np.float32) * np.float32(std)).astype(np.float32)


def cu_seqlens_from(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    return cu


def page_layout(seed: int, kv_lens, page_size: int = 16, permute: bool = True, extra_pages: int = 0):
    """Page table for sequences with the given KV lengths.

    Logical pages of all sequences are numbered consecutively, then mapped to
    physical page ids through a seeded random permutation (identity if
    ``permute`` is false).  Returns ``(page_table int32 [B, max_pages],
    num_pages)``; unused entries are -1.
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    npages = (kv_lens + page_size - 1) // page_size
    total = int(npages.sum())
    num_pages = total + extra_pages
    if permute:
        perm = np.random.default_rng([seed, STREAM_PERM]).permutation(num_pages)[:total]
    else:
        perm = np.arange(total)
    max_pages = max(1, int(npages.max()) if len(npages) else 1)
    table = np.full((len(kv_lens), max_pages), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[pos:pos + n]
        pos += int(n)
    return table, num_pages


def ragged_mixed_lengths(seed: int, num_seqs: int = 32, max_kv: int = 32768,
                         q_lo: int = 128, q_hi: int = 2048):
    """Lengths of the ragged mixed batch.

    Per sequence: kv_len = floor(exp(U(0, ln max_kv))) clamped to [1, max_kv];
    with probability 1/2 the sequence is a decode row (q_len = 1), otherwise a
    prefill chunk with q_len ~ U{q_lo..q_hi}; q_len = min(q_len, kv_len).  The
    new tokens are the last q_len positions of the KV cache.
    """
    rng = np.random.default_rng([seed, STREAM_LENS])
    kv = np.floor(np.exp(rng.uniform(0.0, math.log(max_kv), num_seqs))).astype(np.int64)
    kv = np.clip(kv, 1, max_kv)
    is_decode = rng.uniform(0.0, 1.0, num_seqs) < 0.5
    q = rng.integers(q_lo, q_hi + 1, num_seqs)
    q = np.where(is_decode, 1, q)
    q = np.minimum(q, kv)
    return q.astype(np.int32), kv.astype(np.int32)


# --------------------------------------------------------------------------
# The five workloads.  Sizes: query heads / KV heads / head_dim follow the
# GPT-OSS attention shape (64 / 8 / 64) except the tiny case.
# --------------------------------------------------------------------------
WORKLOADS = {
    "tiny_prefill": dict(kind="prefill", batch=1, seqlen=128, causal=True, hq=4, hkv=1, d=64,
                         sink_std=1.0, sm_scale=0.125, seed=0),
    "paged_decode": dict(kind="decode", batch=64, kv_len=4096, hq=64, hkv=8, d=64, page_size=16,
                         sink_std=1.0, sm_scale=0.125, seed=0),
    "causal_prefill": dict(kind="prefill", batch=4, seqlen=8192, causal=True, hq=64, hkv=8, d=64,
                           sink_std=math.sqrt(2.0), sm_scale=0.125, seed=0),
    "long_decode": dict(kind="decode", batch=8, kv_len=131072, hq=64, hkv=8, d=64, page_size=16,
                        num_splits=32, sink_std=1.0, sm_scale=0.125, seed=0),
    "ragged_mixed": dict(kind="mixed", num_seqs=32, max_kv=32768, causal=True, hq=64, hkv=8, d=64,
                         page_size=16, sink_std=1.0, sm_scale=0.125, seed=0),
}


def make_prefill(seed: int, seqlens, hq: int, hkv: int, d: int, sink_std: float = 1.0,
                 sink_fill: float | None = None):
    """Contiguous ragged prefill inputs: q [T,Hq,D], k/v [T,Hkv,D] (bf16 bits)."""
    cu = cu_seqlens_from(seqlens)
    t = int(cu[-1])
    return dict(
        q=normal_bf16(seed, STREAM_Q, (t, hq, d)),
        k=normal_bf16(seed, STREAM_K, (t, hkv, d)),
        v=normal_bf16(seed, STREAM_V, (t, hkv, d)),
        sinks=sinks_f32(seed, hq, sink_std, sink_fill),
        cu_seqlens=cu,
    )


def make_paged_kv(seed: int, kv_lens, hkv: int, d: int, page_size: int = 16, permute: bool = True,
                  extra_pages: int = 0):
    """Paged K/V caches [num_pages, Hkv, page_size, D] (bf16 bits) plus the page table."""
    table, num_pages = page_layout(seed + 1, kv_lens, page_size, permute, extra_pages)
    shape = (num_pages, hkv, page_size, d)
    return dict(
        k_pages=normal_bf16(seed, STREAM_K, shape),
        v_pages=normal_bf16(seed, STREAM_V, shape),
        page_table=table,
        kv_lens=np.asarray(kv_lens, dtype=np.int32),
        num_pages=num_pages,
    )


def make_decode(seed: int, kv_lens, hq: int, hkv: int, d: int, page_size: int = 16,
                sink_std: float = 1.0, sink_fill: float | None = None, permute: bool = True):
    """Decode inputs: one new query token per sequence, q [B,Hq,D], over a paged KV cache."""
    kv = make_paged_kv(seed, kv_lens, hkv, d, page_size, permute)
    kv["q"] = normal_bf16(seed, STREAM_Q, (len(kv_lens), hq, d))
    kv["sinks"] = sinks_f32(seed, hq, sink_std, sink_fill)
    return kv


def make_mixed(seed: int, q_lens, kv_lens, hq: int, hkv: int, d: int, page_size: int = 16,
               sink_std: float = 1.0, sink_fill: float | None = None, permute: bool = True):
    """Mixed batch over a paged KV cache: q [sum q_len, Hq, D] with cu_seqlens_q."""
    kv = make_paged_kv(seed, kv_lens, hkv, d, page_size, permute)
    cu = cu_seqlens_from(q_lens)
    kv["q"] = normal_bf16(seed, STREAM_Q, (int(cu[-1]), hq, d))
    kv["cu_seqlens_q"] = cu
    kv["sinks"] = sinks_f32(seed, hq, sink_std, sink_fill)
    return kv


# --------------------------------------------------------------------------
# Inputs of the steps around attention (router, QKV projection output).
# --------------------------------------------------------------------------
def make_router_logits(seed: int, num_tokens: int, num_experts: int, std: float = 1.0,
                       levels: int | None = None) -> np.ndarray:
    """bf16 router logits [T, E].  With ``levels`` the values are integers drawn
    uniformly from [-levels, levels] (many exact ties)."""
    if levels is not None:
        rng = np.random.default_rng([seed, STREAM_LOGITS])
        x = rng.integers(-levels, levels + 1, (num_tokens, num_experts)).astype(np.float32)
        return _round_to_bf16_bits(x.ravel()).reshape(num_tokens, num_experts)
    return normal_bf16(seed, STREAM_LOGITS, (num_tokens, num_experts), std)


def make_qkv(seed: int, num_tokens: int, hq: int, hkv: int, d: int = 64, std: float = 1.0,
             bias_std: float = 0.5) -> dict:
    """QKV projection output without bias, bf16 [T, (Hq + 2 Hkv) * d] (q heads, then
    k heads, then v heads), and its bias, bf16 [(Hq + 2 Hkv) * d]."""
    width = (hq + 2 * hkv) * d
    return {"qkv": normal_bf16(seed, STREAM_QKV, (num_tokens, width), std),
            "bias": normal_bf16(seed, STREAM_BIAS, (width,), bias_std)}


def make_linear(seed: int, m: int, n: int, k: int, std: float = 1.0, w_std: float | None = None,
                bias_std: float = 1.0) -> dict:
    """x bf16 [M, K], W bf16 [N, K] (one row per output feature), bias bf16 [N]."""
    w_std = 1.0 / math.sqrt(k) if w_std is None else w_std
    return {"x": normal_bf16(seed, STREAM_X, (m, k), std),
            "w": normal_bf16(seed, STREAM_W, (n, k), w_std),
            "bias": normal_bf16(seed, STREAM_BIAS, (n,), bias_std)}
