"""GQA attention with per-head softmax sinks on GB300 (sm_103a).

Thin ctypes binding of ``libsinkattn.so`` (C ABI in ``include/sink_attn.h``).
Every function below only marshals arguments: it reads shapes off the torch
tensors, allocates outputs when none are given, passes raw device pointers
and the current CUDA stream, and turns a non-zero status into an exception.
All arithmetic runs in the library's CUDA kernels; there is no fallback.

The operation (page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink
Attention"): ``attn = softmax(q k^T * sm_scale + sink) V`` where each query
head's sink is one extra softmax logit that carries no value row.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SinkAttnError", "library_path", "load_library", "sink_attn_prefill", "sink_attn_prefill_paged",
    "sink_attn_decode", "sink_attn_merge", "sink_attn_decode_splits", "sink_attn_device_status",
    "sink_attn_set_wait_timeout_ns", "sink_attn_status_string", "sink_attn_abi_version",
    "sink_attn_selftest_wait_timeout", "sink_attn_decode_noalloc", "moe_router_topk_softmax",
    "qkv_bias_rope", "qkv_bias_rope_append_paged", "linear_bias", "moe_router", "GPT_OSS_YARN",
    "EXPORTED_SYMBOLS", "qkv_bias_rope_kv", "qkv_bias_rope_append_paged_kv", "sink_attn_prefill_qkv",
    "sink_attn_prefill_paged_qkv", "sink_attn_decode_qkv",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsinkattn.so")
_lib = None

EXPORTED_SYMBOLS = (
    "sink_attn_prefill", "sink_attn_prefill_paged", "sink_attn_decode", "sink_attn_merge",
    "sink_attn_decode_splits", "sink_attn_device_status", "sink_attn_set_wait_timeout_ns",
    "sink_attn_status_string", "sink_attn_abi_version", "sink_attn_selftest_wait_timeout",
    "sink_attn_decode_noalloc", "moe_router_topk_softmax", "qkv_bias_rope",
    "qkv_bias_rope_append_paged", "linear_bias", "moe_router", "qkv_bias_rope_kv",
    "qkv_bias_rope_append_paged_kv", "sink_attn_prefill_qkv", "sink_attn_prefill_paged_qkv",
    "sink_attn_decode_qkv",
)

_p, _i, _f, _d, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_longlong
_SIGNATURES = {
    "sink_attn_prefill": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p, _p]),
    "sink_attn_prefill_paged": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                     _f, _i, _p, _p, _p]),
    "sink_attn_decode": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p, _p]),
    "sink_attn_merge": (_i, [_p, _p, _i, _i, _i, _i, _p, _p, _p]),
    "sink_attn_decode_splits": (_i, [_i, _i, _i, _i, _i]),
    "sink_attn_device_status": (_i, [_i]),
    "sink_attn_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "sink_attn_status_string": (ctypes.c_char_p, [_i]),
    "sink_attn_abi_version": (_i, []),
    "sink_attn_selftest_wait_timeout": (_i, [ctypes.c_ulonglong, _p]),
    "sink_attn_decode_noalloc": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p,
                                      _p]),
    "moe_router_topk_softmax": (_i, [_p, _ll, _i, _i, _p, _p, _p, _p]),
    "linear_bias": (_i, [_p, _p, _p, _i, _i, _i, _p, _p]),
    "moe_router": (_i, [_p, _p, _p, _i, _i, _i, _i, _p, _p, _p, _p]),
    "qkv_bias_rope": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _d, _i, _d, _d, _p, _p, _p, _p]),
    "qkv_bias_rope_append_paged": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _d, _i, _d, _d, _p, _p,
                                        _p, _p, _i, _i, _i, _p]),
    "qkv_bias_rope_kv": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _d, _i, _d, _d, _p, _p, _p, _p]),
    "qkv_bias_rope_append_paged_kv": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _d, _i, _d, _d, _p, _p,
                                           _p, _i, _i, _i, _p, _p]),
    "sink_attn_prefill_qkv": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p, _p]),
    "sink_attn_prefill_paged_qkv": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i,
                                         _i, _f, _i, _p, _p, _p]),
    "sink_attn_decode_qkv": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _p,
                                  _p]),
}

# YaRN constants of the public GPT-OSS model configuration (the pages name YaRN
# but give no constants): rotary base, scale factor, original context length,
# beta_fast, beta_slow.
GPT_OSS_YARN = dict(rope_base=150000.0, factor=32.0, orig_len=4096, beta_fast=32.0, beta_slow=1.0)


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({_status_text(status)})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libsinkattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m attention_softmax_sinks_gb300._build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _status_text(status: int) -> str:
    try:
        return load_library().sink_attn_status_string(status).decode()
    except Exception:  # library missing: still produce a message
        return "unknown"


def _check(status: int, where: str):
    if status != 0:
        raise SinkAttnError(status, where)


def _ptr(t):
    """Raw device address (ctypes passes Python ints as void*), or None."""
    return None if t is None else t.data_ptr()


def _dev(t, name, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _out(t, name, dtype, shape, dev):
    """A caller-supplied output: on device index ``dev``, of ``dtype``, contiguous and ``shape``."""
    _dev(t, name, dtype)
    if t.get_device() != dev:
        raise ValueError(f"{name} is on cuda:{t.get_device()}, the inputs on cuda:{dev}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _same_device(dev, *named):
    """Every (name, tensor) pair with a tensor lies on device index ``dev``."""
    for name, t in named:
        if t is not None and t.get_device() != dev:
            raise ValueError(f"{name} is on cuda:{t.get_device()}, expected cuda:{dev} "
                             "(the device of the first input)")


def _call(fn, dev, stream, *args):
    """fn(*args, stream) with device ``dev`` current for the call and ``stream`` (default: that
    device's current stream) as the last argument; the previous current device is restored."""
    if stream is not None and stream.device_index != dev:
        raise ValueError(f"stream is on cuda:{stream.device_index}, the tensors on cuda:{dev}")
    if torch.cuda.current_device() == dev:
        s = torch.cuda.current_stream() if stream is None else stream
        return fn(*args, s.cuda_stream)
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream() if stream is None else stream
        return fn(*args, s.cuda_stream)


# ----------------------------------------------------------------------------- entry points
def _checked(named):
    """Validate (name, tensor, dtype) triples: CUDA, dtype, contiguous.  Returns the first
    tensor's device and device index."""
    for name, t, dt in named:
        _dev(t, name, dt)
    first = named[0][1]
    return first.device, first.get_device()


def sink_attn_prefill(q, k, v, sinks, cu_seqlens, max_seqlen: int, sm_scale: float,
                      causal: bool = True, out=None, lse=None, return_lse: bool = True,
                      stream=None):
    """Prefill over contiguous ragged sequences (q_len == kv_len).

    q [T, Hq, 64] bf16, k/v [T, Hkv, 64] bf16, sinks [Hq] fp32, cu_seqlens [B+1] int32.
    Returns (out [T, Hq, 64] bf16, lse [T, Hq] fp32 or None).
    """
    dev, di = _checked((("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("sinks", sinks, torch.float32), ("cu_seqlens", cu_seqlens, torch.int32)))
    t, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != (t, hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, D] with q's T and D")
    _same_device(di, ("k", k), ("v", v), ("sinks", sinks), ("cu_seqlens", cu_seqlens))
    out = torch.empty_like(q) if out is None else _out(out, "out", torch.bfloat16, q.shape, di)
    if lse is None and return_lse:
        lse = torch.empty((t, hq), dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, (t, hq), di)
    st = _call(load_library().sink_attn_prefill, di, stream,
               _ptr(q), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens), cu_seqlens.numel() - 1, t,
               int(max_seqlen), hq, hkv, d, float(sm_scale), int(bool(causal)), _ptr(out), _ptr(lse))
    _check(st, "sink_attn_prefill")
    return out, lse


def sink_attn_prefill_paged(q, paged_k, paged_v, page_table, cu_seqlens_q, kv_lens, sinks,
                            max_q_len: int, sm_scale: float, causal: bool = True, out=None,
                            lse=None, return_lse: bool = True, stream=None):
    """New tokens of a mixed batch against a paged cache (bottom-right causal).

    q [Tq, Hq, 64] bf16, paged_k/v [P, Hkv, 16, 64] bf16, page_table [B, max_pages] int32,
    cu_seqlens_q [B+1] int32, kv_lens [B] int32, sinks [Hq] fp32.
    """
    dev, di = _checked((("q", q, torch.bfloat16), ("paged_k", paged_k, torch.bfloat16),
                        ("paged_v", paged_v, torch.bfloat16), ("page_table", page_table, torch.int32),
                        ("cu_seqlens_q", cu_seqlens_q, torch.int32), ("kv_lens", kv_lens, torch.int32),
                        ("sinks", sinks, torch.float32)))
    t, hq, d = q.shape
    num_pages, hkv, page_size, _ = paged_k.shape
    _same_device(di, ("paged_k", paged_k), ("paged_v", paged_v), ("page_table", page_table),
                 ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens), ("sinks", sinks))
    out = torch.empty_like(q) if out is None else _out(out, "out", torch.bfloat16, q.shape, di)
    if lse is None and return_lse:
        lse = torch.empty((t, hq), dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, (t, hq), di)
    st = _call(load_library().sink_attn_prefill_paged, di, stream,
               _ptr(q), _ptr(paged_k), _ptr(paged_v), _ptr(page_table), _ptr(cu_seqlens_q), _ptr(kv_lens),
               _ptr(sinks), cu_seqlens_q.numel() - 1, t, int(max_q_len), hq, hkv, d, page_size,
               page_table.shape[1], num_pages, float(sm_scale), int(bool(causal)), _ptr(out), _ptr(lse))
    _check(st, "sink_attn_prefill_paged")
    return out, lse


def _decode_outputs(out, lse, return_lse, b, s, hq, d, dev, di):
    out_shape, out_dtype = ((b, hq, d), torch.bfloat16) if s == 1 else ((b, s, hq, d), torch.float32)
    lse_shape = (b, hq) if s == 1 else (b, s, hq)
    if out is None:
        out = torch.empty(out_shape, dtype=out_dtype, device=dev)
    else:
        _out(out, "out", out_dtype, out_shape, di)
    if lse is None and (return_lse or s > 1):
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, lse_shape, di)
    return out, lse


def sink_attn_decode(q, paged_k, paged_v, page_table, kv_lens, sinks, sm_scale: float,
                     num_splits: int = 1, out=None, lse=None, return_lse: bool = True, stream=None):
    """One new token per sequence against a paged cache.

    num_splits == 1: returns (out [B, Hq, 64] bf16, lse [B, Hq] fp32).
    num_splits > 1: returns the partials (o [B, S, Hq, 64] fp32, lse [B, S, Hq] fp32)
    for sink_attn_merge.
    """
    dev, di = _checked((("q", q, torch.bfloat16), ("paged_k", paged_k, torch.bfloat16),
                        ("paged_v", paged_v, torch.bfloat16), ("page_table", page_table, torch.int32),
                        ("kv_lens", kv_lens, torch.int32), ("sinks", sinks, torch.float32)))
    b, hq, d = q.shape
    num_pages, hkv, page_size, _ = paged_k.shape
    _same_device(di, ("paged_k", paged_k), ("paged_v", paged_v), ("page_table", page_table),
                 ("kv_lens", kv_lens), ("sinks", sinks))
    s = int(num_splits)
    out, lse = _decode_outputs(out, lse, return_lse, b, s, hq, d, dev, di)
    st = _call(load_library().sink_attn_decode, di, stream,
               _ptr(q), _ptr(paged_k), _ptr(paged_v), _ptr(page_table), _ptr(kv_lens), _ptr(sinks), b, hq,
               hkv, d, page_size, page_table.shape[1], num_pages, float(sm_scale), s, _ptr(out), _ptr(lse))
    _check(st, "sink_attn_decode")
    return out, lse


def sink_attn_decode_noalloc(q, paged_k, paged_v, page_table, kv_lens, sinks, sm_scale: float,
                             num_splits: int, out=None, lse=None, return_lse: bool = True,
                             stream=None):
    """Split decode + merge in one library call that allocates no device memory.

    For callers that cannot allocate when they enqueue work: the split partials
    live in the library's fixed 8 MiB device array (batch * num_splits * Hq * 65
    floats at most).  Pass preallocated ``out`` [B, Hq, 64] bf16 and ``lse``
    [B, Hq] fp32 to keep this wrapper allocation-free as well.  Calls that
    overlap on the GPU race on the shared array.
    """
    dev, di = _checked((("q", q, torch.bfloat16), ("paged_k", paged_k, torch.bfloat16),
                        ("paged_v", paged_v, torch.bfloat16), ("page_table", page_table, torch.int32),
                        ("kv_lens", kv_lens, torch.int32), ("sinks", sinks, torch.float32)))
    b, hq, d = q.shape
    num_pages, hkv, page_size, _ = paged_k.shape
    _same_device(di, ("paged_k", paged_k), ("paged_v", paged_v), ("page_table", page_table),
                 ("kv_lens", kv_lens), ("sinks", sinks))
    out, lse = _decode_outputs(out, lse, return_lse, b, 1, hq, d, dev, di)
    st = _call(load_library().sink_attn_decode_noalloc, di, stream,
               _ptr(q), _ptr(paged_k), _ptr(paged_v), _ptr(page_table), _ptr(kv_lens), _ptr(sinks), b, hq,
               hkv, d, page_size, page_table.shape[1], num_pages, float(sm_scale), int(num_splits),
               _ptr(out), _ptr(lse))
    _check(st, "sink_attn_decode_noalloc")
    return out, lse


def sink_attn_merge(partial_o, partial_lse, out=None, lse=None, return_lse: bool = True,
                    stream=None):
    """Merge split partials o [B, S, H, 64] fp32 / lse [B, S, H] fp32 -> (out bf16, lse fp32)."""
    dev, di = _checked((("partial_o", partial_o, torch.float32), ("partial_lse", partial_lse, torch.float32)))
    b, s, h, d = partial_o.shape
    if tuple(partial_lse.shape) != (b, s, h):
        raise ValueError(f"partial_lse must be {(b, s, h)}, got {tuple(partial_lse.shape)}")
    _same_device(di, ("partial_lse", partial_lse))
    out = (torch.empty((b, h, d), dtype=torch.bfloat16, device=dev) if out is None
           else _out(out, "out", torch.bfloat16, (b, h, d), di))
    if lse is None and return_lse:
        lse = torch.empty((b, h), dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, (b, h), di)
    st = _call(load_library().sink_attn_merge, di, stream,
               _ptr(partial_o), _ptr(partial_lse), b, s, h, d, _ptr(out), _ptr(lse))
    _check(st, "sink_attn_merge")
    return out, lse


def sink_attn_decode_splits(batch: int, num_kv_heads: int, max_kv_len: int, page_size: int = 16,
                            num_sms: int = 0) -> int:
    if num_sms <= 0 and torch.cuda.is_available():
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return load_library().sink_attn_decode_splits(batch, num_kv_heads, max_kv_len, page_size, num_sms)


def sink_attn_device_status(clear: bool = True) -> int:
    """Status word of the current device (synchronises); 0 when clean."""
    return load_library().sink_attn_device_status(int(bool(clear)))


def sink_attn_set_wait_timeout_ns(ns: int) -> None:
    load_library().sink_attn_set_wait_timeout_ns(int(ns))


def sink_attn_status_string(status: int) -> str:
    return load_library().sink_attn_status_string(int(status)).decode()


def sink_attn_abi_version() -> int:
    return load_library().sink_attn_abi_version()


def sink_attn_selftest_wait_timeout(timeout_ns: int = 1_000_000, stream=None) -> None:
    """Launch the bounded-wait diagnostic (records SA_ERR_TIMEOUT in the status word)."""
    di = torch.cuda.current_device() if stream is None else stream.device_index
    _check(_call(load_library().sink_attn_selftest_wait_timeout, di, stream, int(timeout_ns)),
           "sink_attn_selftest_wait_timeout")


# ----------------------------------------------------------------------------- around attention
def moe_router_topk_softmax(logits, top_k: int, topk_idx=None, topk_weight=None,
                            expert_counts=None, return_counts: bool = False, stream=None):
    """Top-K-then-softmax router over bf16 logits [T, E] (page "GPT-OSS on day 0",
    section "Kernels for GPT-OSS / MoE").  Returns (idx int32 [T, k], weight bf16
    [T, k]) and, with return_counts or a given expert_counts, the int32 [E] counts."""
    dev, di = _checked((("logits", logits, torch.bfloat16),))
    t, e = logits.shape
    k = int(top_k)
    topk_idx = (torch.empty((t, k), dtype=torch.int32, device=dev) if topk_idx is None
                else _out(topk_idx, "topk_idx", torch.int32, (t, k), di))
    topk_weight = (torch.empty((t, k), dtype=torch.bfloat16, device=dev) if topk_weight is None
                   else _out(topk_weight, "topk_weight", torch.bfloat16, (t, k), di))
    if expert_counts is None and return_counts:
        expert_counts = torch.empty((e,), dtype=torch.int32, device=dev)
    elif expert_counts is not None:
        _out(expert_counts, "expert_counts", torch.int32, (e,), di)
    st = _call(load_library().moe_router_topk_softmax, di, stream,
               _ptr(logits), t, e, k, _ptr(topk_idx), _ptr(topk_weight), _ptr(expert_counts))
    _check(st, "moe_router_topk_softmax")
    if expert_counts is not None:
        return topk_idx, topk_weight, expert_counts
    return topk_idx, topk_weight


def _rope_params(rope):
    r = dict(GPT_OSS_YARN if rope is None else rope)
    return (float(r["rope_base"]), float(r["factor"]), int(r["orig_len"]), float(r["beta_fast"]),
            float(r["beta_slow"]))


def _opt(named):
    """Validate the optional (name, tensor, dtype) triples that are not None."""
    for name, t, dt in named:
        if t is not None:
            _dev(t, name, dt)


def qkv_bias_rope(qkv, bias, cu_seqlens_q, num_qo_heads: int, num_kv_heads: int, kv_lens=None,
                  rope=None, q_out=None, k_out=None, v_out=None, stream=None):
    """QKV bias + YaRN rotation of q and k.  qkv bf16 [T, (Hq + 2 Hkv) * 64] -> (q [T, Hq, 64],
    k [T, Hkv, 64], v [T, Hkv, 64]) bf16.  rope: dict like GPT_OSS_YARN (default)."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32)))
    _opt((("bias", bias, torch.bfloat16), ("kv_lens", kv_lens, torch.int32)))
    t = qkv.shape[0]
    hq, hkv, d = int(num_qo_heads), int(num_kv_heads), 64
    _same_device(di, ("bias", bias), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens))
    q_out = torch.empty((t, hq, d), dtype=torch.bfloat16, device=dev) if q_out is None else q_out
    k_out = torch.empty((t, hkv, d), dtype=torch.bfloat16, device=dev) if k_out is None else k_out
    v_out = torch.empty((t, hkv, d), dtype=torch.bfloat16, device=dev) if v_out is None else v_out
    for name, x, h in (("q_out", q_out, hq), ("k_out", k_out, hkv), ("v_out", v_out, hkv)):
        _out(x, name, torch.bfloat16, (t, h, d), di)
    st = _call(load_library().qkv_bias_rope, di, stream,
               _ptr(qkv), _ptr(bias), _ptr(cu_seqlens_q), _ptr(kv_lens), cu_seqlens_q.numel() - 1, t, hq, hkv,
               qkv.shape[1] // (hq + 2 * hkv), *_rope_params(rope), _ptr(q_out), _ptr(k_out), _ptr(v_out))
    _check(st, "qkv_bias_rope")
    return q_out, k_out, v_out


def qkv_bias_rope_append_paged(qkv, bias, cu_seqlens_q, kv_lens, paged_k, paged_v, page_table,
                               num_qo_heads: int, rope=None, q_out=None, stream=None):
    """QKV bias + YaRN rotation; q returned [T, Hq, 64], k and v written in place into the
    paged cache [num_pages, Hkv, 16, 64] at each new token's position."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("kv_lens", kv_lens, torch.int32), ("paged_k", paged_k, torch.bfloat16),
                        ("paged_v", paged_v, torch.bfloat16), ("page_table", page_table, torch.int32)))
    _opt((("bias", bias, torch.bfloat16),))
    t = qkv.shape[0]
    num_pages, hkv, page_size, d = paged_k.shape
    hq = int(num_qo_heads)
    _same_device(di, ("bias", bias), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens),
                 ("paged_k", paged_k), ("paged_v", paged_v), ("page_table", page_table))
    q_out = torch.empty((t, hq, d), dtype=torch.bfloat16, device=dev) if q_out is None else q_out
    _out(q_out, "q_out", torch.bfloat16, (t, hq, d), di)
    st = _call(load_library().qkv_bias_rope_append_paged, di, stream,
               _ptr(qkv), _ptr(bias), _ptr(cu_seqlens_q), _ptr(kv_lens), cu_seqlens_q.numel() - 1, t, hq, hkv,
               qkv.shape[1] // (hq + 2 * hkv), *_rope_params(rope), _ptr(q_out), _ptr(paged_k), _ptr(paged_v),
               _ptr(page_table), page_size, page_table.shape[1], num_pages)
    _check(st, "qkv_bias_rope_append_paged")
    return q_out


def linear_bias(x, w, bias=None, out=None, stream=None):
    """out [M, N] = x [M, K] @ w[N, K]^T + bias[N] on the tcgen05 tensor cores, bf16 in and out,
    the fp32 accumulator seeded with the bias (page "GPT-OSS on day 0", section "Kernels for
    GPT-OSS / MoE")."""
    dev, di = _checked((("x", x, torch.bfloat16), ("w", w, torch.bfloat16)))
    _opt((("bias", bias, torch.bfloat16),))
    m, k = x.shape
    n = w.shape[0]
    if w.shape[1] != k:
        raise ValueError(f"w is {tuple(w.shape)}, expected [N, {k}]")
    _same_device(di, ("w", w), ("bias", bias))
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev) if out is None else out
    _out(out, "out", torch.bfloat16, (m, n), di)
    st = _call(load_library().linear_bias, di, stream, _ptr(x), _ptr(w), _ptr(bias), m, n, k, _ptr(out))
    _check(st, "linear_bias")
    return out


def moe_router(x, w_router, bias, top_k: int, topk_idx=None, topk_weight=None, expert_counts=None,
               return_counts: bool = False, stream=None):
    """Router projection + bias + bf16 logits + Top-K softmax in one tcgen05 kernel:
    x [T, hidden] bf16, w_router [E, hidden] bf16, bias [E] bf16 or None.  Returns
    (idx int32 [T, k], weight bf16 [T, k]) and the int32 [E] counts when asked."""
    dev, di = _checked((("x", x, torch.bfloat16), ("w_router", w_router, torch.bfloat16)))
    _opt((("bias", bias, torch.bfloat16),))
    t, hidden = x.shape
    e = w_router.shape[0]
    if w_router.shape[1] != hidden:
        raise ValueError(f"w_router is {tuple(w_router.shape)}, expected [E, {hidden}]")
    k = int(top_k)
    _same_device(di, ("w_router", w_router), ("bias", bias))
    topk_idx = (torch.empty((t, k), dtype=torch.int32, device=dev) if topk_idx is None
                else _out(topk_idx, "topk_idx", torch.int32, (t, k), di))
    topk_weight = (torch.empty((t, k), dtype=torch.bfloat16, device=dev) if topk_weight is None
                   else _out(topk_weight, "topk_weight", torch.bfloat16, (t, k), di))
    if expert_counts is None and return_counts:
        expert_counts = torch.empty((e,), dtype=torch.int32, device=dev)
    elif expert_counts is not None:
        _out(expert_counts, "expert_counts", torch.int32, (e,), di)
    st = _call(load_library().moe_router, di, stream, _ptr(x), _ptr(w_router), _ptr(bias), t, hidden, e, k,
               _ptr(topk_idx), _ptr(topk_weight), _ptr(expert_counts))
    _check(st, "moe_router")
    if expert_counts is not None:
        return topk_idx, topk_weight, expert_counts
    return topk_idx, topk_weight


# ----------------------------------------------------------------------------- q rotated on chip
def qkv_bias_rope_kv(qkv, bias, cu_seqlens_q, num_qo_heads: int, num_kv_heads: int, kv_lens=None,
                     rope=None, k_out=None, v_out=None, rope_table=None, stream=None):
    """K/V half of qkv_bias_rope for the *_qkv attention calls: k (biased, rotated) and v
    (biased) written contiguous [T, Hkv, 64] bf16, plus the per-token (cos, sin) table
    [T, 32, 2] fp32 those calls apply to q.  Returns (k, v, rope_table)."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32)))
    _opt((("bias", bias, torch.bfloat16), ("kv_lens", kv_lens, torch.int32)))
    t = qkv.shape[0]
    hq, hkv, d = int(num_qo_heads), int(num_kv_heads), 64
    _same_device(di, ("bias", bias), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens))
    k_out = torch.empty((t, hkv, d), dtype=torch.bfloat16, device=dev) if k_out is None else k_out
    v_out = torch.empty((t, hkv, d), dtype=torch.bfloat16, device=dev) if v_out is None else v_out
    rope_table = (torch.empty((t, d // 2, 2), dtype=torch.float32, device=dev) if rope_table is None
                  else rope_table)
    _out(k_out, "k_out", torch.bfloat16, (t, hkv, d), di)
    _out(v_out, "v_out", torch.bfloat16, (t, hkv, d), di)
    _out(rope_table, "rope_table", torch.float32, (t, d // 2, 2), di)
    st = _call(load_library().qkv_bias_rope_kv, di, stream,
               _ptr(qkv), _ptr(bias), _ptr(cu_seqlens_q), _ptr(kv_lens), cu_seqlens_q.numel() - 1, t, hq, hkv,
               qkv.shape[1] // (hq + 2 * hkv), *_rope_params(rope), _ptr(k_out), _ptr(v_out), _ptr(rope_table))
    _check(st, "qkv_bias_rope_kv")
    return k_out, v_out, rope_table


def qkv_bias_rope_append_paged_kv(qkv, bias, cu_seqlens_q, kv_lens, paged_k, paged_v, page_table,
                                  num_qo_heads: int, rope=None, rope_table=None, stream=None):
    """K/V half of qkv_bias_rope_append_paged: k and v written in place into the paged
    cache at each new token's position, and the (cos, sin) table [T, 32, 2] fp32 of the
    new tokens returned for the *_qkv attention calls."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("kv_lens", kv_lens, torch.int32), ("paged_k", paged_k, torch.bfloat16),
                        ("paged_v", paged_v, torch.bfloat16), ("page_table", page_table, torch.int32)))
    _opt((("bias", bias, torch.bfloat16),))
    t = qkv.shape[0]
    num_pages, hkv, page_size, d = paged_k.shape
    hq = int(num_qo_heads)
    _same_device(di, ("bias", bias), ("cu_seqlens_q", cu_seqlens_q), ("kv_lens", kv_lens),
                 ("paged_k", paged_k), ("paged_v", paged_v), ("page_table", page_table))
    rope_table = (torch.empty((t, d // 2, 2), dtype=torch.float32, device=dev) if rope_table is None
                  else rope_table)
    _out(rope_table, "rope_table", torch.float32, (t, d // 2, 2), di)
    st = _call(load_library().qkv_bias_rope_append_paged_kv, di, stream,
               _ptr(qkv), _ptr(bias), _ptr(cu_seqlens_q), _ptr(kv_lens), cu_seqlens_q.numel() - 1, t, hq, hkv,
               qkv.shape[1] // (hq + 2 * hkv), *_rope_params(rope), _ptr(paged_k), _ptr(paged_v),
               _ptr(page_table), page_size, page_table.shape[1], num_pages, _ptr(rope_table))
    _check(st, "qkv_bias_rope_append_paged_kv")
    return rope_table


def sink_attn_prefill_qkv(qkv, qkv_bias, rope_table, k, v, sinks, cu_seqlens, max_seqlen: int,
                          sm_scale: float, num_qo_heads: int, causal: bool = True, out=None, lse=None,
                          return_lse: bool = True, stream=None):
    """sink_attn_prefill with q taken from the projection output qkv [T, (Hq + 2 Hkv) * 64]:
    the query bias and the rotation by rope_table (from qkv_bias_rope_kv) are applied on
    chip; k, v as written by qkv_bias_rope_kv."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("rope_table", rope_table, torch.float32),
                        ("k", k, torch.bfloat16), ("v", v, torch.bfloat16), ("sinks", sinks, torch.float32),
                        ("cu_seqlens", cu_seqlens, torch.int32)))
    _opt((("qkv_bias", qkv_bias, torch.bfloat16),))
    t = qkv.shape[0]
    hq = int(num_qo_heads)
    _, hkv, d = k.shape
    if k.shape != (t, hkv, d) or v.shape != k.shape or qkv.shape[1] != (hq + 2 * hkv) * d:
        raise ValueError("qkv must be [T, (Hq + 2 Hkv) * D] and k, v [T, Hkv, D]")
    if tuple(rope_table.shape) != (t, d // 2, 2):
        raise ValueError(f"rope_table must be {(t, d // 2, 2)}")
    _same_device(di, ("qkv_bias", qkv_bias), ("rope_table", rope_table), ("k", k), ("v", v), ("sinks", sinks),
                 ("cu_seqlens", cu_seqlens))
    out = (torch.empty((t, hq, d), dtype=torch.bfloat16, device=dev) if out is None
           else _out(out, "out", torch.bfloat16, (t, hq, d), di))
    if lse is None and return_lse:
        lse = torch.empty((t, hq), dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, (t, hq), di)
    st = _call(load_library().sink_attn_prefill_qkv, di, stream,
               _ptr(qkv), _ptr(qkv_bias), _ptr(rope_table), _ptr(k), _ptr(v), _ptr(sinks), _ptr(cu_seqlens),
               cu_seqlens.numel() - 1, t, int(max_seqlen), hq, hkv, d, float(sm_scale), int(bool(causal)),
               _ptr(out), _ptr(lse))
    _check(st, "sink_attn_prefill_qkv")
    return out, lse


def sink_attn_prefill_paged_qkv(qkv, qkv_bias, rope_table, paged_k, paged_v, page_table, cu_seqlens_q,
                                kv_lens, sinks, max_q_len: int, sm_scale: float, num_qo_heads: int,
                                causal: bool = True, out=None, lse=None, return_lse: bool = True,
                                stream=None):
    """sink_attn_prefill_paged with q taken from the projection output (see
    sink_attn_prefill_qkv); the paged cache and rope_table as written by
    qkv_bias_rope_append_paged_kv."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("rope_table", rope_table, torch.float32),
                        ("paged_k", paged_k, torch.bfloat16), ("paged_v", paged_v, torch.bfloat16),
                        ("page_table", page_table, torch.int32), ("cu_seqlens_q", cu_seqlens_q, torch.int32),
                        ("kv_lens", kv_lens, torch.int32), ("sinks", sinks, torch.float32)))
    _opt((("qkv_bias", qkv_bias, torch.bfloat16),))
    t = qkv.shape[0]
    hq = int(num_qo_heads)
    num_pages, hkv, page_size, d = paged_k.shape
    if qkv.shape[1] != (hq + 2 * hkv) * d or tuple(rope_table.shape) != (t, d // 2, 2):
        raise ValueError("qkv must be [T, (Hq + 2 Hkv) * D] and rope_table [T, D / 2, 2]")
    _same_device(di, ("qkv_bias", qkv_bias), ("rope_table", rope_table), ("paged_k", paged_k),
                 ("paged_v", paged_v), ("page_table", page_table), ("cu_seqlens_q", cu_seqlens_q),
                 ("kv_lens", kv_lens), ("sinks", sinks))
    out = (torch.empty((t, hq, d), dtype=torch.bfloat16, device=dev) if out is None
           else _out(out, "out", torch.bfloat16, (t, hq, d), di))
    if lse is None and return_lse:
        lse = torch.empty((t, hq), dtype=torch.float32, device=dev)
    elif lse is not None:
        _out(lse, "lse", torch.float32, (t, hq), di)
    st = _call(load_library().sink_attn_prefill_paged_qkv, di, stream,
               _ptr(qkv), _ptr(qkv_bias), _ptr(rope_table), _ptr(paged_k), _ptr(paged_v), _ptr(page_table),
               _ptr(cu_seqlens_q), _ptr(kv_lens), _ptr(sinks), cu_seqlens_q.numel() - 1, t, int(max_q_len), hq,
               hkv, d, page_size, page_table.shape[1], num_pages, float(sm_scale), int(bool(causal)), _ptr(out),
               _ptr(lse))
    _check(st, "sink_attn_prefill_paged_qkv")
    return out, lse


def sink_attn_decode_qkv(qkv, qkv_bias, rope_table, paged_k, paged_v, page_table, kv_lens, sinks,
                         sm_scale: float, num_qo_heads: int, num_splits: int = 1, out=None, lse=None,
                         return_lse: bool = True, stream=None):
    """sink_attn_decode with q taken from the projection output qkv [B, (Hq + 2 Hkv) * 64] (one
    new token per sequence): bias and rotation by row b of rope_table [B, 32, 2] applied in
    the kernel.  num_splits > 1 returns the fp32 partials, as sink_attn_decode does."""
    dev, di = _checked((("qkv", qkv, torch.bfloat16), ("rope_table", rope_table, torch.float32),
                        ("paged_k", paged_k, torch.bfloat16), ("paged_v", paged_v, torch.bfloat16),
                        ("page_table", page_table, torch.int32), ("kv_lens", kv_lens, torch.int32),
                        ("sinks", sinks, torch.float32)))
    _opt((("qkv_bias", qkv_bias, torch.bfloat16),))
    b = qkv.shape[0]
    hq = int(num_qo_heads)
    num_pages, hkv, page_size, d = paged_k.shape
    if qkv.shape[1] != (hq + 2 * hkv) * d or tuple(rope_table.shape) != (b, d // 2, 2):
        raise ValueError("qkv must be [B, (Hq + 2 Hkv) * D] and rope_table [B, D / 2, 2]")
    _same_device(di, ("qkv_bias", qkv_bias), ("rope_table", rope_table), ("paged_k", paged_k),
                 ("paged_v", paged_v), ("page_table", page_table), ("kv_lens", kv_lens), ("sinks", sinks))
    s = int(num_splits)
    out, lse = _decode_outputs(out, lse, return_lse, b, s, hq, d, dev, di)
    st = _call(load_library().sink_attn_decode_qkv, di, stream,
               _ptr(qkv), _ptr(qkv_bias), _ptr(rope_table), _ptr(paged_k), _ptr(paged_v), _ptr(page_table),
               _ptr(kv_lens), _ptr(sinks), b, hq, hkv, d, page_size, page_table.shape[1], num_pages,
               float(sm_scale), s, _ptr(out), _ptr(lse))
    _check(st, "sink_attn_decode_qkv")
    return out, lse
