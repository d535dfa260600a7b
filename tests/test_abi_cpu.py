"""The C ABI on the CPU: the library builds and loads, exports every function
that include/sink_attn.h declares, and rejects bad arguments with a status
code before touching the GPU (no compute call is made here)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

SA_OK, SA_ERR_NULL, SA_ERR_SHAPE, SA_ERR_UNSUPPORTED = 0, 1, 2, 3
SA_ERR_ALIGNMENT = 7


@pytest.fixture(scope="module")
def lib():
    from attention_softmax_sinks_gb300 import _build
    import attention_softmax_sinks_gb300 as sa
    _build.build()
    return sa.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:sa_status|int|void|const char\*)\s+(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("sink_attn_prefill", "sink_attn_prefill_paged", "sink_attn_decode", "sink_attn_merge"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import attention_softmax_sinks_gb300 as sa
    names = declared_functions()
    assert set(names) == set(sa.EXPORTED_SYMBOLS)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    nm = subprocess.run(["nm", "-D", "--defined-only", sa.library_path()], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r"\sT\s(\w+)", nm.stdout))
        for n in names:
            assert n in exported, f"{n} missing from the dynamic symbol table"


def test_library_targets_sm103a_only():
    from attention_softmax_sinks_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings_and_version(lib):
    assert lib.sink_attn_abi_version() == 1
    for s in range(9):
        assert lib.sink_attn_status_string(s)
    assert lib.sink_attn_status_string(99) == b"unknown status"


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: rejected first
MISALIGNED = ctypes.c_void_p(0x10008)


def _decode(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pt=FAKE, kv=FAKE, sinks=FAKE, batch=2, hq=64, hkv=8, d=64,
             ps=16, max_pages=4, num_pages=8, scale=0.125, splits=1, out=FAKE, lse=FAKE)
    a.update(kw)
    return lib.sink_attn_decode(a["q"], a["k"], a["v"], a["pt"], a["kv"], a["sinks"], a["batch"],
                                a["hq"], a["hkv"], a["d"], a["ps"], a["max_pages"], a["num_pages"],
                                a["scale"], a["splits"], a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), SA_ERR_NULL), (dict(pt=None), SA_ERR_NULL), (dict(sinks=None), SA_ERR_NULL),
    (dict(splits=4, lse=None), SA_ERR_NULL),
    (dict(d=128), SA_ERR_UNSUPPORTED), (dict(ps=32), SA_ERR_UNSUPPORTED),
    (dict(hq=64, hkv=3), SA_ERR_SHAPE), (dict(hq=64, hkv=2), SA_ERR_UNSUPPORTED),
    (dict(scale=0.0), SA_ERR_SHAPE), (dict(scale=float("nan")), SA_ERR_SHAPE),
    (dict(scale=float("inf")), SA_ERR_SHAPE), (dict(splits=0), SA_ERR_SHAPE),
    (dict(splits=257), SA_ERR_SHAPE), (dict(batch=-1), SA_ERR_SHAPE),
    (dict(num_pages=0), SA_ERR_SHAPE), (dict(q=MISALIGNED), SA_ERR_ALIGNMENT),
    (dict(k=MISALIGNED), SA_ERR_ALIGNMENT), (dict(batch=0), SA_OK),
])
def test_decode_rejects_before_launch(lib, kw, status):
    assert _decode(lib, **kw) == status


def _prefill(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sinks=FAKE, cu=FAKE, batch=1, t=128, maxq=128, hq=4, hkv=1,
             d=64, scale=0.125, causal=1, out=FAKE, lse=None)
    a.update(kw)
    return lib.sink_attn_prefill(a["q"], a["k"], a["v"], a["sinks"], a["cu"], a["batch"], a["t"],
                                 a["maxq"], a["hq"], a["hkv"], a["d"], a["scale"], a["causal"],
                                 a["out"], a["lse"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), SA_ERR_NULL), (dict(cu=None), SA_ERR_NULL), (dict(out=None), SA_ERR_NULL),
    (dict(d=96), SA_ERR_UNSUPPORTED), (dict(hq=6, hkv=4), SA_ERR_SHAPE),
    (dict(scale=-1.0), SA_ERR_SHAPE), (dict(t=-5), SA_ERR_SHAPE),
    (dict(out=MISALIGNED), SA_ERR_ALIGNMENT), (dict(batch=0), SA_OK), (dict(t=0), SA_OK),
])
def test_prefill_rejects_before_launch(lib, kw, status):
    assert _prefill(lib, **kw) == status


def test_prefill_paged_rejects(lib):
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 10, 8, 64, 8, 64, 16, 4, 8, 0.125, 1, FAKE, None, None]
    ok = list(args)
    bad_page = list(args); bad_page[13] = 8
    null_pt = list(args); null_pt[3] = None
    no_pages = list(args); no_pages[15] = 0
    assert lib.sink_attn_prefill_paged(*bad_page) == SA_ERR_UNSUPPORTED
    assert lib.sink_attn_prefill_paged(*null_pt) == SA_ERR_NULL
    assert lib.sink_attn_prefill_paged(*no_pages) == SA_ERR_SHAPE
    zero = list(ok); zero[7] = 0
    assert lib.sink_attn_prefill_paged(*zero) == SA_OK


def test_merge_rejects(lib):
    assert lib.sink_attn_merge(None, FAKE, 2, 4, 64, 64, FAKE, None, None) == SA_ERR_NULL
    assert lib.sink_attn_merge(FAKE, FAKE, 2, 0, 64, 64, FAKE, None, None) == SA_ERR_SHAPE
    assert lib.sink_attn_merge(FAKE, FAKE, 2, 4, 64, 32, FAKE, None, None) == SA_ERR_UNSUPPORTED
    assert lib.sink_attn_merge(FAKE, FAKE, 0, 4, 64, 64, FAKE, None, None) == SA_OK


def test_decode_split_heuristic(lib):
    f = lib.sink_attn_decode_splits
    # every result is within [1, 256] and keeps >= 32 pages per split
    for b, hkv, kv in [(1, 8, 131072), (8, 8, 131072), (64, 8, 4096), (256, 8, 512), (1, 1, 1)]:
        s = f(b, hkv, kv, 16, 152)
        assert 1 <= s <= 256
        pages = (kv + 15) // 16
        assert s == 1 or pages // s >= 32
    assert f(1, 8, 16, 16, 152) == 1           # a single page cannot be split
    assert f(8, 8, 131072, 16, 152) >= 16      # long context spreads over the GPU
    assert f(0, 8, 4096, 16, 152) == 1
    assert f(64, 8, 4096, 16, 152) == 4        # 512 (sequence, KV head) units: four waves
    assert f(1, 8, 4096, 16, 152) == 1         # 16-CTA clusters fit one wave: on-chip merge
    assert f(1, 8, 4000, 16, 152) == 1         # 250 pages: clusters of 8, still one wave
    assert f(8, 8, 4096, 16, 152) == 1         # 64 units x clusters of 4 = 256 CTAs
    assert f(16, 8, 4096, 16, 152) == 8        # clusters would exceed one wave: 8 splits of 32 pages
    assert f(8, 8, 131072, 16, 152) >= 16      # long caches: more CTAs than one wave of clusters
    assert f(1, 8, 131072, 16, 152) > 1
    assert f(1, 8, 16384, 16, 152) == 1        # 64 pages per CTA of a 16-CTA cluster
    assert f(1, 8, 32768, 16, 152) == 32       # 128 pages per cluster CTA: ~5/3 CTAs per SM instead
    assert f(1, 8, 131072, 16, 152) == 32
    assert f(2, 8, 65536, 16, 152) == 16
    assert f(4, 8, 131072, 16, 152) == 8
    assert f(8, 8, 131072, 16, 152) == 29      # 64 units: about four waves


def test_router_rejects_before_launch(lib):
    f = lib.moe_router_topk_softmax
    assert f(None, 10, 32, 4, FAKE, FAKE, None, None) == SA_ERR_NULL
    assert f(FAKE, 10, 32, 4, None, FAKE, None, None) == SA_ERR_NULL
    assert f(FAKE, 10, 0, 1, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, 10, 257, 4, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, 10, 32, 0, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, 10, 32, 9, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, 10, 3, 4, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, -1, 32, 4, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, 0, 32, 4, FAKE, FAKE, None, None) == SA_OK


GPT_OSS = (150000.0, 32.0, 4096, 32.0, 1.0)


def _rope(lib, **kw):
    a = dict(qkv=FAKE, bias=None, cu=FAKE, kv=None, batch=2, t=10, hq=64, hkv=8, d=64, yarn=GPT_OSS,
             q=FAKE, k=FAKE, v=FAKE)
    a.update(kw)
    return lib.qkv_bias_rope(a["qkv"], a["bias"], a["cu"], a["kv"], a["batch"], a["t"], a["hq"], a["hkv"],
                             a["d"], *a["yarn"], a["q"], a["k"], a["v"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(qkv=None), SA_ERR_NULL), (dict(cu=None), SA_ERR_NULL), (dict(q=None), SA_ERR_NULL),
    (dict(d=128), SA_ERR_UNSUPPORTED), (dict(hq=6, hkv=4), SA_ERR_SHAPE), (dict(batch=-1), SA_ERR_SHAPE),
    (dict(hq=128, hkv=8), SA_ERR_UNSUPPORTED),
    (dict(yarn=(1.0, 32.0, 4096, 32.0, 1.0)), SA_ERR_SHAPE), (dict(yarn=(1e4, 0.5, 4096, 32.0, 1.0)), SA_ERR_SHAPE),
    (dict(yarn=(1e4, 32.0, 4096, 1.0, 32.0)), SA_ERR_SHAPE), (dict(yarn=(1e4, 32.0, 0, 32.0, 1.0)), SA_ERR_SHAPE),
    (dict(yarn=(1e4, 1.0, 0, 0.0, 0.0)), SA_OK),   # factor 1: plain rotary, YaRN constants unused
    (dict(bias=MISALIGNED), SA_ERR_ALIGNMENT), (dict(k=MISALIGNED), SA_ERR_ALIGNMENT),
    (dict(batch=0), SA_OK), (dict(t=0), SA_OK),
])
def test_rope_rejects_before_launch(lib, kw, status):
    if status == SA_OK and "yarn" in kw:
        kw = dict(kw, batch=0)       # valid arguments, no work: nothing is launched
    assert _rope(lib, **kw) == status


def test_rope_paged_rejects(lib):
    f = lib.qkv_bias_rope_append_paged
    args = [FAKE, None, FAKE, FAKE, 2, 10, 64, 8, 64, *GPT_OSS, FAKE, FAKE, FAKE, FAKE, 16, 8, 64, None]
    assert f(*args[:3], None, *args[4:]) == SA_ERR_NULL          # kv_lens required
    bad = list(args); bad[17] = None                           # page table
    assert f(*bad) == SA_ERR_NULL
    bad = list(args); bad[18] = 8                              # page size
    assert f(*bad) == SA_ERR_UNSUPPORTED
    bad = list(args); bad[20] = 0                              # num_pages
    assert f(*bad) == SA_ERR_SHAPE
    ok = list(args); ok[4] = 0
    assert f(*ok) == SA_OK


def test_linear_rejects_before_launch(lib):
    f = lib.linear_bias
    assert f(FAKE, FAKE, None, -1, 64, 64, FAKE, None) == SA_ERR_SHAPE
    assert f(FAKE, FAKE, None, 4, 0, 64, FAKE, None) == SA_ERR_SHAPE
    assert f(FAKE, FAKE, None, 4, 60, 64, FAKE, None) == SA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, None, 4, 64, 20, FAKE, None) == SA_ERR_UNSUPPORTED
    assert f(None, FAKE, None, 4, 64, 64, FAKE, None) == SA_ERR_NULL
    assert f(FAKE, FAKE, None, 4, 64, 64, None, None) == SA_ERR_NULL
    assert f(MISALIGNED, FAKE, None, 4, 64, 64, FAKE, None) == SA_ERR_ALIGNMENT
    assert f(FAKE, FAKE, ctypes.c_void_p(0x10001), 4, 64, 64, FAKE, None) == SA_ERR_ALIGNMENT
    assert f(None, None, None, 0, 64, 64, None, None) == SA_OK


def test_library_has_no_unresolved_internal_symbols(lib):
    """Every kernel launcher the C ABI calls is linked in (a missing definition
    would otherwise only show when the library is loaded on a machine with a GPU)."""
    import attention_softmax_sinks_gb300 as sa
    nm = subprocess.run(["nm", "-D", "--undefined-only", sa.library_path()], capture_output=True, text=True)
    if nm.returncode != 0:
        pytest.skip("nm unavailable")
    assert "_ZN2sa" not in nm.stdout


def test_linear_rejects_tile_count_overflow(lib):
    # 2^31 - 1 rows x 2^30 features: more output tiles than an int holds
    assert lib.linear_bias(FAKE, FAKE, None, 2**31 - 1, 2**30, 64, FAKE, None) == SA_ERR_SHAPE


def test_fused_router_rejects_before_launch(lib):
    f = lib.moe_router
    assert f(FAKE, FAKE, None, 10, 2880, 0, 1, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, FAKE, None, 10, 2880, 257, 4, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, FAKE, None, 10, 2880, 128, 9, FAKE, FAKE, None, None) == SA_ERR_SHAPE
    assert f(FAKE, FAKE, None, 10, 2884, 128, 4, FAKE, FAKE, None, None) == SA_ERR_UNSUPPORTED
    assert f(None, FAKE, None, 10, 2880, 128, 4, FAKE, FAKE, None, None) == SA_ERR_NULL
    assert f(MISALIGNED, FAKE, None, 10, 2880, 128, 4, FAKE, FAKE, None, None) == SA_ERR_ALIGNMENT
    assert f(None, None, None, 0, 2880, 128, 4, None, None, None, None) == SA_OK
