"""libpa loads, exports every symbol include/pa.h declares, and rejects bad
arguments with status codes (host-side checks only: no kernel runs here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_blocks_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n


def test_version(L):
    assert b"sm_103a" in L.pa_version()


def _decode_args(**kw):
    from paged_kv_cache_blocks_gb300 import binding as b
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, nb=100, tab=1 << 20, mb=8, lens=1 << 20, B=4,
             msl=0, hq=8, hkv=2, d=128, scale=0.1, dtype=b.PA_BF16, out=1 << 20, ws=1 << 20,
             wsb=1 << 30, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return (P(a["q"]), P(a["k"]), P(a["v"]), a["nb"], P(a["tab"]), a["mb"], P(a["lens"]), a["B"],
            a["msl"], a["hq"], a["hkv"], a["d"], a["scale"], a["dtype"], P(a["out"]), P(a["ws"]),
            a["wsb"], a["stream"])


@pytest.mark.parametrize("bad,code", [
    (dict(d=96), 3), (dict(dtype=7), 3), (dict(hq=6, hkv=4), 1), (dict(hq=32, hkv=2), 3),
    (dict(nb=0), 1), (dict(mb=0), 1), (dict(msl=8 * 16 + 1), 1), (dict(scale=float("inf")), 1),
    (dict(q=0), 1), (dict(ws=1 << 20 | 8), 1), (dict(k=(1 << 20) + 2), 1), (dict(wsb=16), 1),
    (dict(B=-1), 1), (dict(nb=1 << 27, hkv=2, hq=2), 3),
])
def test_decode_rejects_bad_arguments(L, bad, code):
    rc = L.pa_decode(*_decode_args(**bad))
    assert rc == code, L.pa_last_error_string()
    assert L.pa_last_error_string()


def test_decode_zero_sequences_is_a_noop(L):
    assert L.pa_decode(*_decode_args(B=0)) == 0


def test_cache_write_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    p = P(1 << 20)
    assert L.pa_cache_write(p, p, p, -1, 8, 128, p, p, 10, 1, None) == 1
    assert L.pa_cache_write(p, p, p, 4, 8, 80, p, p, 10, 1, None) == 3
    assert L.pa_cache_write(p, p, p, 4, 8, 128, p, p, 10, 5, None) == 3
    assert L.pa_cache_write(p, p, P(0), 4, 8, 128, p, p, 10, 1, None) == 1
    assert L.pa_cache_write(P((1 << 20) + 8), p, p, 4, 8, 128, p, p, 10, 1, None) == 1
    assert L.pa_cache_write(p, p, p, 0, 8, 128, p, p, 10, 1, None) == 0   # nothing to do


def test_workspace_size_grows_with_partitions(L):
    a = L.pa_decode_workspace_bytes(8, 32, 128, 512)
    b = L.pa_decode_workspace_bytes(8, 32, 128, 513)
    assert b > a > 0
    # partial results: (max, sum) + head_dim floats per (partition, query head)
    assert b - a >= 8 * 32 * (128 + 2) * 4
    assert L.pa_decode_workspace_bytes(-1, 32, 128, 512) == 0


def _prefill_args(**kw):
    from paged_kv_cache_blocks_gb300 import binding as b
    a = dict(q=1 << 20, k=1 << 20, v=1 << 20, nb=100, tab=1 << 20, mb=8, lens=1 << 20,
             qoff=1 << 20, B=4, Tq=40, msl=0, hq=8, hkv=2, d=128, scale=0.1, dtype=b.PA_BF16,
             out=1 << 20, ws=1 << 20, wsb=1 << 30, stream=None, opts=None)
    a.update(kw)
    P = ctypes.c_void_p
    return (P(a["q"]), P(a["k"]), P(a["v"]), a["nb"], P(a["tab"]), a["mb"], P(a["lens"]),
            P(a["qoff"]), a["B"], a["Tq"], a["msl"], a["hq"], a["hkv"], a["d"], a["scale"],
            a["dtype"], P(a["out"]), P(a["ws"]), a["wsb"], a["stream"], a["opts"])


@pytest.mark.parametrize("bad,code", [
    (dict(d=96), 3), (dict(dtype=7), 3), (dict(hq=6, hkv=4), 1), (dict(hq=32, hkv=2), 3),
    (dict(nb=0), 1), (dict(mb=0), 1), (dict(msl=8 * 16 + 1), 1), (dict(scale=float("nan")), 1),
    (dict(qoff=0), 1), (dict(ws=1 << 20 | 8), 1), (dict(out=(1 << 20) + 2), 1), (dict(wsb=16), 1),
    (dict(B=-1), 1), (dict(Tq=-1), 1), (dict(nb=1 << 27, hkv=2, hq=2), 3),
])
def test_prefill_rejects_bad_arguments(L, bad, code):
    rc = L.pa_prefill(*_prefill_args(**bad))
    assert rc == code, L.pa_last_error_string()
    assert L.pa_last_error_string()


def test_prefill_empty_is_a_noop_and_workspace_sizes(L):
    assert L.pa_prefill(*_prefill_args(B=0)) == 0
    assert L.pa_prefill(*_prefill_args(Tq=0)) == 0
    # one (sequence, tile) record of 16 bytes per 128 query rows, plus one per sequence
    a = L.pa_prefill_workspace_bytes(4, 1000, 64, 8)
    b = L.pa_prefill_workspace_bytes(4, 100000, 64, 8)
    assert b > a > 0
    assert b - a >= (100000 - 1000) // 16 * 16 - 256
    assert L.pa_prefill_workspace_bytes(4, 100, 6, 4) == 0


def test_decode_rejects_unknown_flags(L):
    from paged_kv_cache_blocks_gb300 import binding as b
    o = b.PaDecodeOpts()
    o.flags = 2
    assert L.pa_decode_ex(*_decode_args(), ctypes.byref(o)) == 1
    assert b"flags" in L.pa_last_error_string()
    o.flags = 1
    assert L.pa_prefill(*_prefill_args(opts=ctypes.byref(o))) == 1


def test_decode_partition_tokens_checked(L):
    from paged_kv_cache_blocks_gb300 import binding as b
    o = b.PaDecodeOpts()
    for bad in (256, 513, 4096, -512):
        o.partition_tokens = bad
        assert L.pa_decode_ex(*_decode_args(), ctypes.byref(o)) == b.PA_ERR_INVALID
        assert b"partition_tokens" in L.pa_last_error_string()
    o.partition_tokens = 512
    assert L.pa_prefill(*_prefill_args(opts=ctypes.byref(o))) == b.PA_ERR_INVALID
    assert ctypes.sizeof(b.PaDecodeOpts) == 56     # the size the struct had before the field


def test_selftest_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    assert L.pa_selftest_bounded_wait(0, P(1 << 20), None) == 1
    assert L.pa_selftest_bounded_wait(2_000_000_000, P(1 << 20), None) == 1
    assert L.pa_selftest_bounded_wait(1000, P(0), None) == 1


def test_reuse_plan_needs_a_planned_workspace(L):
    """PA_DECODE_REUSE_PLAN on a workspace no decode call planned (or planned
    for other shapes) is refused on the host, before anything is launched."""
    from paged_kv_cache_blocks_gb300 import binding as b
    o = b.PaDecodeOpts()
    o.flags = b.PA_DECODE_REUSE_PLAN
    for ws in (1 << 24, (1 << 24) + 256 * 7):
        rc = L.pa_decode_ex(*_decode_args(ws=ws), ctypes.byref(o))
        assert rc == b.PA_ERR_INVALID
        assert b"PA_DECODE_REUSE_PLAN" in L.pa_last_error_string()
    P = ctypes.c_void_p
    a = _decode_args(ws=1 << 24)
    p = P(1 << 20)
    rc = L.pa_decode_fp8(a[0], a[1], a[2], p, p, *a[3:], ctypes.byref(o))
    assert rc == b.PA_ERR_INVALID and b"PA_DECODE_REUSE_PLAN" in L.pa_last_error_string()
    rc = L.pa_decode_grouped(*a[:14], p, p, 2, *a[14:], ctypes.byref(o))
    assert rc == b.PA_ERR_INVALID and b"PA_DECODE_REUSE_PLAN" in L.pa_last_error_string()


def test_reuse_plan_without_workspace_raises_before_any_call(monkeypatch):
    """The binding refuses reuse_plan without the planning call's workspace
    before it allocates or calls into the library (all three decode calls)."""
    import torch
    from paged_kv_cache_blocks_gb300 import binding as b

    def no_call():
        raise AssertionError("the library must not be reached")
    monkeypatch.setattr(b, "lib", no_call)
    t = torch.zeros(1)
    with pytest.raises(ValueError, match="reuse_plan"):
        b.pa_decode(t, t, t, t, t, 0.1, reuse_plan=True)
    with pytest.raises(ValueError, match="reuse_plan"):
        b.pa_decode_fp8(t, t, t, t, t, t, t, 0.1, reuse_plan=True)
    with pytest.raises(ValueError, match="reuse_plan"):
        b.pa_decode_grouped(t, t, t, t, t, 0.1, t, t, reuse_plan=True)


def test_noalloc_binding_checks_index_types(monkeypatch):
    """int64 block tables or lengths are refused (they would be read as pairs
    of int32 words) before the library is called."""
    import torch
    from paged_kv_cache_blocks_gb300 import binding as b

    def no_call():
        raise AssertionError("the library must not be reached")
    monkeypatch.setattr(b, "lib", no_call)
    monkeypatch.setattr(b, "_need_cuda", lambda *ts: None)
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    for tab, lens in ((torch.zeros(2, 3, dtype=torch.int64), torch.ones(2, dtype=torch.int32)),
                      (torch.zeros(2, 3, dtype=torch.int32), torch.ones(2, dtype=torch.int64))):
        with pytest.raises(TypeError, match="int32"):
            b.pa_decode_noalloc(q, kc, kc, tab, lens, 0.1, out=q)
        with pytest.raises(TypeError, match="int32"):
            b.pa_decode_fp8(q, kc, kc, torch.ones(2), torch.ones(2), tab, lens, 0.1, out=q,
                            workspace=torch.zeros(256, dtype=torch.uint8))


def test_binding_short_names_are_the_c_calls():
    from paged_kv_cache_blocks_gb300 import binding
    assert binding.cache_write is binding.pa_cache_write
    assert binding.decode is binding.pa_decode
