"""CPU oracle for paged KV-cache decode (fp64).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's ``smoke()`` check
and the bench's CPU-baseline leg may import this package.  The product path
(the CUDA library and its binding) never imports, links or runs it, and the
oracle imports nothing from the product.

Parts:

* ``pa_oracle.c`` -- cache write, copy-on-write block copy, block-table
  gather and textbook softmax attention in fp64 (built to ``liboracle.so``
  by :func:`build`).
* :mod:`oracle.allocator` -- the block allocator model (free queue, ref
  counts, copy-on-write).
* :func:`kv_bytes_per_token` -- the pages' KV size formula.

Every function cites the passage it follows in its own docstring or in the
header of ``pa_oracle.c``.
"""
import concurrent.futures
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

DTYPE_CODES = {"f16": 0, "bf16": 1}


def kv_bytes_per_token(num_layers, num_kv_heads, head_dim, bytes_per_elem):
    """KV bytes per token = 2 x layers x KV heads x head_dim x bytes/element.

    The leading 2 counts K and V.  Defined in "Yerel LLM sistemlerinde
    backpressure ve olcekleme", section "KV butcesi", and restated with a
    worked example in "vLLM Nedir? PagedAttention ile Production LLM
    Serving", section "Asil sisen sey agirlik degil, KV cache".  Both
    insist on the KV-head count (not the attention-head count); the other
    page's version with attention heads lost its formula in extraction.
    """
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


def build(force=False):
    """Compile pa_oracle.c with gcc (OpenMP, no FP contraction) if stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class OracleLib:
    """ctypes handle on one build of pa_oracle.c (the default one, or a
    variant a test compiled from a modified copy of the source)."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_bits_to_double.argtypes = [P, i64, ctypes.c_int, P]
        lib.oracle_bits_to_double.restype = None
        lib.oracle_cache_write.argtypes = [P, P, P, i64, i32, i32, i32, P, P, i64]
        lib.oracle_cache_write.restype = i64
        lib.oracle_copy_blocks.argtypes = [P, P, i64, i32, i32, i32, P, P, i64]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_gather.argtypes = [P, ctypes.c_int, P, i32, i32, i32, i32, i32, P]
        lib.oracle_gather.restype = None
        lib.oracle_decode.argtypes = [P, P, P, ctypes.c_int, P, i32, P, i32, i32, i32, i32, i32,
                                      ctypes.c_double, P, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_e4m3_to_double.argtypes = [P, i64, P]
        lib.oracle_e4m3_to_double.restype = None
        lib.oracle_float_to_e4m3.argtypes = [P, i64, P]
        lib.oracle_float_to_e4m3.restype = None
        lib.oracle_cache_write_fp8.argtypes = [P, P, ctypes.c_int, P, i64, i32, i32, i32, P, P, P, P,
                                               i64]
        lib.oracle_cache_write_fp8.restype = i64
        lib.oracle_decode_fp8.argtypes = [P, P, P, P, P, ctypes.c_int, P, i32, P, i32, i32, i32, i32,
                                          i32, ctypes.c_double, P, ctypes.c_int]
        lib.oracle_decode_fp8.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [P, P, P, ctypes.c_int, P, i32, P, P, i32, P, i64, i32, i32,
                                       i32, i32, ctypes.c_double, P, ctypes.c_int]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path


def compile_source(src, out_path):
    """Compile a pa_oracle.c-like source file to a shared library."""
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _load(handle=None):
    global _lib
    if handle is not None:
        return handle.lib
    if _lib is None:
        build()
        _lib = OracleLib(_LIB_PATH)
    return _lib.lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def max_threads(handle=None):
    return _load(handle).oracle_max_threads()


def bits_to_double(bits, dtype, handle=None):
    """Exact fp64 value of each 16-bit pattern (dtype 'f16' or 'bf16')."""
    bits = _c(np.asarray(bits), np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load(handle).oracle_bits_to_double(_ptr(bits), bits.size, DTYPE_CODES[dtype], _ptr(out))
    return out


def e4m3_to_double(codes, handle=None):
    """fp64 value of each E4M3 byte (NaN for the NaN codes)."""
    codes = _c(np.asarray(codes), np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load(handle).oracle_e4m3_to_double(_ptr(codes), codes.size, _ptr(out))
    return out


def float_to_e4m3(x, handle=None):
    """E4M3 code of each float32 (round to nearest even, saturate to +-448)."""
    x = _c(np.asarray(x, np.float32), np.float32)
    out = np.empty(x.shape, np.uint8)
    _load(handle).oracle_float_to_e4m3(_ptr(x), x.size, _ptr(out))
    return out


def cache_write_fp8(k, v, dtype, slot_mapping, k_scale, v_scale, k_cache8, v_cache8, block_size=16,
                    handle=None):
    """Quantising scatter into copies of the FP8 caches (K [NB,H,16,D], V [NB,H,D,16])."""
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    ks, vs = _c(np.asarray(k_scale, np.float32), np.float32), _c(np.asarray(v_scale, np.float32), np.float32)
    kc, vc = np.array(k_cache8, np.uint8, copy=True), np.array(v_cache8, np.uint8, copy=True)
    T, Hkv, D = k.shape
    nb = kc.shape[0]
    assert kc.shape == (nb, Hkv, block_size, D) and vc.shape == (nb, Hkv, D, block_size)
    bad = _load(handle).oracle_cache_write_fp8(_ptr(k), _ptr(v), DTYPE_CODES[dtype], _ptr(slot_mapping),
                                               T, Hkv, D, block_size, _ptr(ks), _ptr(vs), _ptr(kc),
                                               _ptr(vc), nb)
    return kc, vc, int(bad)


def decode_fp8(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, seq_lens, scale, dtype,
               block_size=16, threads=0, handle=None):
    """fp64 attention over dequantised FP8 K/V (see decode)."""
    q = _c(q, np.uint16)
    k8, v8 = _c(k_cache8, np.uint8), _c(v_cache8, np.uint8)
    ks, vs = _c(np.asarray(k_scale, np.float32), np.float32), _c(np.asarray(v_scale, np.float32), np.float32)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, Hkv, bs, D2 = k8.shape
    assert D2 == D and bs == block_size and v8.shape == (nb, Hkv, D, block_size)
    out = np.empty((B, Hq, D), np.float64)
    rc = _load(handle).oracle_decode_fp8(_ptr(q), _ptr(k8), _ptr(v8), _ptr(ks), _ptr(vs),
                                         DTYPE_CODES[dtype], _ptr(block_tables), block_tables.shape[1],
                                         _ptr(seq_lens), B, Hq, Hkv, D, block_size, float(scale),
                                         _ptr(out), int(threads))
    if rc != 0:
        raise MemoryError("oracle_decode_fp8 could not allocate its gather buffers")
    return out


def cache_write(k, v, slot_mapping, k_cache, v_cache, block_size=16, handle=None):
    """Scatter k/v [T, Hkv, D] (uint16 patterns) into copies of the caches.

    Returns (k_cache', v_cache', n_out_of_range).  Slots < 0 are skipped; so
    are slots past the pool (counted).
    """
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    kc, vc = np.array(k_cache, np.uint16, copy=True), np.array(v_cache, np.uint16, copy=True)
    T, Hkv, D = k.shape
    nb = kc.shape[0]
    assert kc.shape == (nb, Hkv, block_size, D) and vc.shape == kc.shape
    bad = _load(handle).oracle_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, block_size,
                                     _ptr(kc), _ptr(vc), nb)
    return kc, vc, int(bad)


def copy_blocks(k_cache, v_cache, src, dst, block_size=16, handle=None):
    """Copies of the caches with block src[i] copied to block dst[i], K and V.

    Returns (k_cache', v_cache', n_skipped) -- pairs naming a block outside
    the pool are skipped.
    """
    kc, vc = np.array(k_cache, np.uint16, copy=True), np.array(v_cache, np.uint16, copy=True)
    src, dst = _c(np.asarray(src, np.int32), np.int32), _c(np.asarray(dst, np.int32), np.int32)
    nb, Hkv, bs, D = kc.shape
    assert bs == block_size and vc.shape == kc.shape and src.shape == dst.shape
    bad = _load(handle).oracle_copy_blocks(_ptr(kc), _ptr(vc), nb, Hkv, D, block_size, _ptr(src),
                                           _ptr(dst), src.size)
    return kc, vc, int(bad)


def gather(cache, dtype, table_row, seq_len, h, block_size=16, handle=None):
    """Contiguous fp64 [seq_len, D] of KV head h read through one table row."""
    cache = _c(cache, np.uint16)
    table_row = _c(table_row, np.int32)
    nb, Hkv, bs, D = cache.shape
    assert bs == block_size
    out = np.empty((seq_len, D), np.float64)
    _load(handle).oracle_gather(_ptr(cache), DTYPE_CODES[dtype], _ptr(table_row), seq_len, Hkv, h, D,
                          block_size, _ptr(out))
    return out


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, dtype, block_size=16, threads=0,
           handle=None):
    """fp64 attention of each query against its sequence's paged K/V.

    q [B, Hq, D] and the caches [NB, Hkv, bs, D] are uint16 patterns of
    ``dtype``; block_tables [B, max_blocks] int32; seq_lens [B] int32.
    Returns out [B, Hq, D] float64.  threads=0 lets OpenMP choose.
    """
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    nb, Hkv, bs, D2 = k_cache.shape
    assert D2 == D and bs == block_size and v_cache.shape == k_cache.shape
    assert Hq % Hkv == 0 and block_tables.shape[0] == B and seq_lens.shape == (B,)
    out = np.empty((B, Hq, D), np.float64)
    rc = _load(handle).oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype],
                               _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq,
                               Hkv, D, block_size, float(scale), _ptr(out), int(threads))
    if rc != 0:
        raise MemoryError("oracle_decode could not allocate its gather buffers")
    return out


def prefill(q, k_cache, v_cache, block_tables, seq_lens, q_offsets, scale, dtype, rows=None,
            block_size=16, threads=0, handle=None):
    """fp64 causal attention of every query token of each sequence's piece
    (chunked prefill) over the sequence's paged K/V.

    q [Tq, Hq, D] uint16 patterns, the pieces back to back; q_offsets
    [B + 1] int32 with q_offsets[-1] = Tq; seq_lens [B] int32 counts the
    piece's tokens (already in the cache).  ``rows``: query token indices to
    compute (default all).  Returns out [len(rows), Hq, D] float64.
    """
    q = _c(q, np.uint16)
    k_cache, v_cache = _c(k_cache, np.uint16), _c(v_cache, np.uint16)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    q_offsets = _c(q_offsets, np.int32)
    Tq, Hq, D = q.shape
    nb, Hkv, bs, D2 = k_cache.shape
    B = seq_lens.shape[0]
    assert D2 == D and bs == block_size and v_cache.shape == k_cache.shape
    assert Hq % Hkv == 0 and block_tables.shape[0] == B and q_offsets.shape == (B + 1,)
    assert q_offsets[-1] == Tq
    rows_c = None if rows is None else _c(rows, np.int64)
    n = Tq if rows is None else rows_c.shape[0]
    out = np.empty((n, Hq, D), np.float64)
    rc = _load(handle).oracle_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype],
                                      _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                      _ptr(q_offsets), B, None if rows_c is None else _ptr(rows_c),
                                      n, Hq, Hkv, D, block_size, float(scale), _ptr(out),
                                      int(threads))
    if rc == -2:
        raise ValueError("oracle_prefill: a piece is longer than its sequence, q_offsets is "
                         "not non-decreasing from 0, or a row is out of range")
    if rc != 0:
        raise MemoryError("oracle_prefill could not allocate its gather buffers")
    return out


def prefill_dense(q, k_cache, v_cache, block_tables, seq_lens, q_offsets, scale, dtype, rows=None,
                  block_size=16, row_chunk=256, handle=None):
    """The same result as :func:`prefill` -- fp64 causal attention of every
    query token of each sequence's piece over the sequence's paged K/V -- with
    numpy's matrix product as the step that forms the dot products, for
    pieces of thousands of tokens over tens of thousands of keys, where the
    scalar loops of :func:`prefill` take tens of minutes.

    Definition, as for :func:`prefill` ("Yerel LLM sistemlerinde
    backpressure ve olcekleme", section "4. Prefill ve decode"; "vLLM ve
    Triton ile maliyet optimizasyonu", section 03, the scaled dot-product
    attention paragraph): sequence b holds seq_lens[b] tokens; its piece is
    the last n_b = q_offsets[b+1] - q_offsets[b] of them, so query j sits at
    position p = seq_lens[b] - n_b + j and sees tokens 0 .. p.  Query head i
    reads KV head i // G.  Steps, per sequence and KV head: gather the
    sequence's K and V through its table row into contiguous fp64 arrays
    (:func:`gather`, exact); then per query head and group of query rows
    (rows are independent, so grouping them changes nothing):
    S = scale * Q K^T, entries of keys past each row's position set to -inf,
    each row's maximum subtracted, exp, P = exp / row sum, out = P V.
    Returns out [len(rows), Hq, D] float64 (rows default: all).
    """
    q = _c(q, np.uint16)
    block_tables, seq_lens = _c(block_tables, np.int32), _c(seq_lens, np.int32)
    q_offsets = _c(q_offsets, np.int32)
    Tq, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    B = seq_lens.shape[0]
    assert Hq % Hkv == 0 and q_offsets.shape == (B + 1,) and q_offsets[0] == 0
    assert q_offsets[-1] == Tq
    want = np.zeros(Tq, bool)
    if rows is None:
        want[:] = True
    else:
        rows = np.asarray(rows, np.int64)
        if rows.size and (rows.min() < 0 or rows.max() >= Tq):
            raise ValueError("prefill_dense: a row is out of range")
        want[rows] = True
    qd = bits_to_double(q, dtype, handle=handle)
    out = np.zeros((Tq, Hq, D), np.float64)
    for b in range(B):
        a, e = int(q_offsets[b]), int(q_offsets[b + 1])
        n, L = e - a, int(seq_lens[b])
        if n < 0 or n > L:
            raise ValueError("prefill_dense: a piece is longer than its sequence, or q_offsets "
                             "decreases")
        if n == 0 or not want[a:e].any():
            continue
        pos = L - n + np.arange(n)                      # position of each query of the piece

        def one_kv_head(h, a=a, n=n, L=L, pos=pos, b=b):
            K = gather(k_cache, dtype, block_tables[b], L, h, block_size, handle)
            V = gather(v_cache, dtype, block_tables[b], L, h, block_size, handle)
            for c0 in range(0, n, row_chunk):
                rr = np.arange(c0, min(n, c0 + row_chunk))
                rr = rr[want[a + rr]]
                if rr.size == 0:
                    continue
                hi = int(pos[rr[-1]]) + 1               # keys any of these rows can see
                future = np.arange(hi)[None, :] > pos[rr][:, None]
                for g in range(G):
                    i = h * G + g
                    S = qd[a + rr, i, :] @ K[:hi].T
                    S *= scale
                    S[future] = -np.inf
                    S -= S.max(axis=1, keepdims=True)
                    np.exp(S, out=S)                    # S now holds the unnormalised weights
                    out[a + rr, i, :] = (S @ V[:hi]) / S.sum(axis=1, keepdims=True)

        # KV heads are independent and write disjoint outputs; numpy and the
        # gather release the interpreter lock, so they run in threads
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(Hkv, os.cpu_count() or 1)) as ex:
            list(ex.map(one_kv_head, range(Hkv)))
    return out if rows is None else out[rows]
