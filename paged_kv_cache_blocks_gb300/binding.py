"""ctypes binding of libpa (include/pa.h): argument marshalling only.

Every function keeps its C name.  Tensors are torch tensors; only their
data pointers, sizes and the current CUDA stream cross the ABI, and every
step of the computation runs in libpa's kernels.  There is no fallback:
if libpa.so is missing or fails to load, the first call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_UNSUPPORTED, PA_ERR_SHARED_WRITE, PA_ERR_CUDA, \
    PA_ERR_DEVICE = range(7)
PA_F16, PA_BF16 = 0, 1
PA_DEVERR_SEQ_LEN, PA_DEVERR_BLOCK_ID, PA_DEVERR_TIMEOUT, PA_DEVERR_GROUP, PA_DEVERR_PLAN = \
    1, 2, 4, 8, 16
BLOCK_SIZE = 16

_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_OOM", 3: "PA_ERR_UNSUPPORTED",
           4: "PA_ERR_SHARED_WRITE", 5: "PA_ERR_CUDA", 6: "PA_ERR_DEVICE"}


class PaError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_STATUS.get(code, code)}: {msg}")
        self.code = code


class PaStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("num_blocks", "free_blocks", "used_blocks",
                                             "shared_blocks", "refs", "seqs", "frag_tokens")]


class PaDecodeOpts(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("event_before_main", ctypes.c_void_p), ("event_after_main", ctypes.c_void_p),
                ("partition_tokens", ctypes.c_int32), ("reserved32", ctypes.c_int32),
                ("reserved", ctypes.c_int64 * 3)]


_lib = None


PA_DECODE_REUSE_PLAN = 1


def _opts(variant, events, stream, flags=0, partition_tokens=0):
    """pa_decode_opts for a call, or None for the defaults."""
    if not (variant or events or flags or partition_tokens):
        return None
    o = PaDecodeOpts()
    o.variant = variant
    o.flags = flags
    o.partition_tokens = partition_tokens
    if events:
        for e in events:       # torch creates the CUDA event lazily, on first record
            if not e.cuda_event:
                e.record(torch.cuda.current_stream() if stream is None else stream)
        o.event_before_main = events[0].cuda_event
        o.event_after_main = events[1].cuda_event
    return ctypes.byref(o)

P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "pa_last_error_string": ([], ctypes.c_char_p),
    "pa_version": ([], ctypes.c_char_p),
    "pa_alloc_create": ([I32, I32, P, P], ctypes.c_int),
    "pa_alloc_destroy": ([P], None),
    "pa_seq_create": ([P, P], ctypes.c_int),
    "pa_seq_fork": ([P, I64, I32, P], ctypes.c_int),
    "pa_seq_free": ([P, I64], ctypes.c_int),
    "pa_seq_append_slots": ([P, P, I32, I32, P, P, P, I32, P, P, I32, P], ctypes.c_int),
    "pa_seq_block_table": ([P, P, I32, I32, P, P], ctypes.c_int),
    "pa_alloc_stats": ([P, P], ctypes.c_int),
    "pa_cache_write": ([P, P, P, I32, I32, I32, P, P, I64, I32, P], ctypes.c_int),
    "pa_copy_blocks": ([P, P, I64, I32, I32, P, P, I32, P], ctypes.c_int),
    "pa_decode_workspace_bytes": ([I32, I32, I32, I32], SZ),
    "pa_decode": ([P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P, SZ, P],
                  ctypes.c_int),
    "pa_decode_ex": ([P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P, SZ, P, P],
                     ctypes.c_int),
    "pa_decode_check": ([P, P, P], ctypes.c_int),
    "pa_cache_write_fp8": ([P, P, P, I32, I32, I32, P, P, P, P, I64, I32, P], ctypes.c_int),
    "pa_decode_fp8": ([P, P, P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P, SZ, P, P],
                      ctypes.c_int),
    "pa_decode_grouped_workspace_bytes": ([I32, I32, I32, I32], SZ),
    "pa_decode_grouped": ([P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P, I32, P,
                           P, SZ, P, P], ctypes.c_int),
    "pa_decode_noalloc": ([P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F32, I32, P, P],
                          ctypes.c_int),
    "pa_selftest_bounded_wait": ([I64, P, P], ctypes.c_int),
    "pa_prefill_workspace_bytes": ([I32, I32, I32, I32], SZ),
    "pa_prefill": ([P, P, P, I64, P, I32, P, P, I32, I32, I32, I32, I32, I32, F32, I32, P, P, SZ, P,
                    P], ctypes.c_int),
}


def lib():
    """Load libpa.so (raises if it is missing: there is no other path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so not built ({LIB_PATH}); run "
                               "`python -m paged_kv_cache_blocks_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _check(rc, what):
    if rc != PA_OK:
        raise PaError(rc, f"{what}: {lib().pa_last_error_string().decode()}")


def _dtype_code(t, dtype=None):
    if dtype is not None:
        return {"f16": PA_F16, "bf16": PA_BF16, PA_F16: PA_F16, PA_BF16: PA_BF16}[dtype]
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError("pass dtype='f16' or 'bf16' for int16 bit-pattern tensors")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("libpa device arguments must be contiguous CUDA tensors")


def _need(cond, what):
    """Argument check that stays on under ``python -O`` (unlike assert)."""
    if not cond:
        raise TypeError(what)


def _need_reuse_workspace(reuse_plan, workspace):
    """A reused plan lives in the planning call's workspace: a fresh one has none."""
    if reuse_plan and workspace is None:
        raise ValueError("reuse_plan needs the workspace of the call that made the plan")


# --------------------------------------------------------------------------- device calls

def pa_cache_write(k, v, slot_mapping, k_cache, v_cache, dtype=None, stream=None):
    """Scatter k/v [T, Hkv, D] into the caches [NB, Hkv, 16, D] at slot_mapping (int64)."""
    _need_cuda(k, v, slot_mapping, k_cache, v_cache)
    _need(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    T, H, D = k.shape
    rc = lib().pa_cache_write(_ptr(k), _ptr(v), _ptr(slot_mapping), T, H, D, _ptr(k_cache),
                              _ptr(v_cache), k_cache.shape[0], _dtype_code(k, dtype), _stream(stream))
    _check(rc, "pa_cache_write")


def pa_copy_blocks(k_cache, v_cache, src, dst, stream=None):
    """Copy-on-write: block dst[i] of both caches becomes a copy of block src[i]."""
    _need_cuda(k_cache, v_cache, src, dst)
    _need(src.dtype == torch.int32 and dst.dtype == torch.int32 and src.shape == dst.shape,
          "src and dst must be int32 tensors of one shape")
    NB, Hkv, _, D = k_cache.shape
    rc = lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), NB, Hkv, D, _ptr(src), _ptr(dst),
                              src.numel(), _stream(stream))
    _check(rc, "pa_copy_blocks")


def pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len):
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len))


def pa_decode(q, k_cache, v_cache, block_tables, seq_lens, scale, max_seq_len=0, out=None,
              workspace=None, dtype=None, variant=0, events=None, stream=None, reuse_plan=False,
              partition_tokens=0):
    """out[b, i] = softmax(scale q[b,i] K_b^T) V_b over each sequence's paged K/V.

    q [B, Hq, D]; caches [NB, Hkv, 16, D]; block_tables [B, max_blocks] int32;
    seq_lens [B] int32 (device).  Returns out [B, Hq, D].  ``workspace`` is a
    uint8 CUDA tensor of at least pa_decode_workspace_bytes() bytes (one is
    allocated when None).  ``events`` = (before, after) torch.cuda.Event pair
    recorded around the attention kernel.  ``reuse_plan``: skip the prep
    kernel and reuse the plan of the previous call on this workspace (same
    lengths and shapes; e.g. the later layers of one step).
    ``partition_tokens``: 0 (the prep kernel chooses) or 512 / 1024 / 2048.
    """
    _need_reuse_workspace(reuse_plan, workspace)
    _need_cuda(q, k_cache, v_cache, block_tables, seq_lens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    B, Hq, D = q.shape
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    mb = block_tables.shape[1]
    msl = max_seq_len if max_seq_len > 0 else mb * BLOCK_SIZE
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(pa_decode_workspace_bytes(B, Hq, D, msl), 256),
                                dtype=torch.uint8, device=q.device)
    opts = _opts(variant, events, stream, PA_DECODE_REUSE_PLAN if reuse_plan else 0,
                 partition_tokens)
    rc = lib().pa_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), mb,
                            _ptr(seq_lens), B, msl, Hq, Hkv, D, float(scale), _dtype_code(q, dtype),
                            _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream), opts)
    _check(rc, "pa_decode")
    return out


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, seq_lens, scale, max_seq_len=0, out=None,
                      dtype=None, stream=None):
    """pa_decode for callers that cannot allocate: the scratch is a fixed
    64 MiB static device array inside libpa (batches needing more are
    rejected).  Allocates nothing itself when ``out`` is given."""
    _need_cuda(q, k_cache, v_cache, block_tables, seq_lens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    rc = lib().pa_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                 _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
                                 max_seq_len, Hq, k_cache.shape[1], D, float(scale),
                                 _dtype_code(q, dtype), _ptr(out), _stream(stream))
    _check(rc, "pa_decode_noalloc")
    return out


def pa_cache_write_fp8(k, v, slot_mapping, k_scale, v_scale, k_cache8, v_cache8, dtype=None,
                       stream=None):
    """Quantise k/v [T, Hkv, 128] (16-bit) to E4M3 into k_cache8 [NB, Hkv, 16, 128]
    and the dimension-major v_cache8 [NB, Hkv, 128, 16] (uint8 tensors)."""
    _need_cuda(k, v, slot_mapping, k_scale, v_scale, k_cache8, v_cache8)
    _need(k_cache8.dtype == torch.uint8 and v_cache8.dtype == torch.uint8,
          "FP8 caches must be uint8 tensors of E4M3 codes")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32,
          "k_scale and v_scale must be float32")
    T, H, D = k.shape
    rc = lib().pa_cache_write_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), T, H, D, _ptr(k_scale),
                                  _ptr(v_scale), _ptr(k_cache8), _ptr(v_cache8), k_cache8.shape[0],
                                  _dtype_code(k, dtype), _stream(stream))
    _check(rc, "pa_cache_write_fp8")


def pa_decode_fp8(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, seq_lens, scale,
                  max_seq_len=0, out=None, workspace=None, dtype=None, stream=None, events=None,
                  reuse_plan=False):
    """pa_decode over E4M3 caches (see pa_cache_write_fp8 for the layout);
    ``events`` and ``reuse_plan`` as for pa_decode."""
    _need_reuse_workspace(reuse_plan, workspace)
    _need_cuda(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, seq_lens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32,
          "k_scale and v_scale must be float32")
    B, Hq, D = q.shape
    NB, Hkv = k_cache8.shape[0], k_cache8.shape[1]
    mb = block_tables.shape[1]
    msl = max_seq_len if max_seq_len > 0 else mb * BLOCK_SIZE
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(pa_decode_workspace_bytes(B, Hq, D, msl), 256),
                                dtype=torch.uint8, device=q.device)
    rc = lib().pa_decode_fp8(_ptr(q), _ptr(k_cache8), _ptr(v_cache8), _ptr(k_scale), _ptr(v_scale), NB,
                             _ptr(block_tables), mb, _ptr(seq_lens), B, msl, Hq, Hkv, D, float(scale),
                             _dtype_code(q, dtype), _ptr(out), _ptr(workspace), workspace.numel(),
                             _stream(stream),
                             _opts(0, events, stream, PA_DECODE_REUSE_PLAN if reuse_plan else 0))
    _check(rc, "pa_decode_fp8")
    return out


def pa_decode_grouped_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len):
    return int(lib().pa_decode_grouped_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len))


def pa_decode_grouped(q, k_cache, v_cache, block_tables, seq_lens, scale, group_offsets,
                      group_prefix_tokens, max_seq_len=0, out=None, workspace=None, dtype=None,
                      stream=None, variant=0, events=None, reuse_plan=False):
    """pa_decode where contiguous groups of sequences share a prefix:
    group_offsets [G+1] and group_prefix_tokens [G] are int32 CUDA tensors.
    ``events`` bracket the attention kernel over the members' own tokens."""
    _need_reuse_workspace(reuse_plan, workspace)
    _need_cuda(q, k_cache, v_cache, block_tables, seq_lens, group_offsets, group_prefix_tokens)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(group_offsets.dtype == torch.int32 and group_prefix_tokens.dtype == torch.int32,
          "group_offsets and group_prefix_tokens must be int32")
    B, Hq, D = q.shape
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    mb = block_tables.shape[1]
    msl = max_seq_len if max_seq_len > 0 else mb * BLOCK_SIZE
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(pa_decode_grouped_workspace_bytes(B, Hq, D, msl), 256),
                                dtype=torch.uint8, device=q.device)
    rc = lib().pa_decode_grouped(_ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), mb,
                                 _ptr(seq_lens), B, msl, Hq, Hkv, D, float(scale),
                                 _dtype_code(q, dtype), _ptr(group_offsets),
                                 _ptr(group_prefix_tokens), group_prefix_tokens.numel(), _ptr(out),
                                 _ptr(workspace), workspace.numel(), _stream(stream),
                                 _opts(variant, events, stream,
                                       PA_DECODE_REUSE_PLAN if reuse_plan else 0))
    _check(rc, "pa_decode_grouped")
    return out


def pa_prefill_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads):
    return int(lib().pa_prefill_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads))


PREFILL_VARIANTS = {"auto": 0, "mma": 2, "tc": 3}


def pa_prefill(q, k_cache, v_cache, block_tables, seq_lens, q_offsets, scale, max_seq_len=0,
               out=None, workspace=None, dtype=None, stream=None, events=None, variant=0):
    """Causal attention of each sequence's piece of query tokens (chunked
    prefill; a decode token is a piece of one) over its paged K/V.

    q [Tq, Hq, D], the pieces back to back; q_offsets [B + 1] int32 (device)
    with q_offsets[-1] = Tq; seq_lens [B] int32 count the piece's tokens,
    whose K/V are already in the cache.  ``variant``: 0 auto (tcgen05 at
    head_dim 128), 2 mma.sync, 3 tcgen05.  Returns out [Tq, Hq, D].
    """
    _need_cuda(q, k_cache, v_cache, block_tables, seq_lens, q_offsets)
    _need(block_tables.dtype == torch.int32 and seq_lens.dtype == torch.int32,
          "block_tables and seq_lens must be int32")
    _need(q_offsets.dtype == torch.int32, "q_offsets must be int32")
    Tq, Hq, D = q.shape
    NB, Hkv = k_cache.shape[0], k_cache.shape[1]
    B = seq_lens.shape[0]
    mb = block_tables.shape[1]
    msl = max_seq_len if max_seq_len > 0 else mb * BLOCK_SIZE
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(pa_prefill_workspace_bytes(B, Tq, Hq, Hkv), 256),
                                dtype=torch.uint8, device=q.device)
    rc = lib().pa_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), NB, _ptr(block_tables), mb,
                          _ptr(seq_lens), _ptr(q_offsets), B, Tq, msl, Hq, Hkv, D, float(scale),
                          _dtype_code(q, dtype), _ptr(out), _ptr(workspace), workspace.numel(),
                          _stream(stream), _opts(variant, events, stream))
    _check(rc, "pa_prefill")
    return out


def pa_selftest_bounded_wait(limit_ns, stream=None):
    """Run the bounded-wait diagnostic; returns (wait succeeded, error bits,
    abort flag, microseconds waited) once it has finished."""
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    _check(lib().pa_selftest_bounded_wait(int(limit_ns), _ptr(status), _stream(stream)),
           "pa_selftest_bounded_wait")
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    return tuple(int(x) for x in status.cpu().tolist())


def pa_decode_check(workspace, stream=None):
    """Device error bits left by the last decode on this workspace (0 = clean)."""
    bits = ctypes.c_int32(0)
    rc = lib().pa_decode_check(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    if rc not in (PA_OK, PA_ERR_DEVICE):
        _check(rc, "pa_decode_check")
    return bits.value


# --------------------------------------------------------------------------- allocator

class Allocator:
    """Host block allocator (free queue, ref counts, copy-on-write)."""

    def __init__(self, num_blocks, free_order=None, block_size=BLOCK_SIZE):
        self._h = ctypes.c_void_p()
        arr = None
        if free_order is not None:
            arr = (ctypes.c_int32 * num_blocks)(*[int(x) for x in free_order])
        _check(lib().pa_alloc_create(num_blocks, block_size, arr, ctypes.byref(self._h)),
               "pa_alloc_create")

    def close(self):
        if self._h:
            lib().pa_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def seq_create(self):
        sid = ctypes.c_int64()
        _check(lib().pa_seq_create(self._h, ctypes.byref(sid)), "pa_seq_create")
        return sid.value

    def seq_fork(self, parent, prefix_tokens):
        sid = ctypes.c_int64()
        _check(lib().pa_seq_fork(self._h, parent, prefix_tokens, ctypes.byref(sid)), "pa_seq_fork")
        return sid.value

    def seq_free(self, sid):
        _check(lib().pa_seq_free(self._h, sid), "pa_seq_free")

    def append_slots(self, seq_ids, tokens_each, block_table=None, seq_lens=None, cow_capacity=None):
        """Returns (slots list, [(src, dst) copy-on-write pairs]).  Optional
        block_table ([n, max_blocks] int32) / seq_lens ([n] int32) CPU tensors
        (or numpy arrays) are updated in place."""
        n = len(seq_ids)
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        slots = (ctypes.c_int64 * max(n * tokens_each, 1))()
        cap = n if cow_capacity is None else cow_capacity
        src = (ctypes.c_int32 * max(cap, 1))()
        dst = (ctypes.c_int32 * max(cap, 1))()
        ncow = ctypes.c_int32()
        tab_p, mb, len_p = None, 0, None
        if block_table is not None:
            tab_p = ctypes.c_void_p(block_table.ctypes.data if hasattr(block_table, "ctypes")
                                    else block_table.data_ptr())
            mb = block_table.shape[1]
        if seq_lens is not None:
            len_p = ctypes.c_void_p(seq_lens.ctypes.data if hasattr(seq_lens, "ctypes")
                                    else seq_lens.data_ptr())
        _check(lib().pa_seq_append_slots(self._h, ids, n, tokens_each, slots, src, dst, cap,
                                         ctypes.byref(ncow), tab_p, mb, len_p),
               "pa_seq_append_slots")
        return list(slots[:n * tokens_each]), [(src[i], dst[i]) for i in range(ncow.value)]

    def append_slots_into(self, ids_arr, n, tokens_each, slots_ptr, table_ptr, max_blocks,
                          lens_ptr):
        """Fast path for a step loop: raw pointers to preallocated host buffers
        (ids int64[n], slots int64[n*tokens], table int32[n, max_blocks],
        lens int32[n]).  Copy-on-write is not expected here (capacity 0)."""
        _check(lib().pa_seq_append_slots(self._h, ids_arr, n, tokens_each, slots_ptr, None, None, 0,
                                         None, table_ptr, max_blocks, lens_ptr),
               "pa_seq_append_slots")

    def block_table(self, seq_ids, max_blocks):
        n = len(seq_ids)
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        tab = (ctypes.c_int32 * max(n * max_blocks, 1))()
        lens = (ctypes.c_int32 * max(n, 1))()
        _check(lib().pa_seq_block_table(self._h, ids, n, max_blocks, tab, lens),
               "pa_seq_block_table")
        rows = [list(tab[i * max_blocks:(i + 1) * max_blocks]) for i in range(n)]
        return rows, list(lens[:n])

    def stats(self):
        st = PaStats()
        _check(lib().pa_alloc_stats(self._h, ctypes.byref(st)), "pa_alloc_stats")
        return {"num_blocks": st.num_blocks, "free": st.free_blocks, "used": st.used_blocks,
                "shared": st.shared_blocks, "refs": st.refs, "seqs": st.seqs,
                "frag_tokens": st.frag_tokens}


# The two calls of the decode step under their short names as well:
# cache_write(k, v, slot_mapping, k_cache, v_cache) and
# decode(q, k_cache, v_cache, block_tables, seq_lens, scale) -> out.
cache_write = pa_cache_write
decode = pa_decode
