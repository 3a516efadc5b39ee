"""Seeded synthetic decode batches for paged KV-cache attention.

This module only draws random numbers and lays them out: sequence lengths,
a permutation of physical block ids, query/key/value values and the pool
placement that a block table implies.  It holds no attention arithmetic and
no allocator policy, and it imports neither the CUDA binding nor the oracle,
so both sides can be fed from it.

Workloads (all values ~N(0,1) drawn in fp32 and rounded to the storage type
with round-to-nearest-even; block size 16):

=============  =======================================================
tiny           1 layer, 4 sequences of lengths {1,17,33,100}, 4 query /
               2 KV heads, head_dim 64, fp16, scale 1/8, 24-block pool
llama8b        Llama-3-8B-shaped layer: 32 q / 8 KV heads, head_dim 128,
               bf16, 64 sequences with lengths U{128..2048}
llama70b       Llama-3-70B-shaped layer: 64 q / 8 KV heads, head_dim 128,
               bf16, 256 sequences: 90% of 300+U{1..100} tokens, 10% of
               30000+U{1..4000} tokens (capped at 34000)
long           32 q / 8 KV heads, head_dim 128, bf16, 8 sequences of
               32768 tokens (long-context partitioned decode)
fullstep       32 layers of the 8B shape, 128 sequences in 4 groups of 32;
               each group shares a 1024-token prefix (64 full blocks);
               lengths 1024+U{256..7168}
chunked        (make_prefill_batch) Llama-3-70B-shaped layer: a
               30000-token document prompt prefilled in 8 pieces of
               3750 tokens, each iteration together with one decode
               token of 20 running chats of 300+U{1..100} tokens
=============  =======================================================

Pools hold the needed blocks plus 25% (the tiny one holds 24 blocks); the
physical id of each logical block comes from a seeded permutation.  One
extra "poison" block pads the block tables past each sequence's last block.
With ``poison=True`` every pool slot that holds no token (unused blocks,
the poison block, tails of last blocks, and the slot the new token will be
written to) is NaN, so a stray read shows up as NaN in the output.

Draw order (one torch.Generator seeded from the workload seed): lengths,
permutation, then per layer q, contiguous K, contiguous V, new k, new v.

Each sequence of length L holds L-1 tokens in the pool before the step; the
step writes the new token (position L-1) and attends over all L.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

BLOCK_SIZE = 16

_NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}
_TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str
    num_layers: int
    scale: float
    description: str

    @property
    def group_size(self):
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 4, 4, 2, 64, "f16", 1, 1.0 / 8.0,
                     "1 layer, 4 seqs lens {1,17,33,100}, 4q/2kv heads, d64, fp16, 24-block pool"),
    "llama8b": Workload("llama8b", 64, 32, 8, 128, "bf16", 1, 1.0 / math.sqrt(128),
                        "Llama-3-8B-shaped layer, 64 seqs lens U{128..2048}, 32q/8kv, d128, bf16"),
    "llama70b": Workload("llama70b", 256, 64, 8, 128, "bf16", 1, 1.0 / math.sqrt(128),
                         "Llama-3-70B-shaped layer, 256 seqs: 230 x ~400 + 26 x ~34000 tokens, "
                         "64q/8kv, d128, bf16"),
    "long": Workload("long", 8, 32, 8, 128, "bf16", 1, 1.0 / math.sqrt(128),
                     "8 seqs x 32768 tokens, 32q/8kv, d128, bf16, 512-token partitions"),
    "fullstep": Workload("fullstep", 128, 32, 8, 128, "bf16", 32, 1.0 / math.sqrt(128),
                         "32 layers of the 8B shape, 128 seqs in 4 groups of 32 sharing a "
                         "1024-token prefix, lens 1024+U{256..7168}"),
    "chunked": Workload("chunked", 21, 64, 8, 128, "bf16", 1, 1.0 / math.sqrt(128),
                        "Llama-3-70B-shaped layer, chunked prefill: a 30000-token prompt in 8 "
                        "pieces of 3750 tokens, each with the decode tokens of 20 chats of "
                        "300+U{1..100} tokens"),
}
CHUNK_DOC_TOKENS = 30000
CHUNK_PIECES = 8
CHUNK_CHATS = 20

_SEED_SALT = {"tiny": 11, "llama8b": 22, "llama70b": 33, "long": 44, "fullstep": 55,
              "chunked": 66}
PREFIX_TOKENS = 1024
PREFIX_GROUPS = 4


def _draw_lengths(w, g):
    if w.name == "tiny":
        return torch.tensor([1, 17, 33, 100], dtype=torch.int64)
    if w.name == "llama8b":
        return torch.randint(128, 2049, (w.num_seqs,), generator=g)
    if w.name == "llama70b":
        n_long = round(0.1 * w.num_seqs)
        n_short = w.num_seqs - n_long
        short = 300 + torch.randint(1, 101, (n_short,), generator=g)
        long = torch.clamp(30000 + torch.randint(1, 4001, (n_long,), generator=g), max=34000)
        lens = torch.cat([short, long])
        return lens[torch.randperm(w.num_seqs, generator=g)]
    if w.name == "long":
        return torch.full((w.num_seqs,), 32768, dtype=torch.int64)
    if w.name == "fullstep":
        return PREFIX_TOKENS + torch.randint(256, 7169, (w.num_seqs,), generator=g)
    raise KeyError(w.name)


def workload_lengths(name, seed=0):
    """The sequence lengths make_batch(name, seed) draws (int64 numpy)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000 + _SEED_SALT[name])
    return _draw_lengths(WORKLOADS[name], g).numpy()


def _bits(x, dtype):
    """fp32 tensor -> int16 tensor holding the RNE-rounded 16-bit patterns."""
    return x.to(_TORCH_DTYPE[dtype]).view(torch.int16)


@dataclass
class Layer:
    q: torch.Tensor          # int16 [B, Hq, D] bit patterns
    k_cache: torch.Tensor    # int16 [NB, Hkv, 16, D], the L-1 past tokens placed
    v_cache: torch.Tensor
    new_k: torch.Tensor      # int16 [B, Hkv, D], token L-1 of each sequence
    new_v: torch.Tensor
    k_past: torch.Tensor = None  # int16 [rows, Hkv, D] contiguous draw (keep_contig only)
    v_past: torch.Tensor = None


@dataclass
class Batch:
    workload: Workload
    seq_lens: np.ndarray         # int32 [B], new token included
    block_tables: np.ndarray     # int32 [B, max_blocks], padded with poison_block
    num_blocks: int
    poison_block: int
    slot_mapping: np.ndarray     # int64 [B], slot of token L-1
    layers: list = field(default_factory=list)
    num_unique_blocks: int = 0
    # contiguous-draw bookkeeping (keep_contig only): per sequence, the list
    # of (row_start, row_count) ranges of the past draw that form it, in order
    past_ranges: list = None
    seed: int = 0
    groups: list = None          # (members, shared prefix tokens), contiguous
    has_new: np.ndarray = None   # sequence has a token of its own to write

    # numpy views (host tensors only)
    def np_layer(self, i):
        L = self.layers[i]
        f = lambda t: t.numpy().view(np.uint16)
        return f(L.q), f(L.k_cache), f(L.v_cache), f(L.new_k), f(L.new_v)

    def contiguous_kv(self, layer, b):
        """Contiguous [L_b, Hkv, D] uint16 K and V of sequence b (keep_contig)."""
        Lr = self.layers[layer]
        tail = bool(self.has_new[b])
        ks = [Lr.k_past[s:s + n] for s, n in self.past_ranges[b]] + ([Lr.new_k[b:b + 1]] if tail else [])
        vs = [Lr.v_past[s:s + n] for s, n in self.past_ranges[b]] + ([Lr.new_v[b:b + 1]] if tail else [])
        f = lambda t: torch.cat(t).numpy().view(np.uint16)
        return f(ks), f(vs)

    def logical_kv_bytes(self):
        """Sum over sequences of L x Hkv x D x 2 (K,V) x 2 bytes, per layer."""
        w = self.workload
        return int(self.seq_lens.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 2 * 2

    def unique_kv_bytes(self):
        """KV bytes counting the tokens of a shared prefix once per group."""
        w = self.workload
        per_token = w.num_kv_heads * w.head_dim * 2 * 2
        repeated = sum((m - 1) * p for m, p in self.groups if m > 1)
        return (int(self.seq_lens.astype(np.int64).sum()) - repeated) * per_token

    def group_arrays(self):
        """(offsets [G+1], prefix tokens [G]) int32 for grouped decode."""
        sizes = [m for m, _ in self.groups]
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        return off, np.array([p for _, p in self.groups], np.int32)


def make_batch(name, seed=0, poison=True, num_layers=None, keep_contig=False, device="cpu",
               lens_override=None, groups=None):
    """Build one decode batch.  ``device='cuda'`` draws values on the GPU
    (timing runs; not comparable bit-for-bit with a CPU draw).

    ``groups``: list of (members, prefix_tokens) covering the sequences in
    order; members of a group share the physical blocks of their first
    prefix_tokens tokens (a multiple of 16, at most every member's length).
    The fullstep workload uses 4 groups sharing 1024 tokens."""
    w = WORKLOADS[name]
    layers_n = w.num_layers if num_layers is None else num_layers
    gseed = int(seed) * 1000 + _SEED_SALT[name]
    g = torch.Generator(device="cpu")
    g.manual_seed(gseed)
    lens = _draw_lengths(w, g) if lens_override is None else torch.as_tensor(lens_override, dtype=torch.int64)
    B = int(lens.numel())
    if B != w.num_seqs and lens_override is None:
        raise AssertionError
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    lens_np = lens.numpy().astype(np.int32)

    # --- groups sharing a prefix (contiguous) ---------------------------------------
    if groups is None and name == "fullstep" and lens_override is None:
        groups = [(B // PREFIX_GROUPS, PREFIX_TOKENS)] * PREFIX_GROUPS
    if groups is None:
        groups = [(1, 0)] * B
    if sum(m for m, _ in groups) != B:
        raise ValueError("groups must cover every sequence")
    group_of = np.repeat(np.arange(len(groups)), [m for m, _ in groups])
    prefix_of = np.array([groups[gi][1] for gi in group_of], np.int64)
    for b in range(B):
        if prefix_of[b] % BLOCK_SIZE or prefix_of[b] > lens_np[b]:
            raise ValueError("a shared prefix must be whole blocks within every member")
    shared = [m > 1 and p > 0 for m, p in groups]

    # --- logical block -> unique block index ---------------------------------------
    uniq = []  # per sequence: list of unique block indices
    n_unique = 0
    group_prefix_idx = {}
    for b in range(B):
        row = []
        gi = int(group_of[b])
        for j in range(int(nblk[b])):
            if shared[gi] and j < prefix_of[b] // BLOCK_SIZE:
                key = (gi, j)
                if key not in group_prefix_idx:
                    group_prefix_idx[key] = n_unique
                    n_unique += 1
                row.append(group_prefix_idx[key])
            else:
                row.append(n_unique)
                n_unique += 1
        uniq.append(row)
    if name == "tiny" and lens_override is None:
        pool = 24
    else:
        pool = max(int(math.ceil(1.25 * n_unique)), n_unique + 1)
    perm = torch.randperm(pool, generator=g).numpy().astype(np.int32)
    poison_block = int(perm[n_unique])
    max_nb = max(1, int(nblk.max()) if B else 1)
    tables = np.full((B, max_nb), poison_block, np.int32)
    for b in range(B):
        if uniq[b]:
            tables[b, :len(uniq[b])] = perm[np.asarray(uniq[b], np.int64)]
    # A member whose whole length lies in the shared prefix has no token of
    # its own to write: its last token is part of the shared draw.
    pos = lens_np.astype(np.int64) - 1
    has_new = (pos >= 0) & ~np.array([shared[int(group_of[b])] and lens_np[b] <= prefix_of[b]
                                      for b in range(B)], bool)
    slot = np.where(has_new, tables[np.arange(B), np.maximum(pos, 0) // BLOCK_SIZE].astype(np.int64)
                    * BLOCK_SIZE + np.maximum(pos, 0) % BLOCK_SIZE, -1).astype(np.int64)

    # --- placement of the tokens already cached (layout only) ------------------------
    # Draw rows, per group in order: the shared prefix once, then each member's
    # own tokens before its new one; a lone sequence is a group of one.
    ranges = [None] * B
    dst_blk, dst_off = [], []
    row = 0

    def place(b, t0, t1):
        nonlocal row
        t = np.arange(t0, t1, dtype=np.int64)
        dst_blk.append(tables[b, t // BLOCK_SIZE].astype(np.int64))
        dst_off.append(t % BLOCK_SIZE)
        start = row
        row += t1 - t0
        return (start, t1 - t0)

    first = 0
    for gi, (M, pre) in enumerate(groups):
        members = range(first, first + M)
        first += M
        if shared[gi]:
            pr = place(members[0], 0, pre)
            for b in members:
                end_b = int(lens_np[b]) - 1 if has_new[b] else int(lens_np[b])
                ranges[b] = [pr] + ([place(b, pre, end_b)] if end_b > pre else [])
        else:
            for b in members:
                ranges[b] = [place(b, 0, max(int(lens_np[b]) - 1, 0))]
    dst_blk = np.concatenate(dst_blk) if dst_blk else np.zeros(0, np.int64)
    dst_off = np.concatenate(dst_off) if dst_off else np.zeros(0, np.int64)
    n_rows = row

    H, Hq, D = w.num_kv_heads, w.num_q_heads, w.head_dim
    dev = torch.device(device)
    gv = g
    if dev.type == "cuda":
        gv = torch.Generator(device=dev)
        gv.manual_seed(gseed + 7)
    fill = _NAN_BITS[w.dtype] if poison else 0
    fill_i16 = fill - 65536 if fill >= 32768 else fill
    t_blk = torch.from_numpy(dst_blk).to(dev)
    t_off = torch.from_numpy(dst_off).to(dev)
    layers = []
    for _ in range(layers_n):
        q = _bits(torch.randn((B, Hq, D), generator=gv, device=dev), w.dtype)
        k_past = _bits(torch.randn((n_rows, H, D), generator=gv, device=dev), w.dtype)
        v_past = _bits(torch.randn((n_rows, H, D), generator=gv, device=dev), w.dtype)
        new_k = _bits(torch.randn((B, H, D), generator=gv, device=dev), w.dtype)
        new_v = _bits(torch.randn((B, H, D), generator=gv, device=dev), w.dtype)
        kc = torch.full((pool, H, BLOCK_SIZE, D), fill_i16, dtype=torch.int16, device=dev)
        vc = torch.full((pool, H, BLOCK_SIZE, D), fill_i16, dtype=torch.int16, device=dev)
        if n_rows:
            kc[t_blk, :, t_off, :] = k_past
            vc[t_blk, :, t_off, :] = v_past
        Lr = Layer(q, kc, vc, new_k, new_v)
        if keep_contig:
            Lr.k_past, Lr.v_past = k_past, v_past
        else:
            del k_past, v_past
        layers.append(Lr)
    bt = Batch(w, lens_np, tables, pool, poison_block, slot, layers, n_unique,
               ranges if keep_contig else None, seed)
    bt.groups = list(groups)
    bt.has_new = has_new
    return bt


def place_new_tokens(batch, layer):
    """Pool copies with each sequence's new token placed at its slot (layout
    only; used to build decode-only inputs without running a cache write)."""
    Lr = batch.layers[layer]
    kc, vc = Lr.k_cache.clone(), Lr.v_cache.clone()
    s = torch.from_numpy(batch.slot_mapping).to(kc.device)
    ok = s >= 0
    kc[s[ok] // BLOCK_SIZE, :, s[ok] % BLOCK_SIZE, :] = Lr.new_k[ok]
    vc[s[ok] // BLOCK_SIZE, :, s[ok] % BLOCK_SIZE, :] = Lr.new_v[ok]
    return kc, vc


def relabel_blocks(batch, seed):
    """Same logical contents under another physical placement: a seeded
    permutation of the pool ids applied to tables, slots and pools."""
    g = torch.Generator(device="cpu")
    g.manual_seed(10_000 + int(seed))
    sigma = torch.randperm(batch.num_blocks, generator=g).numpy().astype(np.int32)
    new = Batch(batch.workload, batch.seq_lens.copy(), sigma[batch.block_tables],
                batch.num_blocks, int(sigma[batch.poison_block]), None, [],
                batch.num_unique_blocks, batch.past_ranges, batch.seed, batch.groups,
                batch.has_new)
    s = batch.slot_mapping
    new.slot_mapping = np.where(s >= 0, sigma[np.maximum(s, 0) // BLOCK_SIZE].astype(np.int64)
                                * BLOCK_SIZE + np.maximum(s, 0) % BLOCK_SIZE, -1)
    inv = np.empty_like(sigma)
    inv[sigma] = np.arange(batch.num_blocks, dtype=np.int32)
    idx = torch.from_numpy(inv.astype(np.int64))
    for Lr in batch.layers:
        ix = idx.to(Lr.k_cache.device)
        n = Layer(Lr.q, Lr.k_cache[ix], Lr.v_cache[ix], Lr.new_k, Lr.new_v, Lr.k_past, Lr.v_past)
        new.layers.append(n)
    return new


# ----------------------------------------------------------------------------------
# Multi-query batches (chunked prefill)

@dataclass
class PrefillBatch:
    workload: Workload
    seq_lens: np.ndarray         # int32 [B], the piece's tokens included
    pieces: np.ndarray           # int32 [B], query tokens of each sequence (>= 1)
    q_offsets: np.ndarray        # int32 [B + 1], pieces back to back
    block_tables: np.ndarray     # int32 [B, max_blocks], padded with poison_block
    num_blocks: int
    poison_block: int
    slot_mapping: np.ndarray     # int64 [Tq], slots of the pieces' tokens
    q: torch.Tensor              # int16 [Tq, Hq, D] bit patterns
    k_cache: torch.Tensor        # int16 [NB, Hkv, 16, D], the L - piece past tokens placed
    v_cache: torch.Tensor
    new_k: torch.Tensor          # int16 [Tq, Hkv, D], the pieces' keys and values
    new_v: torch.Tensor
    k_past: torch.Tensor = None  # int16 [rows, Hkv, D] contiguous past draw (keep_contig)
    v_past: torch.Tensor = None
    past_start: np.ndarray = None  # int64 [B], first row of each sequence's past draw

    @property
    def num_q_tokens(self):
        return int(self.q_offsets[-1])

    def contiguous_kv(self, b):
        """Contiguous [L_b, Hkv, D] uint16 K and V of sequence b (keep_contig)."""
        n_past = int(self.seq_lens[b] - self.pieces[b])
        s0, q0, q1 = int(self.past_start[b]), int(self.q_offsets[b]), int(self.q_offsets[b + 1])
        f = lambda a, n: torch.cat([a[s0:s0 + n_past], n[q0:q1]]).numpy().view(np.uint16)
        return f(self.k_past, self.new_k), f(self.v_past, self.new_v)

    def placed_pools(self):
        """Pool copies with the pieces' tokens placed at their slots (layout
        only; the inputs of an attention call that follows the cache write)."""
        kc, vc = self.k_cache.clone(), self.v_cache.clone()
        s = torch.from_numpy(self.slot_mapping).to(kc.device)
        kc[s // BLOCK_SIZE, :, s % BLOCK_SIZE, :] = self.new_k
        vc[s // BLOCK_SIZE, :, s % BLOCK_SIZE, :] = self.new_v
        return kc, vc


def chunked_iteration_shape(iteration, seed=0):
    """(lens, pieces) of iteration k (1..8) of the chunked workload: the
    document (sequence 0) holds k pieces of 3750 tokens, the last of them
    its query; each chat holds its drawn length + k tokens, one query."""
    if not 1 <= iteration <= CHUNK_PIECES:
        raise ValueError("iteration must be in 1..8")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000 + _SEED_SALT["chunked"])
    chats = 300 + torch.randint(1, 101, (CHUNK_CHATS,), generator=g).numpy()
    piece = CHUNK_DOC_TOKENS // CHUNK_PIECES
    lens = np.concatenate([[piece * iteration], chats + iteration]).astype(np.int32)
    pieces = np.concatenate([[piece], np.ones(CHUNK_CHATS, np.int64)]).astype(np.int32)
    return lens, pieces


def make_prefill_batch(name, seed=0, iteration=CHUNK_PIECES, poison=True, keep_contig=False,
                       device="cpu", lens=None, pieces=None):
    """One multi-query batch: sequence b holds lens[b] tokens once its piece
    of pieces[b] query tokens is written; the lens[b] - pieces[b] earlier
    tokens are already in the pool.  Defaults: the chunked workload at
    ``iteration``; ``lens``/``pieces`` override the shape (any workload's
    head layout).  Draw order: permutation, q, contiguous past K, past V,
    the pieces' k, v."""
    w = WORKLOADS[name]
    if lens is None:
        if name != "chunked":
            raise ValueError("lens/pieces are required for workloads other than chunked")
        lens, pieces = chunked_iteration_shape(iteration, seed)
    lens = np.asarray(lens, np.int64)
    pieces = np.asarray(pieces, np.int64)
    if lens.shape != pieces.shape or (pieces < 0).any() or (pieces > lens).any():
        raise ValueError("every piece must hold 0..len tokens")
    gseed = int(seed) * 1000 + _SEED_SALT[name] + 500 + int(iteration)
    g = torch.Generator(device="cpu")
    g.manual_seed(gseed)
    B = lens.shape[0]
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    n_unique = int(nblk.sum())
    pool = max(int(math.ceil(1.25 * n_unique)), n_unique + 1)
    perm = torch.randperm(pool, generator=g).numpy().astype(np.int32)
    poison_block = int(perm[n_unique])
    tables = np.full((B, max(1, int(nblk.max()))), poison_block, np.int32)
    first = np.concatenate([[0], np.cumsum(nblk)])
    for b in range(B):
        tables[b, :nblk[b]] = perm[first[b]:first[b + 1]]
    q_off = np.concatenate([[0], np.cumsum(pieces)]).astype(np.int32)
    Tq = int(q_off[-1])
    # slots: the past tokens (pool placement) and the pieces' tokens (written by the step)
    past_blk, past_off, new_slot = [], [], []
    past_start = np.zeros(B, np.int64)
    rows = 0
    for b in range(B):
        n_past = int(lens[b] - pieces[b])
        t = np.arange(n_past, dtype=np.int64)
        past_blk.append(tables[b, t // BLOCK_SIZE].astype(np.int64))
        past_off.append(t % BLOCK_SIZE)
        past_start[b] = rows
        rows += n_past
        t = np.arange(n_past, int(lens[b]), dtype=np.int64)
        new_slot.append(tables[b, t // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE + t % BLOCK_SIZE)
    past_blk = np.concatenate(past_blk)
    past_off = np.concatenate(past_off)
    slots = np.concatenate(new_slot)

    H, Hq, D = w.num_kv_heads, w.num_q_heads, w.head_dim
    dev = torch.device(device)
    gv = g
    if dev.type == "cuda":
        gv = torch.Generator(device=dev)
        gv.manual_seed(gseed + 7)
    fill = _NAN_BITS[w.dtype] if poison else 0
    fill_i16 = fill - 65536 if fill >= 32768 else fill
    q = _bits(torch.randn((Tq, Hq, D), generator=gv, device=dev), w.dtype)
    k_past = _bits(torch.randn((rows, H, D), generator=gv, device=dev), w.dtype)
    v_past = _bits(torch.randn((rows, H, D), generator=gv, device=dev), w.dtype)
    new_k = _bits(torch.randn((Tq, H, D), generator=gv, device=dev), w.dtype)
    new_v = _bits(torch.randn((Tq, H, D), generator=gv, device=dev), w.dtype)
    kc = torch.full((pool, H, BLOCK_SIZE, D), fill_i16, dtype=torch.int16, device=dev)
    vc = torch.full((pool, H, BLOCK_SIZE, D), fill_i16, dtype=torch.int16, device=dev)
    if rows:
        tb, to = torch.from_numpy(past_blk).to(dev), torch.from_numpy(past_off).to(dev)
        kc[tb, :, to, :] = k_past
        vc[tb, :, to, :] = v_past
    pb = PrefillBatch(w, lens.astype(np.int32), pieces.astype(np.int32), q_off, tables, pool,
                      poison_block, slots, q, kc, vc, new_k, new_v)
    if keep_contig:
        pb.k_past, pb.v_past, pb.past_start = k_past, v_past, past_start
    return pb
