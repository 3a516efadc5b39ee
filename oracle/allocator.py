"""Reference model of the paged KV block allocator (host side).

TEST INFRASTRUCTURE ONLY: the product's allocator is the C++ one inside the
CUDA library; this model is what the tests hold it to.  Plain Python, one
dictionary per sequence, no cleverness.

What it models, and where that is defined:

* Fixed blocks of ``block_size`` (16) tokens, taken from a pool of free
  physical blocks only when the sequence's current block is full; waste is
  at most ``block_size - 1`` tokens per sequence.
  "vLLM Nedir? PagedAttention ile Production LLM Serving", section
  "PagedAttention"; "vLLM ve Triton ile maliyet optimizasyonu", section 03,
  step 3 (on-demand allocation).
* allocate_slots: 17 new tokens with 16-token blocks take 2 blocks.
  "vLLM Nedir?", section "Bir istek motorun icinde", step 2.
* Freed blocks go back to the free queue.  "vLLM Nedir?", same section,
  step 5.
* Blocks shared by several sequences (common prefix, beam search, parallel
  sampling) carry a reference count; a block returns to the free queue only
  when its last reference is dropped.  "vLLM Nedir?", section
  "PagedAttention", last paragraph; "vLLM ve Triton", section 03.
* Copy-on-write: a shared block is copied when one holder writes into it.
  "vLLM ve Triton", section 03.

Readings where the pages are silent (the C++ allocator follows the same
ones):

* The free queue is first-in first-out.  Its initial order is given by the
  caller (a permutation of the block ids); freed blocks join at the back,
  in the order of the freed sequence's table.
* append_slots is all-or-nothing: if the free queue cannot cover every new
  block (and copy-on-write target) of the call, nothing changes and OOM is
  returned.
* A call that would write into a block other sequences still hold, but
  gives no room (``cow_capacity``) to report the copy that must come first,
  is refused with SHARED_WRITE before anything changes: the write would
  alter the other holders' tokens ("vLLM ve Triton", section 03, the
  copy-on-write paragraph).  This check precedes the OOM check.
* A fork shares the blocks covering the parent's first ``prefix_tokens``
  tokens.  If the last of them is only partly covered, the next write into
  it from either holder triggers copy-on-write.
* Sequence ids are handed out as 0, 1, 2, ... and never reused.
"""

OK, ERR_INVALID, ERR_OOM, ERR_SHARED_WRITE = 0, 1, 2, 4


class AllocError(Exception):
    def __init__(self, code, msg):
        super().__init__(msg)
        self.code = code


class AllocatorModel:
    def __init__(self, num_blocks, block_size=16, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise AllocError(ERR_INVALID, "bad pool size")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise AllocError(ERR_INVALID, "free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(order)          # front = next block handed out
        self.ref = [0] * num_blocks
        self.seqs = {}                   # id -> {"table": [...], "len": int}
        self.next_id = 0

    # -- sequences -------------------------------------------------------
    def seq_create(self):
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"table": [], "len": 0}
        return sid

    def _get(self, sid):
        if sid not in self.seqs:
            raise AllocError(ERR_INVALID, f"unknown sequence {sid}")
        return self.seqs[sid]

    def seq_fork(self, parent, prefix_tokens):
        p = self._get(parent)
        if prefix_tokens < 0 or prefix_tokens > p["len"]:
            raise AllocError(ERR_INVALID, "prefix longer than parent")
        nblk = -(-prefix_tokens // self.block_size)
        shared = p["table"][:nblk]
        for blk in shared:
            self.ref[blk] += 1
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"table": list(shared), "len": prefix_tokens}
        return sid

    def seq_free(self, sid):
        s = self._get(sid)
        for blk in s["table"]:
            self.ref[blk] -= 1
            if self.ref[blk] == 0:
                self.free.append(blk)
        del self.seqs[sid]

    # -- slots -------------------------------------------------------------
    def _needs(self, s, tokens):
        """Blocks this sequence will take from the free queue for `tokens` more."""
        bs = self.block_size
        need = 0
        n = s["len"]
        last_shared = bool(s["table"]) and n % bs != 0 and self.ref[s["table"][-1]] > 1
        if tokens > 0 and last_shared:
            need += 1                      # copy-on-write target
        have = len(s["table"]) * bs        # token capacity of the table
        need += max(0, -(-(n + tokens - have) // bs))
        return need

    def _writes_shared(self, s, tokens):
        """True when the sequence's next token lands in a block another holds."""
        n = s["len"]
        return (tokens > 0 and bool(s["table"]) and n % self.block_size != 0
                and self.ref[s["table"][-1]] > 1)

    def append_slots(self, seq_ids, tokens_each, cow_capacity=None):
        """Returns (slot_mapping, cow_pairs); slot order is seq-major.
        ``cow_capacity``: room for copy-on-write pairs (None = unlimited)."""
        if tokens_each < 0 or len(set(seq_ids)) != len(seq_ids):
            raise AllocError(ERR_INVALID, "bad token count or repeated sequence")
        seqs = [self._get(sid) for sid in seq_ids]
        n_shared = sum(1 for s in seqs if self._writes_shared(s, tokens_each))
        if cow_capacity is not None and n_shared > cow_capacity:
            raise AllocError(ERR_SHARED_WRITE, "write into a shared block without room for its copy")
        if sum(self._needs(s, tokens_each) for s in seqs) > len(self.free):
            raise AllocError(ERR_OOM, "free queue exhausted")
        bs = self.block_size
        slots, cow = [], []
        for s in seqs:
            for _ in range(tokens_each):
                pos = s["len"]
                j, off = divmod(pos, bs)
                if j == len(s["table"]):             # current block is full
                    s["table"].append(self.free.pop(0))
                    self.ref[s["table"][-1]] = 1
                elif self.ref[s["table"][j]] > 1:    # writing into a shared block
                    src = s["table"][j]
                    dst = self.free.pop(0)
                    self.ref[dst] = 1
                    self.ref[src] -= 1
                    s["table"][j] = dst
                    cow.append((src, dst))
                slots.append(s["table"][j] * bs + off)
                s["len"] = pos + 1
        return slots, cow

    # -- views -----------------------------------------------------------------
    def block_table(self, seq_ids, max_blocks):
        rows, lens = [], []
        for sid in seq_ids:
            s = self._get(sid)
            if len(s["table"]) > max_blocks:
                raise AllocError(ERR_INVALID, "row longer than max_blocks")
            rows.append(s["table"] + [-1] * (max_blocks - len(s["table"])))
            lens.append(s["len"])
        return rows, lens

    def stats(self):
        used = sum(1 for r in self.ref if r > 0)
        return {
            "num_blocks": self.num_blocks,
            "free": len(self.free),
            "used": used,
            "shared": sum(1 for r in self.ref if r > 1),
            "refs": sum(self.ref),
            "seqs": len(self.seqs),
            "frag_tokens": sum(len(s["table"]) * self.block_size - s["len"] for s in self.seqs.values()),
        }
