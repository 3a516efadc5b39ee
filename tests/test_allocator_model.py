"""The allocator model (oracle side) against the pages' facts and invariants."""
import json
import os

import pytest

from oracle.allocator import AllocatorModel, AllocError, ERR_OOM, ERR_INVALID

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def check_invariants(m):
    """Free queue + referenced blocks = pool; refs = table references."""
    free = set(m.free)
    assert len(free) == len(m.free), "block twice in the free queue"
    for blk in range(m.num_blocks):
        assert (m.ref[blk] == 0) == (blk in free), blk
    refs = {}
    for s in m.seqs.values():
        assert len(s["table"]) == -(-s["len"] // m.block_size)
        for blk in s["table"]:
            refs[blk] = refs.get(blk, 0) + 1
    for blk in range(m.num_blocks):
        assert m.ref[blk] == refs.get(blk, 0), blk
    st = m.stats()
    assert st["free"] + st["used"] == m.num_blocks
    assert st["refs"] == sum(len(s["table"]) for s in m.seqs.values())


def test_golden_allocation_facts():
    g = json.load(open(os.path.join(GOLD, "allocation.json")))
    c17, cw = g["cases"]
    m = AllocatorModel(8, c17["block_size"])
    s = m.seq_create()
    slots, cow = m.append_slots([s], c17["new_tokens"])
    assert len(m.seqs[s]["table"]) == c17["expect_blocks"], c17["cite"]
    assert cow == [] and len(slots) == 17
    for L in range(1, 200):
        m = AllocatorModel(64, cw["block_size"])
        s = m.seq_create()
        m.append_slots([s], L)
        assert m.stats()["frag_tokens"] <= cw["max_waste_tokens"], cw["cite"]
        check_invariants(m)


def test_slots_follow_table_and_free_order():
    order = [5, 2, 7, 0, 1, 3, 4, 6]
    m = AllocatorModel(8, 16, order)
    a, b = m.seq_create(), m.seq_create()
    slots, _ = m.append_slots([a, b], 17)
    # append is sequence-major: a takes 5 and 2, then b takes 7 and 0
    assert m.seqs[a]["table"] == [5, 2] and m.seqs[b]["table"] == [7, 0]
    assert slots[:17] == [5 * 16 + i for i in range(16)] + [2 * 16]
    assert slots[17:] == [7 * 16 + i for i in range(16)] + [0]
    check_invariants(m)


def test_fork_shares_and_copy_on_write():
    m = AllocatorModel(16, 16)
    p = m.seq_create()
    m.append_slots([p], 40)          # 3 blocks, last one holds 8 tokens
    c = m.seq_fork(p, 40)            # shares all three
    assert m.seqs[c]["table"] == m.seqs[p]["table"]
    assert m.stats()["shared"] == 3
    check_invariants(m)
    shared_tail = m.seqs[p]["table"][2]
    slots, cow = m.append_slots([c], 1)   # writes into the shared partial block
    assert len(cow) == 1 and cow[0][0] == shared_tail
    assert m.seqs[c]["table"][2] == cow[0][1] != shared_tail
    assert slots == [cow[0][1] * 16 + 8]
    assert m.ref[shared_tail] == 1
    check_invariants(m)
    # the parent's next write is no longer shared: no copy
    _, cow2 = m.append_slots([p], 1)
    assert cow2 == []
    check_invariants(m)


def test_free_returns_block_only_at_last_reference():
    m = AllocatorModel(8, 16)
    p = m.seq_create()
    m.append_slots([p], 32)
    c = m.seq_fork(p, 32)
    m.seq_free(p)
    assert len(m.free) == 6           # both blocks still held by c
    m.seq_free(c)
    assert len(m.free) == 8
    check_invariants(m)


def test_oom_is_atomic_and_errors_are_codes():
    m = AllocatorModel(3, 16)
    a, b = m.seq_create(), m.seq_create()
    m.append_slots([a], 16)
    before = (list(m.free), {k: dict(v, table=list(v["table"])) for k, v in m.seqs.items()})
    with pytest.raises(AllocError) as e:
        m.append_slots([a, b], 20)    # needs 2 + 2 blocks, 2 free
    assert e.value.code == ERR_OOM
    assert (list(m.free), m.seqs) == before
    with pytest.raises(AllocError) as e:
        m.seq_free(99)
    assert e.value.code == ERR_INVALID
    m.seq_free(a)
    with pytest.raises(AllocError) as e:
        m.seq_free(a)                 # double free
    assert e.value.code == ERR_INVALID


def test_random_operation_sequences():
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    ops = st.lists(st.tuples(st.sampled_from(["new", "app", "fork", "free"]),
                             st.integers(0, 7), st.integers(0, 40)), max_size=60)

    @hyp.settings(max_examples=150, deadline=None)
    @hyp.given(ops)
    def run(seq):
        m = AllocatorModel(24, 16)
        live = []
        for op, i, n in seq:
            try:
                if op == "new" or not live:
                    live.append(m.seq_create())
                elif op == "app":
                    sid = live[i % len(live)]
                    slots, cow = m.append_slots([sid], n)
                    for s in slots:        # every written slot is in an unshared block
                        assert m.ref[s // 16] == 1
                elif op == "fork":
                    sid = live[i % len(live)]
                    live.append(m.seq_fork(sid, min(n, m.seqs[sid]["len"])))
                else:
                    m.seq_free(live.pop(i % len(live)))
            except AllocError as e:
                assert e.code == ERR_OOM
            check_invariants(m)

    run()
