"""The C++ allocator in libpa against the oracle's allocator model: the same
slots, tables, copy-on-write pairs, statistics and error codes."""
import numpy as np
import pytest

from oracle.allocator import AllocatorModel, AllocError


@pytest.fixture(scope="module")
def binding():
    from paged_kv_cache_blocks_gb300 import build, binding
    build.build()
    binding.lib()
    return binding


def same_state(m, a, live, max_blocks=64):
    rows, lens = a.block_table(live, max_blocks)
    mrows, mlens = m.block_table(live, max_blocks)
    assert rows == mrows and lens == mlens
    st = a.stats()
    ms = m.stats()
    for k in ("free", "used", "shared", "refs", "seqs", "frag_tokens"):
        assert st[k] == ms[k], k


def test_golden_facts(binding):
    a = binding.Allocator(8)
    s = a.seq_create()
    slots, cow = a.append_slots([s], 17)
    rows, lens = a.block_table([s], 4)
    assert rows[0][:2] != [-1, -1] and rows[0][2] == -1 and lens == [17]   # 17 tokens -> 2 blocks
    assert a.stats()["frag_tokens"] == 15


def test_matches_model_on_scripted_sequence(binding):
    order = list(np.random.default_rng(3).permutation(40))
    a, m = binding.Allocator(40, order), AllocatorModel(40, 16, order)
    s0, t0 = a.seq_create(), m.seq_create()
    assert s0 == t0
    got, want = a.append_slots([s0], 40), m.append_slots([t0], 40)
    assert got[0] == want[0] and got[1] == want[1] == []
    c = a.seq_fork(s0, 40)
    mc = m.seq_fork(t0, 40)
    assert c == mc
    r1 = a.append_slots([c, s0], 3)
    r2 = m.append_slots([mc, t0], 3)
    assert r1[0] == r2[0] and r1[1] == r2[1]
    same_state(m, a, [s0, c])
    a.seq_free(s0)
    m.seq_free(t0)
    same_state(m, a, [c])


def test_errors_are_codes(binding):
    a = binding.Allocator(3)
    s, t = a.seq_create(), a.seq_create()
    a.append_slots([s], 16)
    with pytest.raises(binding.PaError) as e:
        a.append_slots([s, t], 20)
    assert e.value.code == binding.PA_ERR_OOM
    assert a.stats()["free"] == 2                 # nothing changed
    with pytest.raises(binding.PaError) as e:
        a.seq_free(77)
    assert e.value.code == binding.PA_ERR_INVALID
    with pytest.raises(binding.PaError) as e:
        a.append_slots([s, s], 1)
    assert e.value.code == binding.PA_ERR_INVALID
    a.seq_free(s)
    with pytest.raises(binding.PaError) as e:
        a.seq_free(s)
    assert e.value.code == binding.PA_ERR_INVALID
    with pytest.raises(binding.PaError):
        binding.Allocator(4, free_order=[0, 1, 1, 2])
    with pytest.raises(binding.PaError) as e:
        binding.Allocator(4, block_size=32)
    assert e.value.code == binding.PA_ERR_UNSUPPORTED


def test_shared_write_without_room_for_its_copy(binding):
    """A write into a block another sequence still holds, with no room to
    report the copy that must come first, is PA_ERR_SHARED_WRITE and changes
    nothing; with room it moves the writer onto a copy (same as the model)."""
    from oracle.allocator import ERR_SHARED_WRITE
    a, m = binding.Allocator(8), AllocatorModel(8, 16)
    s, t = a.seq_create(), m.seq_create()
    a.append_slots([s], 40)
    m.append_slots([t], 40)
    c, mc = a.seq_fork(s, 40), m.seq_fork(t, 40)     # block 2 of both is partly filled and shared
    before = a.stats()
    with pytest.raises(binding.PaError) as e:
        a.append_slots([c], 1, cow_capacity=0)
    with pytest.raises(AllocError) as me:
        m.append_slots([mc], 1, cow_capacity=0)
    assert e.value.code == binding.PA_ERR_SHARED_WRITE == me.value.code == ERR_SHARED_WRITE
    assert a.stats() == before
    same_state(m, a, [s, c])
    got, want = a.append_slots([c], 1, cow_capacity=1), m.append_slots([mc], 1, cow_capacity=1)
    assert got == want and len(got[1]) == 1
    # a whole shared block is never written: the next token starts a new block
    d, md = a.seq_fork(s, 32), m.seq_fork(t, 32)
    assert a.append_slots([d], 1, cow_capacity=0) == m.append_slots([md], 1, cow_capacity=0)
    same_state(m, a, [s, c, d])


def test_table_and_lengths_updated_in_place(binding):
    a = binding.Allocator(16, list(range(15, -1, -1)))
    ids = [a.seq_create() for _ in range(3)]
    tab = np.full((3, 6), -1, np.int32)
    lens = np.zeros(3, np.int32)
    a.append_slots(ids, 20, block_table=tab, seq_lens=lens)
    rows, ln = a.block_table(ids, 6)
    assert tab.tolist() == rows and lens.tolist() == ln == [20, 20, 20]
    a.append_slots(ids, 13, block_table=tab, seq_lens=lens)
    rows, ln = a.block_table(ids, 6)
    assert tab.tolist() == rows and lens.tolist() == ln == [33, 33, 33]


def test_random_sequences_match_model(binding):
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    ops = st.lists(st.tuples(st.sampled_from(["new", "app", "app2", "app0", "fork", "free"]),
                             st.integers(0, 7), st.integers(0, 40)), max_size=50)

    @hyp.settings(max_examples=120, deadline=None)
    @hyp.given(ops, st.integers(0, 1000))
    def run(seq, seed):
        order = list(np.random.default_rng(seed).permutation(24))
        a, m = binding.Allocator(24, order), AllocatorModel(24, 16, order)
        live = []
        for op, i, n in seq:
            if op == "new" or not live:
                x, y = a.seq_create(), m.seq_create()
                assert x == y
                live.append(x)
                continue
            sid = live[i % len(live)]
            if op in ("app", "app2", "app0"):
                group = [sid] if op != "app2" else sorted(set([sid, live[(i + 1) % len(live)]]))
                cap = 0 if op == "app0" else None   # app0: no room for copy-on-write pairs
                try:
                    want = m.append_slots(group, n, cow_capacity=cap)
                except AllocError as e:
                    with pytest.raises(binding.PaError) as ge:
                        a.append_slots(group, n, cow_capacity=cap)
                    assert ge.value.code == e.code
                else:
                    got = a.append_slots(group, n, cow_capacity=cap)
                    assert got[0] == want[0] and got[1] == want[1]
            elif op == "fork":
                k = min(n, m.seqs[sid]["len"])
                x, y = a.seq_fork(sid, k), m.seq_fork(sid, k)
                assert x == y
                live.append(x)
            else:
                a.seq_free(sid)
                m.seq_free(sid)
                live.remove(sid)
            same_state(m, a, live)

    run()
