"""Model check of the attention kernel's shared-memory ring protocol (CPU).

The kernel's producer warp streams blocks into S stages; consumer warps wait
on a per-stage "full" mbarrier with a parity bit and release the stage on an
"empty" mbarrier.  A parity wait only asks "has the phase of this parity
completed", so if two consecutive uses of one stage could be consumed by
different warps without an ordering between them, a warp waiting for round
r+1 could pass on round r-1's completed phase and read the stage before its
copy lands.

The kernel gives block g of the CTA's whole block stream to consumer
g % NC and requires S % NC == 0, so every stage has one consumer and no
barrier is needed between work items: at the end of an item each consumer
hands its state to a combiner warp and goes on with the next item.  (Which
warp sums which blocks of an item then depends on where the item starts in
the stream, but the blocks of one residue class j % NC are always summed
together and in order, and the combiner folds the classes in class order,
so the outputs stay bit-reproducible.)  The earlier rule, block j of an item
to consumer j % NC, is safe only with a barrier between items; without one
it reads stale stages, which the model shows too.

This test runs a randomised discrete-event model of the protocol with exact
mbarrier parity semantics (try_wait.parity(P) is true iff the barrier's
current phase parity differs from P) and checks that no consumer ever reads
a stage holding another block: safe for every S that is a multiple of NC
under the kernel's rule without a merge barrier, unsafe (stale reads or
deadlock) for S = 6 or 10 with NC = 4, and unsafe for the item-relative rule
without the barrier.

The FP8 kernel has two copy threads: thread p refills the stages of the
blocks g with g % 2 == p, in order, each independently of the other (one
may run ahead).  The model runs P independent producers the same way and
checks that the protocol stays safe with them.

The consumers hand their per-item states to the combiner warp through two
merge slots guarded by a full and an empty mbarrier each; a second model
runs that hand-off with random timing and checks that the combiner only
ever reads the states of the item it is folding (and that the empty wait
needs its parity flipped on first use)."""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = count
        self.phase = 0            # completed phases
        self.tx = 0

    def try_wait(self, parity):
        return (self.phase & 1) != parity

    def arrive(self):
        self.pending -= 1
        self._maybe_complete()

    def expect_tx(self, n):
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count


def simulate(S, NC, rule, items, seed, producers=1, merge_barrier=True):
    """Returns the number of stale reads (0 = protocol safe), or -1 if the
    protocol deadlocks (nobody can move for a long time).  merge_barrier:
    consumers wait for each other at the end of every item."""
    rng = random.Random(seed)
    full = [Barrier(1) for _ in range(S)]
    empty = [Barrier(1) for _ in range(S)]
    stage_tag = [None] * S
    in_flight = []                     # (land_time, stage, block)
    g0s, g = [], 0
    for n in items:
        g0s.append(g)
        g += n
    total = g
    # consumer state: (item index, next position in its block list)
    def blocks_of(w, it):
        g0, n = g0s[it], items[it]
        if rule == "global":
            j0 = (w - g0 % NC) % NC
        else:                           # item-relative (the old rule)
            j0 = w
        return [g0 + j for j in range(j0, n, NC)]

    cons = [{"it": 0, "list": blocks_of(w, 0), "pos": 0, "at_merge": False} for w in range(NC)]
    merge_arrived = [0] * len(items)
    assert S % producers == 0           # each stage has one producer
    next_issue = list(range(producers))  # producer p issues blocks p, p + P, ...
    stale = 0
    t = 0
    done = [False] * NC
    while not all(done):
        t += 1
        if t > 200 * total + 20000:
            return -1
        # copies land after a random delay
        for rec in [r for r in in_flight if r[0] <= t]:
            in_flight.remove(rec)
            _, s, blk = rec
            stage_tag[s] = blk
            full[s].complete_tx(1)
        actor = rng.randrange(NC + producers)
        if actor >= NC:                 # producer p issues its next block
            p = actor - NC
            nxt = next_issue[p]
            if nxt < total:
                s, r = nxt % S, nxt // S
                if empty[s].try_wait((r & 1) ^ 1):
                    full[s].expect_tx(1)
                    stage_tag[s] = ("landing", nxt)
                    in_flight.append((t + rng.randint(1, 40), s, nxt))
                    next_issue[p] += producers
            continue
        c = cons[actor]
        if done[actor]:
            continue
        if c["at_merge"]:               # merge barrier: all consumers of the item
            if merge_arrived[c["it"]] == NC:
                c["it"] += 1
                c["at_merge"] = False
                if c["it"] == len(items):
                    done[actor] = True
                else:
                    c["list"], c["pos"] = blocks_of(actor, c["it"]), 0
            continue
        if c["pos"] == len(c["list"]):
            merge_arrived[c["it"]] += 1
            if merge_barrier:
                c["at_merge"] = True
            else:                       # hand the state over and go on
                c["it"] += 1
                if c["it"] == len(items):
                    done[actor] = True
                else:
                    c["list"], c["pos"] = blocks_of(actor, c["it"]), 0
            continue
        blk = c["list"][c["pos"]]
        s, r = blk % S, blk // S
        if full[s].try_wait(r & 1):
            if stage_tag[s] != blk:
                stale += 1
            empty[s].arrive()
            c["pos"] += 1
    return stale


def random_items(rng, n):
    return [rng.randint(1, 40) for _ in range(n)]


@pytest.mark.parametrize("rule", ["item", "global"])
@pytest.mark.parametrize("S,NC", [(4, 4), (8, 4), (12, 4), (8, 2), (8, 8)])
def test_stage_multiple_of_consumers_never_reads_a_stale_stage(S, NC, rule):
    rng = random.Random(S * 100 + NC)
    for seed in range(40):
        assert simulate(S, NC, rule, random_items(rng, 12), seed) == 0


@pytest.mark.parametrize("producers", [1, 2])
@pytest.mark.parametrize("S", [6, 10])
def test_stages_not_a_multiple_of_consumers_are_unsafe(S, producers):
    rng = random.Random(7)
    results = [simulate(S, 4, "item", random_items(rng, 12), seed, producers)
               for seed in range(10)]
    assert any(r != 0 for r in results)     # stale reads or deadlock


@pytest.mark.parametrize("rule", ["item", "global"])
@pytest.mark.parametrize("S,NC", [(16, 4), (8, 4), (4, 4), (8, 2), (8, 8)])
def test_two_producers_on_alternate_stages_never_read_a_stale_stage(S, NC, rule):
    rng = random.Random(S * 1000 + NC)
    for seed in range(40):
        assert simulate(S, NC, rule, random_items(rng, 12), seed, producers=2) == 0


@pytest.mark.parametrize("producers", [1, 2])
@pytest.mark.parametrize("S,NC", [(4, 4), (8, 4), (16, 4), (8, 2), (8, 8)])
def test_stage_owned_consumers_need_no_barrier_between_items(S, NC, producers):
    """The kernel's protocol: block g to consumer g % NC, no merge barrier."""
    rng = random.Random(S * 10 + NC + producers)
    for seed in range(40):
        assert simulate(S, NC, "global", random_items(rng, 12), seed, producers,
                        merge_barrier=False) == 0


def test_item_relative_consumers_without_barrier_are_unsafe():
    """Block j of an item to consumer j % NC is safe only with the barrier."""
    rng = random.Random(11)
    results = [simulate(8, 4, "item", random_items(rng, 12), seed, merge_barrier=False)
               for seed in range(40)]
    assert any(r != 0 for r in results)


def simulate_merge_slots(NC, n_items, seed, slots=2, empty_parity_flip=True):
    """The hand-off between the consumer warps and the combiner warp: at the
    end of item `it` each consumer waits merge_empty[it % slots] (parity
    ((it // slots) & 1) ^ 1), stores its state into merge slot it % slots
    and arrives merge_full[it % slots]; the combiner, item by item, waits
    merge_full[it % slots] (parity (it // slots) & 1), reads the NC states
    and arrives merge_empty[it % slots].  Returns the number of reads that
    saw a state of another item (0 = safe), or -1 on deadlock."""
    rng = random.Random(seed)
    full = [Barrier(NC) for _ in range(slots)]
    empty = [Barrier(1) for _ in range(slots)]
    slot_state = [[None] * NC for _ in range(slots)]
    cons_it = [0] * NC            # next item each consumer finishes
    comb_it = 0
    bad = 0
    steps = 0
    while comb_it < n_items:
        steps += 1
        if steps > 200 * n_items * (NC + 1) + 10000:
            return -1
        actor = rng.randrange(NC + 1)
        if actor < NC:
            it = cons_it[actor]
            if it >= n_items:
                continue
            s, r = it % slots, it // slots
            parity = ((r & 1) ^ 1) if empty_parity_flip else (r & 1)
            if empty[s].try_wait(parity):
                slot_state[s][actor] = it
                full[s].arrive()
                cons_it[actor] += 1
        else:
            s, r = comb_it % slots, comb_it // slots
            if full[s].try_wait(r & 1):
                bad += sum(1 for w in range(NC) if slot_state[s][w] != comb_it)
                empty[s].arrive()
                comb_it += 1
    return bad


@pytest.mark.parametrize("NC", [1, 2, 4])
def test_combiner_hand_off_never_reads_another_items_state(NC):
    for seed in range(60):
        assert simulate_merge_slots(NC, 25, seed) == 0


def test_combiner_hand_off_without_the_empty_parity_flip_is_unsafe():
    """Waiting merge_empty on the full barrier's parity (no flip) lets the
    first uses of a slot block forever or overwrite: the flip is needed."""
    results = [simulate_merge_slots(4, 25, seed, empty_parity_flip=False) for seed in range(20)]
    assert any(r != 0 for r in results)
