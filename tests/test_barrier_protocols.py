"""Models of the prefill kernel's mbarrier protocols, run under random interleavings: the
cluster schedule's hand-offs between CTAs (first part) and the two-slot ring inside one CTA
(second part).

The cluster schedule of the prefill kernel splits a unit over four CTAs: the home CTA runs
the chain over three slots, helper h prepares chunks c = h (mod 3) in its own two slots, and
the home CTA's pulling warps copy each finished chunk across.  Their hand-offs are mbarrier
phases: FULLOP and HFREE per home slot, READY per (helper, helper slot), COPIED and the box
loads (FULLTMA) per helper slot.  An mbarrier wait names only a phase's parity, so a wait
passes as soon as the barrier's completion count has the other parity: one completion too
few or one too many both look alike.  The kernel relies on every wait being for the
completion right after the last one its thread saw, and on no barrier completing twice
before its waiter looks.

This model replays the same waits and arrivals (the same slot indices and parities) with
that hardware rule, in random orders, and checks that nothing deadlocks, that every wait
passes on exactly the completion it stands for, and that no slot is overwritten before it
is read.  A variant with one READY barrier per helper instead of one per helper slot, a
plausible simplification, must fail: its parity waits block on a completion that needs the
waiter's own progress, or pass on the wrong one.

The ring model covers one CTA's slots (box loads and beta on FULLTMA, v on FULLV, the prep
group's AREADY and FULLP, the inverse warp's LFREE and FULLD) and the slot regions each step
writes and reads; without LFREE, the prep group rewrites L before the inverse has read it.
"""
import random

import pytest

NH, NSH = 3, 3   # helpers, home slots


class Barrier:
    def __init__(self, name):
        self.name, self.done = name, 0

    def arrive(self):
        self.done += 1


class Aliased(AssertionError):
    pass


class Deadlock(AssertionError):
    pass


BLOCKED, WORK = 0, 1


def make_actors(n_chunks, ready_per_slot=True):
    bars = {}

    def bar(*key):
        if key not in bars:
            bars[key] = Barrier(key)
        return bars[key]

    home = [None] * NSH                          # (state, chunk) of each home slot
    helper = [[None, None] for _ in range(NH)]   # (state, chunk) of each helper slot
    consumed = []

    def wait(b, k):
        """Wait for completion k (0-based) of barrier b: parity k & 1, the hardware rule."""
        while (b.done & 1) == (k & 1):   # the phase with parity k & 1 has not completed
            yield BLOCKED
        if b.done != k + 1:
            raise Aliased(f"{b.name}: waited for completion {k}, passed at {b.done} completions")

    def ready(h, b):
        return bar("READY", h, b) if ready_per_slot else bar("READY", h)

    def ready_index(j):
        return j >> 1 if ready_per_slot else j

    def chain():
        yield from wait(bar("FULLOP", 0), 0)                       # a of chunk 0
        for c in range(n_chunks):
            s = c % NSH
            assert home[s] == ("pulled", c), (c, home[s])           # GEMM1..GEMM3 read the slot
            home[s] = ("consumed", c)
            consumed.append(c)
            bar("HFREE", s).arrive()
            if c + 1 < n_chunks:
                yield from wait(bar("FULLOP", (c + 1) % NSH), (c + 1) // NSH)
            yield WORK

    def puller():
        for c in range(n_chunks):
            h, j, hs, r = c % NH, c // NH, c % NSH, c // NSH
            b = j & 1
            if r > 0:
                yield from wait(bar("HFREE", hs), r - 1)
            yield from wait(ready(h, b), ready_index(j))
            assert helper[h][b] == ("prepared", c), (c, helper[h][b])
            assert home[hs] is None or home[hs] == ("consumed", c - NSH), (c, home[hs])
            home[hs] = ("pulled", c)
            helper[h][b] = ("copied", c)
            bar("FULLOP", hs).arrive()
            bar("COPIED", h, b).arrive()
            yield WORK

    def loader(h):
        j = 0
        while h + NH * j < n_chunks:
            c, b = h + NH * j, j & 1
            if j >= 2:
                yield from wait(bar("COPIED", h, b), (j - 2) >> 1)
            assert helper[h][b] is None or helper[h][b] == ("copied", c - 2 * NH), (c, helper[h][b])
            helper[h][b] = ("loading", c)
            yield WORK                                              # the boxes are in flight
            helper[h][b] = ("loaded", c)
            bar("FULLTMA", h, b).arrive()
            j += 1

    def prep(h):   # prep group, inverse warp and the READY notifier of helper h
        j = 0
        while h + NH * j < n_chunks:
            c, b = h + NH * j, j & 1
            yield from wait(bar("FULLTMA", h, b), j >> 1)
            assert helper[h][b] == ("loaded", c), (c, helper[h][b])
            yield WORK
            helper[h][b] = ("prepared", c)
            ready(h, b).arrive()
            j += 1

    actors = [chain(), puller()] + [loader(h) for h in range(NH)] + [prep(h) for h in range(NH)]
    return actors, consumed


def run(n_chunks, seed, ready_per_slot=True):
    rng = random.Random(seed)
    actors, consumed = make_actors(n_chunks, ready_per_slot)
    live = list(actors)
    idle = 0   # consecutive steps in which the chosen actor was polling a blocked wait
    while live:
        a = rng.choice(live)
        try:
            idle = idle + 1 if next(a) == BLOCKED else 0
        except StopIteration:
            live.remove(a)
            idle = 0
        if idle > 200 * len(live):
            raise Deadlock(f"{len(live)} actors all waiting")
    assert consumed == list(range(n_chunks))


@pytest.mark.parametrize("n_chunks", [1, 2, 3, 4, 5, 6, 7, 12, 13, 31, 64])
def test_protocol_holds_under_random_interleavings(n_chunks):
    for seed in range(25):
        run(n_chunks, seed)


def test_one_ready_barrier_per_helper_would_alias():
    """With READY shared by a helper's two slots, a fast helper completes it twice before the
    home CTA looks: the parity wait then stands for the wrong phase."""
    broken = 0
    for seed in range(20):
        try:
            run(40, seed, ready_per_slot=False)
        except (Aliased, Deadlock):
            broken += 1
    assert broken > 0


# ---------------------------------------------------------------------------------------
# The two-slot ring of one CTA (the two-CTA and one-CTA-per-SM schedules): the chain, the
# prep group and the inverse warp, with the slot regions each step writes and reads.
# ---------------------------------------------------------------------------------------

def make_ring_actors(n_chunks, lfree=True):
    bars = {}

    def bar(*key):
        if key not in bars:
            bars[key] = Barrier(key)
        return bars[key]

    def wait(b, k):   # completion k (0-based); the kernel passes its parity k & 1
        while (b.done & 1) == (k & 1):
            yield BLOCKED
        if b.done != k + 1:
            raise Aliased(f"{b.name}: waited for completion {k}, passed at {b.done} completions")

    # what each region of each slot holds: (chunk, stage); L is the prep scratch the inverse reads
    slot = [dict() for _ in range(2)]
    L = {"chunk": None, "read": True}
    tmafill = {0: 0, 1: 0}          # FULLTMA arrivals this phase: the box load and beta
    consumed = []

    def fulltma_arrive(s):
        tmafill[s] += 1
        if tmafill[s] == 2:         # 33 arrivals and the transaction bytes, as two events
            tmafill[s] = 0
            bar("FULLTMA", s).arrive()

    def load_qkg(c, s):            # the TMA engine, asynchronous
        assert slot[s].get("mqk", (c - 2, "read"))[1] == "read" or c < 2, (c, slot[s])
        slot[s]["qkg"] = (c, "loading")
        yield WORK
        slot[s]["qkg"] = (c, "raw")
        fulltma_arrive(s)

    def put_beta(c, s):
        assert slot[s].get("beta", (c - 2, "read"))[1] == "read" or c < 2, (c, slot[s])
        slot[s]["beta"] = (c, "put")
        fulltma_arrive(s)

    def load_v(c, s):
        slot[s]["v"] = (c, "loading")
        yield WORK
        slot[s]["v"] = (c, "landed")
        bar("FULLV", s).arrive()

    engines = []

    def chain():
        first = min(n_chunks, 2)
        for c in range(first):
            engines.append(load_qkg(c, c))
            put_beta(c, c)
            engines.append(load_v(c, c))
        if n_chunks == 0:
            return
        yield from wait(bar("AREADY", 0), 0)
        assert slot[0]["a"] == (0, "written")
        for c in range(n_chunks):
            s, k = c & 1, c >> 1                         # slot, and the completion of its barriers
            refill = c + 2 < n_chunks
            yield from wait(bar("FULLP", s), k)
            yield from wait(bar("FULLV", s), k)
            assert slot[s]["ops"] == (c, "written") and slot[s]["v"] == (c, "landed"), (c, slot[s])
            yield WORK                                   # GEMM1 reads [Q_d | K_d] and v
            yield from wait(bar("FULLD", s), k)
            assert slot[s]["inv"] == (c, "written"), (c, slot[s])
            slot[s]["beta"] = (c, "read")                # the inverse has read beta
            if refill:
                put_beta(c + 2, s)
            yield WORK                                   # GEMM2 reads -B2, GEMM3 K_r and Mqk
            assert slot[s]["mqk"] == (c, "written"), (c, slot[s])
            slot[s]["mqk"] = (c, "read")
            slot[s]["ops"] = (c, "read")
            consumed.append(c)
            if refill:
                engines.append(load_qkg(c + 2, s))
            slot[s]["v"] = (c, "staging")                # the output tile, then its store
            if c + 1 < n_chunks:
                yield from wait(bar("AREADY", s ^ 1), (c + 1) >> 1)
                assert slot[s ^ 1]["a"] == (c + 1, "written"), (c, slot[s ^ 1])
                yield WORK                               # copy and decay with a of chunk c + 1
                if refill:
                    engines.append(load_v(c + 2, s))

    def prep():
        for c in range(n_chunks):
            s, k = c & 1, c >> 1
            yield from wait(bar("FULLTMA", s), k)
            assert slot[s]["qkg"] == (c, "raw") and slot[s]["beta"] == (c, "put"), (c, slot[s])
            yield WORK
            slot[s]["ops"] = (c, "written")              # Q_d, K_d, K_r over the raw boxes
            slot[s]["a"] = (c, "written")
            bar("AREADY", s).arrive()
            if c > 0 and lfree:
                yield from wait(bar("LFREE"), c - 1)
            assert L["read"], (c, L)                     # L of chunk c - 1 has been read
            L.update(chunk=c, read=False)
            slot[s]["mqk"] = (c, "written")
            bar("FULLP", s).arrive()

    def inverse():
        for c in range(n_chunks):
            s, k = c & 1, c >> 1
            yield from wait(bar("FULLP", s), k)
            assert L["chunk"] == c and slot[s]["beta"] == (c, "put"), (c, L, slot[s])
            yield WORK
            L["read"] = True
            bar("LFREE").arrive()
            slot[s]["inv"] = (c, "written")
            bar("FULLD", s).arrive()

    return [chain(), prep(), inverse()], engines, consumed


def run_ring(n_chunks, seed, lfree=True):
    rng = random.Random(seed)
    actors, engines, consumed = make_ring_actors(n_chunks, lfree)
    live = list(actors)
    idle = 0
    while live or engines:
        live += engines
        engines.clear()
        a = rng.choice(live)
        try:
            idle = idle + 1 if next(a) == BLOCKED else 0
        except StopIteration:
            live.remove(a)
            idle = 0
        if idle > 200 * max(1, len(live)):
            raise Deadlock(f"{len(live)} actors all waiting")
    assert consumed == list(range(n_chunks))


@pytest.mark.parametrize("n_chunks", [0, 1, 2, 3, 4, 5, 8, 17, 64])
def test_ring_protocol_holds_under_random_interleavings(n_chunks):
    for seed in range(25):
        run_ring(n_chunks, seed)


def test_ring_without_lfree_overwrites_l():
    """Without the inverse warp's LFREE, the prep group rewrites L before it has been read."""
    broken = 0
    for seed in range(20):
        try:
            run_ring(12, seed, lfree=False)
        except AssertionError:
            broken += 1
    assert broken > 0
