"""A model of the cluster schedule's barrier protocol, run under random interleavings.

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
