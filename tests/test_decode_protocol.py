"""The copy ring of the split-K decode partial kernel (decode_mma), checked
on the CPU under random schedules.

The model has the kernel's copy protocol and none of its arithmetic: a
ring of STAGES shared-memory stages, one mbarrier per stage counting a
tile's bytes in; thread 0 issues the first wave (for one sequence its size
comes from the split before the context length is known, so it may hold
tiles past the real end); each of the 4 consumer warps waits for tile
it + 1 with parity ((it + 1) / STAGES) & 1 while it still reads tile it
(the software pipeline: q.k of the next tile beside p.v of this one), then
releases tile it; the warp that releases a stage last resets its counter
and issues the refill (tile it + STAGES, if the split has it); at the end
thread 0 waits, bounded, for the last STAGES tiles it may have issued.
The wait rule is the hardware's: a parity wait returns once the current
phase has the other parity.  Copies land in random order.

Checked in every schedule: a warp's wait returns only when its own tile has
landed (never an older phase of the stage); no copy lands in a stage a warp
still reads; no copy is still in flight when the CTA exits; nothing
deadlocks.  Planted mistakes must be caught: the first releaser refilling,
a parity off by one, and a drain that misses the first wave's extra tiles.
"""
import random

import pytest

WARPS = 4


class Barrier:
    def __init__(self):
        self.phase = 0          # completed phases (one arrival each: the copy's bytes)

    def ready(self, parity):
        return (self.phase & 1) != parity


class Ring:
    def __init__(self, stages, n_tiles, n_pre, rng, plant=None):
        self.S, self.n, self.rng, self.plant = stages, n_tiles, rng, plant
        self.n_first = min(n_pre, stages)          # first wave, sized before the length is known
        self.full = [Barrier() for _ in range(stages)]
        self.rel = [0] * stages
        self.in_flight = []                         # tiles whose copy has not landed
        self.landed = {}                            # stage -> tile whose bytes it holds
        self.reading = [set() for _ in range(WARPS)]   # tiles each warp still reads

    def issue(self, t):
        self.in_flight.append(t)

    def land(self, i):
        t = self.in_flight.pop(i)
        s = t % self.S
        for w in range(WARPS):
            for r in self.reading[w]:
                assert r % self.S != s, f"tile {t} landed in stage {s} while warp {w} reads tile {r}"
        self.landed[s] = t
        self.full[s].phase += 1

    def producer_first_wave(self):
        for t in range(self.n_first):
            self.issue(t)
        yield None

    def consumer(self, w):
        S = self.S
        if self.n == 0:
            return
        yield self.full[0], 0
        assert self.landed.get(0) == 0, f"warp {w} read tile 0 before it landed"
        self.reading[w].add(0)
        it = 0
        while it + 1 < self.n:
            sn = (it + 1) % S
            par = ((it + 1) // S) & 1
            if self.plant == "parity":
                par ^= 1 if it + 1 >= S else 0
            yield self.full[sn], par
            assert self.landed.get(sn) == it + 1, f"warp {w} read stage {sn} as tile {it + 1}, " \
                                                  f"it holds tile {self.landed.get(sn)}"
            self.reading[w].add(it + 1)
            yield None                               # q.k of it + 1 beside p.v of it
            self.release(w, it)
            it += 1
        yield None
        self.release(w, it)                          # the last tile

    def release(self, w, it):
        self.reading[w].discard(it)
        s = it % self.S
        prev = self.rel[s]
        self.rel[s] += 1
        if prev == WARPS - 1:
            self.rel[s] = 0                          # the last releaser resets the count
        refill = (prev == 0) if self.plant == "first_releaser" else (prev == WARPS - 1)
        if refill and it + self.S < self.n:
            self.issue(it + self.S)

    def producer_drain(self):
        n_all = self.n if self.plant == "short_drain" else max(self.n, self.n_first)
        for t in range(max(0, n_all - self.S), n_all):
            yield self.full[t % self.S], (t // self.S) & 1

    def run(self):
        actors = [self.producer_first_wave()] + [self.consumer(w) for w in range(WARPS)]
        # the CTA barrier after the first wave: consumers start after it
        list(actors[0])
        waiting = {a: self.step(a) for a in actors[1:]}
        live = [a for a in actors[1:] if waiting[a] is not False]
        drain = None
        while True:
            if not live and drain is None:
                drain = self.producer_drain()
                waiting[drain] = self.step(drain)
                live = [drain] if waiting[drain] is not False else []
            if not live:
                break
            runnable = [a for a in live if waiting[a] is None or waiting[a][0].ready(waiting[a][1])]
            assert runnable or self.in_flight, "deadlock: every warp waits and no copy is in flight"
            # copies are slow next to the warps: a warp step is taken when one
            # can run, most of the time, so copies stay in flight for a while
            if runnable and (not self.in_flight or self.rng.random() < 0.75):
                kind, x = "a", self.rng.choice(runnable)
            else:
                kind, x = "c", self.rng.randrange(len(self.in_flight))
            if kind == "a":
                waiting[x] = self.step(x)
                if waiting[x] is False:
                    live.remove(x)
            else:
                self.land(x)
        assert not self.in_flight, f"copies of tiles {self.in_flight} in flight when the CTA exits"

    @staticmethod
    def step(actor):
        try:
            return next(actor)
        except StopIteration:
            return False


@pytest.mark.parametrize("stages,n_tiles,n_pre", [(2, 1, 1), (3, 7, 7), (3, 2, 7), (4, 1, 7),
                                                  (4, 30, 30), (2, 9, 9), (3, 0, 7)])
def test_copy_ring_holds_under_random_schedules(stages, n_tiles, n_pre):
    for seed in range(200):
        Ring(stages, n_tiles, n_pre, random.Random(seed * 7919 + n_tiles)).run()


@pytest.mark.parametrize("plant,stages,n_tiles,n_pre,message", [
    ("first_releaser", 3, 12, 12, "while warp"),
    ("parity", 3, 12, 12, "read stage"),
    ("short_drain", 4, 2, 7, "in flight when the CTA exits"),
])
def test_planted_ring_mistakes_are_caught(plant, stages, n_tiles, n_pre, message):
    caught = 0
    for seed in range(300):
        try:
            Ring(stages, n_tiles, n_pre, random.Random(seed), plant=plant).run()
        except AssertionError as e:
            assert message in str(e) or "deadlock" in str(e), str(e)
            caught += 1
    assert caught > 0
