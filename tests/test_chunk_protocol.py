"""The mbarrier protocol of the prompt-chunk kernel (chunk_attn_tc), checked
on the CPU under random schedules.

The model has the kernel's roles and their waits, arrivals and commits, in
the kernel's order: the K and V copy producers (stages of KST and VST
tiles), the thread issuing S_j = Q K_j^T, the thread issuing O += P_j V_j,
and the softmax warps (one actor: they wait and arrive together).  It has
none of the arithmetic.  An mbarrier is an arrival count per phase; a wait
on parity P returns once the barrier's current phase has the other parity
(the phase of parity P that precedes it has completed), which is the
hardware rule, so a barrier two phases behind a waiter is misread as done.
Copies and MMA groups complete later, in a random order that keeps each
issuing thread's MMAs in order; an MMA commit arrives once every MMA its
thread issued before it has completed.

Checked in every schedule: each wait that returns has seen the completion
it stands for (the tile's copy, S, P or product, never an older phase);
no S is issued into a buffer whose product is still running; the rescale
of O and the output read see every earlier product complete; and the
protocol runs to the end (no deadlock).  Planted mistakes must be caught:
an earlier epilogue (a parity wait on a barrier committed once per
product), an S issued without waiting for its buffer's product, a rescale
that waits for the wrong tile's product, and a K stage refilled one phase
early.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.arrived = 0
        self.phase = 0          # completed phases

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.phase += 1

    def ready(self, parity):
        # mbarrier.try_wait.parity: true once the current phase's parity
        # differs from `parity`
        return (self.phase & 1) != parity


class Kernel:
    """One CTA of chunk_attn_tc over n key tiles."""

    def __init__(self, n, kst, vst, rng, old_epilogue=False, rises=0.3, plant=None):
        self.n, self.kst, self.vst, self.rng = n, kst, vst, rng
        self.old_epilogue = old_epilogue
        self.plant = plant          # a planted mistake, for the checker's own test
        self.rises = rises
        b = lambda c=1: Barrier(c)
        self.kfull = [b() for _ in range(kst)]
        self.kempty = [b() for _ in range(kst)]
        self.vfull = [b() for _ in range(vst)]
        self.vempty = [b() for _ in range(vst)]
        self.sfull = [b() for _ in range(3)]
        self.pfull = [b() for _ in range(3)]
        self.sfree = [b() for _ in range(3)]
        self.qready = b()
        self.alldone = b()
        self.odone = b()            # the planted old epilogue's barrier
        # what has actually completed
        self.k_loaded, self.v_loaded = set(), set()
        self.s_done, self.pv_done = set(), set()
        self.p_written = set()
        # in-flight asynchronous work: (kind, thread, tile, barriers to arrive on)
        self.copies = []
        self.mmas = {"S": [], "PV": []}      # per issuing thread, in issue order
        self.commits = {"S": [], "PV": []}   # (mmas issued before it, barriers)
        self.issued = {"S": 0, "PV": 0}
        self.completed = {"S": 0, "PV": 0}
        self.actors = [self.producer("K"), self.producer("V"), self.s_thread(),
                       self.pv_thread(), self.softmax()]

    # ---- asynchronous completions ----
    def commit(self, who, bars):
        self.commits[who].append((self.issued[who], bars))

    def events(self):
        ev = [("copy", i) for i in range(len(self.copies))]
        ev += [("mma", w) for w in ("S", "PV") if self.mmas[w]]
        return ev

    def complete(self, ev):
        kind, x = ev
        if kind == "copy":
            what, j, bar = self.copies.pop(x)
            (self.k_loaded if what == "K" else self.v_loaded).add(j)
            bar.arrive()
        else:
            what, j = self.mmas[x].pop(0)
            (self.s_done if what == "S" else self.pv_done).add(j)
            self.completed[x] += 1
        for w in ("S", "PV"):
            while self.commits[w] and self.commits[w][0][0] <= self.completed[w]:
                for bar in self.commits[w].pop(0)[1]:
                    bar.arrive()

    # ---- roles, as generators yielding the barrier waits they block on ----
    def producer(self, what):
        st = self.kst if what == "K" else self.vst
        full = self.kfull if what == "K" else self.vfull
        empty = self.kempty if what == "K" else self.vempty
        for j in range(self.n):
            if j >= st:
                off = 0 if (self.plant == "kempty_parity" and what == "K") else 1
                yield empty[j % st], (j // st - off) & 1
                # the stage's previous tile has been consumed
                if what == "K":
                    assert j - st in self.s_done, f"K stage refilled before S({j - st}) completed"
                else:
                    assert j - st in self.pv_done, f"V stage refilled before PV({j - st}) completed"
            self.copies.append((what, j, full[j % st]))

    def s_thread(self):
        yield self.qready, 0
        for j in range(self.n):
            yield self.kfull[j % self.kst], (j // self.kst) & 1
            assert j in self.k_loaded, f"S({j}) issued before K({j}) landed"
            if j >= 3 and self.plant != "no_sfree_wait":
                yield self.sfree[j % 3], (j // 3 - 1) & 1
            if j >= 3:
                assert j - 3 in self.pv_done, f"S({j}) overwrites the P of PV({j - 3}) still running"
            self.mmas["S"].append(("S", j))
            self.issued["S"] += 1
            self.commit("S", [self.sfull[j % 3], self.kempty[j % self.kst]])

    def pv_thread(self):
        for j in range(self.n):
            yield self.pfull[j % 3], (j // 3) & 1
            assert j in self.p_written, f"PV({j}) issued before P({j}) was written"
            yield self.vfull[j % self.vst], (j // self.vst) & 1
            assert j in self.v_loaded, f"PV({j}) issued before V({j}) landed"
            self.mmas["PV"].append(("PV", j))
            self.issued["PV"] += 1
            self.commit("PV", [self.sfree[j % 3], self.vempty[j % self.vst]] +
                        ([self.odone] if self.old_epilogue else []))
        self.commit("PV", [self.alldone])

    def softmax(self):
        self.qready.arrive()
        for j in range(self.n):
            yield self.sfull[j % 3], (j // 3) & 1
            assert j in self.s_done, f"softmax read S({j}) before it completed"
            if j > 0 and self.rng.random() < self.rises:
                # a raised maximum: O is rescaled after the previous product
                if self.plant == "rescale_wrong_buffer":
                    yield self.sfree[j % 3], (j // 3 - 1) & 1      # the product of tile j - 3
                else:
                    yield self.sfree[(j - 1) % 3], ((j - 1) // 3) & 1
                assert set(range(j)) <= self.pv_done, f"O rescaled at tile {j} with a product running"
            self.p_written.add(j)
            self.pfull[j % 3].arrive()
        if self.old_epilogue:
            yield self.odone, (self.n - 1) & 1
        else:
            yield self.alldone, 0
        assert set(range(self.n)) <= self.pv_done, "O read before the last product completed"

    def run(self):
        waiting = {}
        for a in self.actors:
            waiting[a] = self.step(a)
        live = [a for a in self.actors if waiting[a] is not False]
        while live or self.events():
            runnable = [a for a in live if waiting[a] is None or waiting[a][0].ready(waiting[a][1])]
            ev = self.events()
            choices = [("actor", a) for a in runnable] + [("event", e) for e in ev]
            assert choices, "deadlock: every role waits and nothing is in flight"
            kind, x = self.rng.choice(choices)
            if kind == "actor":
                waiting[x] = self.step(x)
                if waiting[x] is False:
                    live.remove(x)
            else:
                self.complete(x)

    @staticmethod
    def step(actor):
        try:
            return next(actor)
        except StopIteration:
            return False


@pytest.mark.parametrize("n,kst,vst", [(1, 2, 2), (2, 2, 2), (7, 2, 2), (40, 2, 2),
                                       (1, 2, 1), (5, 2, 1), (40, 2, 1)])
def test_protocol_holds_under_random_schedules(n, kst, vst):
    for seed in range(150):
        Kernel(n, kst, vst, random.Random(seed * 1009 + n)).run()


def test_planted_old_epilogue_is_caught():
    # the epilogue once waited with parity (n - 1) & 1 on a barrier
    # committed after every product: two products can still run then, and
    # the parity wait reads the barrier two phases behind as done
    caught = 0
    for seed in range(300):
        try:
            Kernel(12, 2, 1, random.Random(seed), old_epilogue=True).run()
        except AssertionError as e:
            assert "O read before the last product completed" in str(e)
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("plant,message", [
    ("no_sfree_wait", "overwrites the P"),
    ("rescale_wrong_buffer", "O rescaled"),
    ("kempty_parity", "K stage refilled"),
])
def test_planted_protocol_mistakes_are_caught(plant, message):
    caught = 0
    for seed in range(300):
        try:
            Kernel(12, 2, 2, random.Random(seed), rises=0.6, plant=plant).run()
        except AssertionError as e:
            assert message in str(e) or "deadlock" in str(e), str(e)
            caught += 1
    assert caught > 0
