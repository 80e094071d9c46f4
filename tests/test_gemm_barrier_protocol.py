"""Randomized model of the wide W4A4 GEMM kernel's mbarrier protocol (CPU).

`w4a4_gemm_wide_kernel` (nvfp4_w4a4_gemm_gb300/csrc/gemm.cu) runs six roles
on a 4-stage shared-memory ring: the TMA warp, two scale-copy warps, the MMA
warp and eight epilogue warps, which also scale each tile's compensation
residual tiles.  They hand stages to one another through mbarriers, and an
mbarrier wait only compares the PARITY of the barrier's phase, so a waiter
that falls two phases behind (or waits two phases ahead) passes on the wrong
use of a stage.  Such a mistake faults or corrupts data only under some
timings, so it is checked here, on the CPU, against a model of every role's
waits and arrivals under random delays:

* every arrival fits in its barrier's pending count (no overflow);
* every role that touches a stage finds in it the use it expects (the TMA
  data of that use, the scale copies of that use, the residual scaled by all
  eight epilogue warps before the MMA reads it);
* no schedule deadlocks.

The model is run with the kernel's protocol and with two protocols that are
known to be wrong (the MMA warp not waiting for the first copy warp on
compensation uses; the epilogue warps waiting on the stage's `full` barrier
with a parity computed from the use count), which the checks must reject.
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise AssertionError(f"arrival overflow on {self.name} in phase {self.done}")
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def passed(self, parity):
        """try_wait.parity: true once the phase of this parity has completed."""
        return (self.done & 1) != parity


class WideGemmModel:
    """Roles of the wide kernel as generators that yield wait predicates.

    `uses` numbers the ring's stage uses in the order every role walks them:
    per output tile, n_kt FP4 k-tiles then n_ct compensation k-tiles."""

    def __init__(self, seed, n_tiles, n_kt, n_ct, protocol="kernel", stages=4):
        self.r = random.Random(seed)
        self.S, self.n_kt, self.n_ct, self.T = stages, n_kt, n_ct, n_tiles
        self.protocol = protocol
        ring = lambda name, count: [Barrier(f"{name}[{i}]", count) for i in range(stages)]
        self.full, self.empty = ring("full", 1), ring("empty", 1)
        self.sf_full, self.sf_full2 = ring("sf_full", 1), ring("sf_full2", 1)
        self.comp_ready, self.ct_landed = ring("comp_ready", 8), ring("ct_landed", 1)
        self.acc_full, self.acc_empty = Barrier("acc_full", 1), Barrier("acc_empty", 8)
        self.content = [None] * stages   # the use whose TMA data the stage holds
        self.sfa = [None] * stages       # the use whose A / B-low scales are in TMEM
        self.sfb2 = [None] * stages      # the use whose B-high scales are in TMEM
        self.scaled = [set() for _ in range(stages)]
        self.events = []
        self.now, self.seq = 0.0, 0
        self.last_async = {}

    def later(self, fn, issuer, lo, hi):
        """An asynchronous completion (TMA landing, tcgen05.commit); one
        issuer's commits complete in issue order."""
        t = max(self.now + self.r.uniform(lo, hi), self.last_async.get(issuer, 0.0) + 1e-6)
        self.last_async[issuer] = t
        self.seq += 1
        self.events.append((t, self.seq, fn))

    def uses(self):
        u = 0
        for t in range(self.T):
            for j in range(self.n_kt + self.n_ct):
                yield t, j, u
                u += 1

    def slot(self, u):
        return u % self.S, (u // self.S) & 1

    def tma(self):
        for _, _, u in self.uses():
            st, ph = self.slot(u)
            yield lambda: self.empty[st].passed(ph ^ 1)

            def land(st=st, u=u):
                self.content[st] = u
                self.scaled[st] = set()
                self.full[st].arrive()
            self.later(land, "tma", 5, 60)

    def copy_warp_a(self):          # warp 2: A + B rows 0..127 scale copies
        for _, j, u in self.uses():
            st, ph = self.slot(u)
            yield lambda: self.full[st].passed(ph)
            assert self.content[st] == u, ("copy warp A saw", self.content[st], "for use", u)
            if j < self.n_kt:
                def copied(st=st, u=u):
                    self.sfa[st] = u
                    self.sf_full[st].arrive()
                self.later(copied, "w2", 2, 20)
            else:
                self.sf_full[st].arrive()

    def copy_warp_b(self):          # warp 3: B rows 128..255 + compensation relay
        for _, j, u in self.uses():
            st, ph = self.slot(u)
            yield lambda: self.full[st].passed(ph)
            assert self.content[st] == u, ("copy warp B saw", self.content[st], "for use", u)
            if j < self.n_kt:
                self.comp_ready[st].arrive(8)

                def copied(st=st, u=u):
                    self.sfb2[st] = u
                    self.sf_full2[st].arrive()
                self.later(copied, "w3", 2, 20)
            else:
                self.sf_full2[st].arrive()
                self.ct_landed[st].arrive()

    def mma(self):
        acc_ph = 0
        walk = self.uses()
        for _ in range(self.T):
            yield lambda: self.acc_empty.passed(acc_ph ^ 1)
            acc_ph ^= 1
            for j in range(self.n_kt + self.n_ct):
                _, _, u = next(walk)
                st, ph = self.slot(u)
                if j < self.n_kt:
                    yield lambda: self.sf_full[st].passed(ph) and self.sf_full2[st].passed(ph)
                    assert (self.content[st], self.sfa[st], self.sfb2[st]) == (u, u, u), ("MMA", u)
                else:
                    if self.protocol == "mma_skips_copy_warp":
                        yield lambda: self.comp_ready[st].passed(ph)
                    else:
                        yield lambda: self.comp_ready[st].passed(ph) and self.sf_full[st].passed(ph)
                    assert self.content[st] == u and len(self.scaled[st]) == 8, ("MMA on compensation", u)

                def consumed(st=st):
                    self.content[st] = "consumed"
                    self.empty[st].arrive()
                self.later(consumed, "mma", 5, 40)
            self.later(self.acc_full.arrive, "mma", 5, 40)

    def epilogue_warp(self, w):
        acc_ph, stage, ct_phase, u0 = 0, 0, 0, 0
        for _ in range(self.T):
            if self.n_ct:
                stage = (stage + self.n_kt) % self.S
                for ct in range(self.n_ct):
                    u, st = u0 + self.n_kt + ct, stage
                    if self.protocol == "epilogue_waits_full":
                        ph = (u // self.S) & 1
                        yield lambda: self.full[st].passed(ph)
                    else:
                        par = (ct_phase >> st) & 1
                        yield lambda: self.ct_landed[st].passed(par)
                        ct_phase ^= 1 << st
                    assert self.content[st] == u, ("epilogue warp", w, "saw", self.content[st], "for use", u)
                    self.scaled[st].add(w)
                    self.comp_ready[st].arrive()
                    stage = (stage + 1) % self.S
            u0 += self.n_kt + self.n_ct
            yield lambda: self.acc_full.passed(acc_ph)
            acc_ph ^= 1
            self.acc_empty.arrive()
            stored = [False]                       # the tile's stores take a while
            self.later(lambda: stored.__setitem__(0, True), f"epi{w}", 0, 80)
            yield lambda: stored[0]

    def run(self):
        roles = [self.tma(), self.copy_warp_a(), self.copy_warp_b(), self.mma()]
        roles += [self.epilogue_warp(w) for w in range(8)]
        waiting = {}
        for g in roles:
            waiting[g] = next(g)
        while waiting or self.events:
            ready = [g for g, pred in waiting.items() if pred()]
            if ready and (not self.events or self.r.random() < 0.7):
                g = self.r.choice(ready)
                try:
                    waiting[g] = g.send(None)
                except StopIteration:
                    del waiting[g]
                self.now += self.r.uniform(0, 2)
            elif self.events:
                self.events.sort()
                t, _, fn = self.events.pop(0)
                self.now = max(self.now, t)
                fn()
            else:
                raise AssertionError(f"deadlock with {len(waiting)} roles waiting")


def _shapes(seed):
    r = random.Random(seed)
    return r.randint(1, 5), r.choice([1, 2, 3, 5, 16]), r.choice([0, 1, 2, 3, 4, 5, 8])


def _failures(protocol, n):
    bad = 0
    for seed in range(n):
        n_tiles, n_kt, n_ct = _shapes(seed)
        try:
            WideGemmModel(seed, n_tiles, n_kt, n_ct, protocol).run()
        except AssertionError:
            bad += 1
    return bad


def test_kernel_protocol_holds_under_random_schedules():
    assert _failures("kernel", 400) == 0


@pytest.mark.parametrize("protocol", ["mma_skips_copy_warp", "epilogue_waits_full"])
def test_model_rejects_known_wrong_protocols(protocol):
    assert _failures(protocol, 400) > 0
