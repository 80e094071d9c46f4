"""Randomized models of the W4A4 GEMM kernels' mbarrier protocols (CPU).

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

`NarrowGemmModel` does the same for `w4a4_gemm_kernel` (four copy warps on one
barrier, two accumulators plus a compensation accumulator, split-K units, and
the early weight loads issued before the wait for the preceding kernel).
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, count, 0
        self.tx = 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise AssertionError(f"arrival overflow on {self.name} in phase {self.done}")
        self._maybe_complete()

    def expect_tx(self, nbytes):
        """mbarrier.arrive.expect_tx: one arrival plus bytes still to land."""
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        if self.tx < 0:
            raise AssertionError(f"transaction bytes below zero on {self.name}")
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def passed(self, parity):
        """try_wait.parity: true once the phase of this parity has completed."""
        return (self.done & 1) != parity


class WideGemmModel:
    """Roles of the wide kernel as generators that yield wait predicates.

    `uses` numbers the ring's stage uses in the order every role walks them:
    per output tile, n_kt FP4 k-tiles then n_ct compensation k-tiles."""

    def __init__(self, seed, n_tiles, n_kt, n_ct, protocol="kernel", stages=4, early=False, scale_r=True):
        self.r = random.Random(seed)
        self.S, self.n_kt, self.n_ct, self.T = stages, n_kt, n_ct, n_tiles
        self.protocol, self.early = protocol, early
        # scale_r: the epilogue warps scale each compensation residual tile
        # (False: a residual pre-scaled by the quantizer goes to the MMA as is)
        self.scale_r = scale_r and n_ct > 0
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
        # each stage use lands in two halves (activations, weights); with
        # early weights the weight halves of the first FP4 k-tiles go out
        # before the wait for the preceding kernel, under one expect_tx
        pre = min(self.S, self.n_kt) if (self.early and self.T) else 0
        halves = [dict() for _ in range(self.S)]

        def land(st, u, half):
            halves[st][half] = u
            if halves[st].get("a") == u and halves[st].get("b") == u:
                self.content[st] = u
                self.scaled[st] = set()
            self.full[st].complete_tx(1)
        for i in range(pre):
            self.full[i].expect_tx(2)
            self.later(lambda i=i: land(i, i, "b"), "tma", 5, 60)
        yield lambda: True  # griddepcontrol.wait
        for _, _, u in self.uses():
            st, ph = self.slot(u)
            if u >= pre:
                yield lambda: self.empty[st].passed(ph ^ 1)
                self.full[st].expect_tx(2)
                self.later(lambda st=st, u=u: land(st, u, "b"), "tma", 5, 60)
            self.later(lambda st=st, u=u: land(st, u, "a"), "tma", 5, 60)

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
                if self.scale_r:
                    self.comp_ready[st].arrive(8)

                def copied(st=st, u=u):
                    self.sfb2[st] = u
                    self.sf_full2[st].arrive()
                self.later(copied, "w3", 2, 20)
            else:
                self.sf_full2[st].arrive()
                if self.scale_r:
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
                elif not self.scale_r:
                    # pre-scaled residual: the tile goes to the MMA as it lands,
                    # once both copy warps (which wait on `full` too) passed it
                    yield lambda: (self.full[st].passed(ph) and self.sf_full[st].passed(ph)
                                   and self.sf_full2[st].passed(ph))
                    assert self.content[st] == u, ("MMA on compensation", u)
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
            if self.scale_r:
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

    def roles(self):
        return ([self.tma(), self.copy_warp_a(), self.copy_warp_b(), self.mma()]
                + [self.epilogue_warp(w) for w in range(8)])

    def run(self):
        roles = self.roles()
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


class NarrowGemmModel(WideGemmModel):
    """Roles of `w4a4_gemm_kernel` (128-row tiles, decode and small M): the
    TMA warp, four scale-copy warps that each commit once per stage on
    `sf_full` (count 4), the MMA warp with two accumulators and one
    compensation accumulator, and four epilogue warps.  Work units carry a
    k-tile range (split-K) and compensation k-tiles only on their first split.
    With early weights the producer issues the weight half of its first
    stages (one arrive.expect_tx for the whole stage) before the wait for the
    preceding kernel, and the activation half after it."""

    def __init__(self, seed, units, protocol="kernel", stages=4, early=False):
        self.r = random.Random(seed)
        self.S, self.units, self.protocol, self.early = stages, units, protocol, early
        ring = lambda name, count: [Barrier(f"{name}[{i}]", count) for i in range(stages)]
        self.full, self.empty = ring("full", 1), ring("empty", 1)
        self.sf_full = ring("sf_full", 3 if protocol == "sf_full_count_3" else 4)
        self.acc_full = [Barrier(f"acc_full[{i}]", 1) for i in range(2)]
        self.acc_empty = [Barrier(f"acc_empty[{i}]", 4) for i in range(2)]
        self.comp_empty = Barrier("comp_empty", 4)
        self.a_part = [None] * stages     # use whose activation half landed
        self.b_part = [None] * stages     # use whose weight half landed
        self.chunks = [dict() for _ in range(stages)]  # copy warp -> use whose chunk is in TMEM
        self.acc = [None, None]           # (unit, complete?) held by each accumulator
        self.comp = None
        self.events, self.now, self.seq, self.last_async = [], 0.0, 0, {}
        self.waited = False               # the producer's wait for the preceding kernel

    def walk(self):
        """(unit index, k-tile index within the unit, is compensation, use)."""
        u = 0
        for i, (n_kt, n_ct) in enumerate(self.units):
            for j in range(n_kt + n_ct):
                yield i, j, j >= n_kt, u
                u += 1

    def tma(self):
        first_kt = self.units[0][0] if self.units else 0
        pre = min(self.S, first_kt) if self.early else 0
        for i in range(pre):               # weight halves before the wait, ring known empty
            self.full[i].expect_tx(2)
            self.later(lambda i=i: (self.b_part.__setitem__(i, i), self.full[i].complete_tx(1)), "tma", 5, 60)
            if self.protocol == "early_double_arrive":
                self.full[i].expect_tx(0)
        yield lambda: True
        self.waited = True
        for _, _, comp, u in self.walk():
            st, ph = self.slot(u)
            early = u < pre
            if not early:
                yield lambda: self.empty[st].passed(ph ^ 1)
                self.full[st].expect_tx(2)
                self.later(lambda st=st, u=u: (self.b_part.__setitem__(st, u), self.full[st].complete_tx(1)),
                           "tma", 5, 60)
            self.later(lambda st=st, u=u: (self.a_part.__setitem__(st, u), self.full[st].complete_tx(1)),
                       "tma", 5, 60)

    def copy_warp(self, w):
        for _, _, comp, u in self.walk():
            st, ph = self.slot(u)
            yield lambda: self.full[st].passed(ph)
            assert (self.a_part[st], self.b_part[st]) == (u, u), ("copy warp", w, "use", u)
            if comp:
                self.sf_full[st].arrive()
            else:
                def copied(st=st, u=u):
                    self.chunks[st][w] = u
                    self.sf_full[st].arrive()
                self.later(copied, f"cp{w}", 2, 20)

    def mma(self):
        acc, acc_ph, comp_ph = 0, 0, 0
        walk = self.walk()
        for i, (n_kt, n_ct) in enumerate(self.units):
            yield lambda: self.acc_empty[acc].passed(acc_ph ^ 1)
            assert self.acc[acc] is None or self.acc[acc][1] == "read", ("accumulator still unread", i)
            self.acc[acc] = (i, "writing")
            for j in range(n_kt + n_ct):
                _, _, comp, u = next(walk)
                st, ph = self.slot(u)
                if j == n_kt:  # as the kernel: the compensation accumulator is claimed after the FP4 k-tiles
                    if self.protocol != "mma_skips_comp_empty":
                        yield lambda: self.comp_empty.passed(comp_ph ^ 1)
                    comp_ph ^= 1
                yield lambda: self.sf_full[st].passed(ph)
                assert (self.a_part[st], self.b_part[st]) == (u, u), ("MMA", u)
                if comp:
                    if j == n_kt:  # the unit's first compensation k-tile
                        assert self.comp is None or self.comp[1] == "read", ("compensation accumulator unread", i)
                        self.comp = (i, "writing")
                else:
                    assert all(self.chunks[st].get(w) == u for w in range(4)), ("MMA before all scale chunks", u)

                def consumed(st=st):
                    self.a_part[st] = self.b_part[st] = "consumed"
                    self.empty[st].arrive()
                self.later(consumed, "mma", 5, 40)

            def done(a=acc, i=i, c=bool(n_ct)):
                self.acc[a] = (i, "complete")
                if c:
                    self.comp = (i, "complete")
                self.acc_full[a].arrive()
            self.later(done, "mma", 5, 40)
            acc ^= 1
            if acc == 0:
                acc_ph ^= 1

    def epilogue_warp(self, w):
        acc, acc_ph = 0, 0
        for i, (n_kt, n_ct) in enumerate(self.units):
            yield lambda: self.acc_full[acc].passed(acc_ph)
            assert self.acc[acc] == (i, "complete"), ("epilogue read", self.acc[acc], "for unit", i)
            if n_ct:
                assert self.comp == (i, "complete"), ("epilogue compensation read", self.comp, "for unit", i)
            stored = [False]
            self.later(lambda stored=stored: stored.__setitem__(0, True), f"epi{w}", 0, 30)
            yield lambda stored=stored: stored[0]
            self.epi_done = getattr(self, "epi_done", {})
            self.epi_done[(i, w)] = True
            if all(self.epi_done.get((i, x)) for x in range(4)):
                self.acc[acc] = (i, "read")
                if n_ct:
                    self.comp = (i, "read")
            self.acc_empty[acc].arrive()
            if n_ct:
                self.comp_empty.arrive()
            acc ^= 1
            if acc == 0:
                acc_ph ^= 1

    def roles(self):
        return [self.tma(), self.mma()] + [self.copy_warp(w) for w in range(4)] + \
               [self.epilogue_warp(w) for w in range(4)]


def _narrow_units(seed):
    """A CTA's work units: (FP4 k-tiles, compensation k-tiles); compensation
    only on a unit's first split."""
    r = random.Random(seed)
    units = []
    for _ in range(r.randint(1, 4)):
        split = r.choice([1, 1, 2, 3])
        n_kt, n_ct = r.choice([1, 2, 4, 16]), r.choice([0, 1, 2])
        for p in range(split):
            lo, hi = p * n_kt // split, (p + 1) * n_kt // split
            if hi > lo or p == 0:
                units.append((max(hi - lo, 1), n_ct if p == 0 else 0))
    return units


def _narrow_failures(protocol, n, early):
    bad = 0
    for seed in range(n):
        try:
            NarrowGemmModel(seed, _narrow_units(seed), protocol, stages=random.Random(seed).choice([4, 7]),
                            early=early).run()
        except AssertionError:
            bad += 1
    return bad


@pytest.mark.parametrize("early", [False, True])
def test_narrow_kernel_protocol_holds_under_random_schedules(early):
    assert _narrow_failures("kernel", 300, early) == 0


@pytest.mark.parametrize("protocol,early", [("sf_full_count_3", False), ("mma_skips_comp_empty", False),
                                            ("early_double_arrive", True)])
def test_narrow_model_rejects_known_wrong_protocols(protocol, early):
    assert _narrow_failures(protocol, 300, early) > 0


def _shapes(seed):
    r = random.Random(seed)
    return r.randint(1, 5), r.choice([1, 2, 3, 5, 16]), r.choice([0, 1, 2, 3, 4, 5, 8])


def _failures(protocol, n, early=False, scale_r=True):
    bad = 0
    for seed in range(n):
        n_tiles, n_kt, n_ct = _shapes(seed)
        try:
            WideGemmModel(seed, n_tiles, n_kt, n_ct, protocol, early=early, scale_r=scale_r).run()
        except AssertionError:
            bad += 1
    return bad


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("scale_r", [False, True])
def test_kernel_protocol_holds_under_random_schedules(early, scale_r):
    assert _failures("kernel", 400, early, scale_r) == 0


@pytest.mark.parametrize("protocol", ["mma_skips_copy_warp", "epilogue_waits_full"])
def test_model_rejects_known_wrong_protocols(protocol):
    assert _failures(protocol, 400) > 0


# ------------------------------------------------------- pair-tile kernel --
class SignedTxBarrier(Barrier):
    """An mbarrier whose transaction count may go below zero for a while: in
    the pair kernel the peer CTA's copies can land on the leader's `full`
    barrier before the leader's arrive.expect_tx of that phase."""

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()


class PairGemmModel(WideGemmModel):
    """Roles of `w4a4_gemm_pair_kernel`: two CTAs (rank 0 = leader, rank 1 =
    peer).  Each CTA runs an operand TMA warp (a 5-stage ring), a scale TMA
    warp (an 8-stage ring of its own, running ahead of the operands) and
    eight epilogue warps; the leader alone runs the MMA warp and the copy warp,
    which moves a k-tile's scales into the TMEM slot of its operand stage as
    soon as they have landed and the slot's previous MMAs are done.  Barrier
    homes as in the kernel: `full`, `sf_full`, `comp_ready` (16), `sfl_full`
    and `acc_empty` (16) in the leader; `empty`, `acc_full`, `ct_landed` and
    `sfl_empty` in each CTA.  Both CTAs' copies complete on the leader's
    barriers; the MMA and copy warps' commits and the leader's relays arrive on
    both CTAs; the peer's epilogue warps arrive remotely on the leader.  Remote
    arrivals are asynchronous and unordered with the leader's own.  With
    `scale_r` the epilogue warps scale each compensation residual tile before
    the MMA reads it; without it (a residual the quantizer pre-scaled) the
    compensation tiles go straight to the MMA.  Besides the wide model's
    checks, the model asserts that no TMEM scale slot or scale stage is
    overwritten while still in use, and that when both CTAs have finished every
    role (the final cluster barrier, after which a CTA may exit) nothing is
    still in flight towards either CTA."""

    SF_STAGES = 8

    def __init__(self, seed, n_tiles, n_kt, n_ct, protocol="kernel", stages=5, early=False, scale_r=True):
        self.r = random.Random(seed)
        self.S, self.n_kt, self.n_ct, self.T = stages, n_kt, n_ct, n_tiles
        self.protocol, self.early, self.scale_r = protocol, early, scale_r and n_ct > 0
        ring = lambda name, count, cls=Barrier, n=stages: [cls(f"{name}[{i}]", count) for i in range(n)]
        self.full = ring("full", 1, SignedTxBarrier)
        self.sf_full = ring("sf_full", 1)
        self.comp_ready = ring("comp_ready", 16)
        self.sfl_full = ring("sfl_full", 1, SignedTxBarrier, self.SF_STAGES)
        self.acc_empty = Barrier("acc_empty", 16)
        self.empty = [ring(f"empty.{c}", 1) for c in range(2)]
        self.ct_landed = [ring(f"ct_landed.{c}", 1) for c in range(2)]
        self.sfl_empty = [ring(f"sfl_empty.{c}", 1, Barrier, self.SF_STAGES) for c in range(2)]
        self.acc_full = [Barrier(f"acc_full.{c}", 1) for c in range(2)]
        self.content = [[None] * stages for _ in range(2)]
        self.sf_content = [[None] * self.SF_STAGES for _ in range(2)]
        self.sf_copied = [None] * self.SF_STAGES   # k-tile whose scales the copies finished reading
        self.tmem_sf = [None] * stages             # use whose scales are in the stage's TMEM slot
        self.mma_done = [None] * stages            # last use of the stage whose MMAs completed
        self.scaled = [[set() for _ in range(stages)] for _ in range(2)]
        self.acc = [None, None]
        self.events, self.now, self.seq, self.last_async = [], 0.0, 0, {}
        self.finished = 0

    def fp4_index(self, u):
        """FP4 k-tile counter of use u (compensation uses carry none)."""
        t, j = divmod(u, self.n_kt + self.n_ct)
        return t * self.n_kt + j if j < self.n_kt else None

    def tma_cta(self, c):
        leader = c == 0
        pre = min(self.S, self.n_kt) if (self.early and self.T) else 0
        halves = [dict() for _ in range(self.S)]

        def land(st, u, half):
            halves[st][half] = u
            if halves[st].get("a") == u and halves[st].get("b") == u:
                self.content[c][st] = u
                self.scaled[c][st] = set()
            self.full[st].complete_tx(1)
        for i in range(pre):
            if leader:
                self.full[i].expect_tx(4)
            self.later(lambda i=i: land(i, i, "b"), f"tma{c}", 5, 60)
        yield lambda: True  # griddepcontrol.wait
        n_uses = 0
        for _, _, u in self.uses():
            st, ph = self.slot(u)
            if u >= pre:
                yield lambda: self.empty[c][st].passed(ph ^ 1)
                if leader:
                    self.full[st].expect_tx(4)
                self.later(lambda st=st, u=u: land(st, u, "b"), f"tma{c}", 5, 60)
            self.later(lambda st=st, u=u: land(st, u, "a"), f"tma{c}", 5, 60)
            n_uses += 1
        if self.protocol != "no_wind_down":
            for i in range(self.S):
                if n_uses > i:
                    last = (n_uses - 1 - i) // self.S
                    yield lambda i=i, last=last: self.empty[c][i].passed(last & 1)
        self.finished += 1

    def sf_producer(self, c):
        leader = c == 0
        R = self.SF_STAGES
        n = self.T * self.n_kt

        def land(sl, g):
            assert self.sf_copied[sl] == (g - R if g >= R else None), ("scale stage overwritten", sl, g)
            self.sf_content[c][sl] = g
            self.sfl_full[sl].complete_tx(1)
        yield lambda: True  # griddepcontrol.wait
        for g in range(n):
            sl, ph = g % R, (g // R) & 1
            yield lambda sl=sl, ph=ph: self.sfl_empty[c][sl].passed(ph ^ 1)
            if leader:
                self.sfl_full[sl].expect_tx(2)
            self.later(lambda sl=sl, g=g: land(sl, g), f"sftma{c}", 5, 40)
        if self.protocol != "no_wind_down":
            for i in range(R):
                if n > i:
                    last = (n - 1 - i) // R
                    yield lambda i=i, last=last: self.sfl_empty[c][i].passed(last & 1)
        self.finished += 1

    def copy_warp(self):
        R = self.SF_STAGES
        for _, j, u in self.uses():
            st, ph = self.slot(u)
            if self.protocol != "copier_skips_slot_wait":
                yield lambda: self.empty[0][st].passed(ph ^ 1)
            if j < self.n_kt:
                g = self.fp4_index(u)
                sl, sph = g % R, (g // R) & 1
                yield lambda sl=sl, sph=sph: self.sfl_full[sl].passed(sph)
                assert self.sf_content[0][sl] == g and self.sf_content[1][sl] == g, ("copy warp scales", g)
                assert self.mma_done[st] == (u - self.S if u >= self.S else None), ("TMEM scale slot in use", u)
                if self.scale_r:
                    self.comp_ready[st].arrive(16)

                def copied(st=st, u=u, sl=sl, g=g):
                    # the commits arrive once the copies are done: on the
                    # leader's barriers, and (remote, unordered) on the peer's
                    self.tmem_sf[st] = u
                    self.sf_copied[sl] = g
                    self.sf_full[st].arrive()
                    self.sfl_empty[0][sl].arrive()
                    self.later(lambda: self.sfl_empty[1][sl].arrive(), "w3peer", 0, 40)
                self.later(copied, "w3", 2, 20)
            else:
                if self.scale_r:
                    yield lambda: self.full[st].passed(ph)
                    assert self.content[0][st] == u and self.content[1][st] == u, ("relay", u)
                    self.ct_landed[0][st].arrive()
                    self.later(self.ct_landed[1][st].arrive, "w3remote", 1, 15)
                self.sf_full[st].arrive()
        self.finished += 1

    def mma(self):
        acc_ph = 0
        walk = self.uses()
        for t in range(self.T):
            yield lambda: self.acc_empty.passed(acc_ph ^ 1)
            acc_ph ^= 1
            for c in range(2):
                assert self.acc[c] is None or self.acc[c][1] == "read", ("accumulator unread", c, t)
                self.acc[c] = (t, "writing")
            for j in range(self.n_kt + self.n_ct):
                _, _, u = next(walk)
                st, ph = self.slot(u)
                if j < self.n_kt:
                    yield lambda: self.full[st].passed(ph) and self.sf_full[st].passed(ph)
                    assert self.tmem_sf[st] == u, ("MMA scales", u)
                elif self.scale_r:
                    yield lambda: self.sf_full[st].passed(ph) and self.comp_ready[st].passed(ph)
                    assert all(len(self.scaled[c][st]) == 8 for c in range(2)), ("MMA on unscaled residual", u)
                else:
                    yield lambda: self.sf_full[st].passed(ph) and self.full[st].passed(ph)
                assert self.content[0][st] == u and self.content[1][st] == u, ("MMA operands", u)

                def consumed(st, c, u):
                    if c == 0:
                        self.mma_done[st] = u
                    self.content[c][st] = "consumed"
                    self.empty[c][st].arrive()
                self.later(lambda st=st, u=u: consumed(st, 0, u), "mma", 5, 40)
                self.later(lambda st=st, u=u: consumed(st, 1, u), "mma_peer", 5, 60)

            def done(c, t=t):
                self.acc[c] = (t, "complete")
                self.acc_full[c].arrive()
            self.later(lambda: done(0), "mma", 5, 40)
            self.later(lambda: done(1), "mma_peer", 5, 60)
        if self.T and self.protocol != "no_wind_down":
            yield lambda: self.acc_empty.passed(acc_ph ^ 1)
        self.finished += 1

    def epilogue_warp_cta(self, c, w):
        acc_ph, stage, ct_phase, u0 = 0, 0, 0, 0
        for t in range(self.T):
            if self.scale_r:
                stage = (stage + self.n_kt) % self.S
                for ct in range(self.n_ct):
                    u, st = u0 + self.n_kt + ct, stage
                    par = (ct_phase >> st) & 1
                    yield lambda st=st, par=par: self.ct_landed[c][st].passed(par)
                    ct_phase ^= 1 << st
                    assert self.content[c][st] == u, ("epilogue", c, w, "saw", self.content[c][st], "for", u)
                    self.scaled[c][st].add(w)
                    if c == 0:
                        self.comp_ready[st].arrive()
                    else:
                        self.later(lambda st=st: self.comp_ready[st].arrive(), f"e{c}{w}", 1, 15)
                    stage = (stage + 1) % self.S
            u0 += self.n_kt + self.n_ct
            yield lambda: self.acc_full[c].passed(acc_ph)
            acc_ph ^= 1
            assert self.acc[c] == (t, "complete"), ("epilogue read", self.acc[c], "for tile", t)
            self.epi_read = getattr(self, "epi_read", {})
            self.epi_read[(c, t, w)] = True
            if all(self.epi_read.get((c, t, x)) for x in range(8)):
                self.acc[c] = (t, "read")
            if c == 0:
                self.acc_empty.arrive()
            else:
                self.later(self.acc_empty.arrive, f"e{c}{w}", 1, 120)
            stored = [False]
            self.later(lambda stored=stored: stored.__setitem__(0, True), f"st{c}{w}", 0, 80)
            yield lambda stored=stored: stored[0]
        self.finished += 1

    def roles(self):
        return ([self.tma_cta(0), self.tma_cta(1), self.sf_producer(0), self.sf_producer(1), self.copy_warp(),
                 self.mma()] + [self.epilogue_warp_cta(c, w) for c in range(2) for w in range(8)])

    def check_quiet_at_exit(self):
        """Called when every role has finished: nothing may still land."""
        assert not self.events, ("in flight at exit", len(self.events))


def _pair_failures(protocol, n, early=False, scale_r=True):
    bad = 0
    for seed in range(n):
        n_tiles, n_kt, n_ct = _shapes(seed)
        m = PairGemmModel(seed, n_tiles, n_kt, n_ct, protocol, early=early, scale_r=scale_r)
        try:
            m.run_to_exit()
        except AssertionError:
            bad += 1
    return bad


def _run_to_exit(self):
    """run(), but stop as soon as every role has finished and check that no
    asynchronous copy or arrival is still pending at that moment."""
    roles = self.roles()
    n = len(roles)
    waiting = {g: next(g) for g in roles}
    while True:
        if self.finished == n and not waiting:
            self.check_quiet_at_exit()
            return
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


PairGemmModel.run_to_exit = _run_to_exit


@pytest.mark.parametrize("early", [False, True])
@pytest.mark.parametrize("scale_r", [False, True])
def test_pair_kernel_protocol_holds_under_random_schedules(early, scale_r):
    assert _pair_failures("kernel", 400, early, scale_r) == 0


def test_pair_model_rejects_a_missing_wind_down():
    # without the producers' and the MMA warp's final waits, commits and
    # remote arrivals can still be in flight when the CTAs pass the final
    # cluster barrier
    assert _pair_failures("no_wind_down", 400) > 0


def test_pair_model_rejects_copies_into_a_busy_scale_slot():
    # the copy warp must wait for the MMAs of the stage's previous use before
    # it overwrites that stage's TMEM scale slot
    assert _pair_failures("copier_skips_slot_wait", 400) > 0
