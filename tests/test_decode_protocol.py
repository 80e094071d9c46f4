"""Randomized model of the decode layer's barrier protocol (CPU).

`w4a4_decode_kernel` (nvfp4_w4a4_gemm_gb300/csrc/gemm.cu) runs as clusters of
four CTAs.  Each CTA streams its weight tiles through a ring (producer warp ->
`full`, MMA warp -> `empty`), while the cluster quantizes the token rows
together: CTA r quantizes the 256-column k-tiles r, r + 4, ... and the
64-slot residual tiles r, r + 4, ..., writes them into its own shared memory
(then one local arrival on the k-tile group's `xready` barrier, or on
`rready`) and sends them to the other three CTAs with bulk copies whose bytes
complete on those CTAs' barriers (whose byte counts were set when the
barriers were initialized).  The dynamic tensor scale needs every CTA's amax
partial first, exchanged the same way on `amax_bar`.

The checks, under random delays of every copy and commit:

* every role finds what it expects: the MMA warp the weight tile of the use
  and the token codes / residual tiles of every k-tile it multiplies; the
  quantizing warps every CTA's amax partial;
* arrivals and transaction bytes never overshoot a barrier's phase;
* no bulk copy into or out of a CTA is still in flight when the cluster
  passes its closing barrier (a CTA with no output tile of its own does not
  wait for its token data in the MMA loop, so the quantizing warps wait for
  it before the CTA leaves);
* no schedule deadlocks.

Three protocols known to be wrong must be rejected: no final wait for the
incoming copies, barriers that do not expect the bytes of the other CTAs'
k-tiles, and the local arrival made before the k-tile is written.
"""
import random

import pytest

C = 4            # CTAs per cluster
KT_BYTES = 3072  # codes 2 KB + scale chunks 1 KB per k-tile
RES_BYTES = 2048


class Barrier:
    """An mbarrier phase counter: pending arrivals and transaction bytes."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise AssertionError(f"arrival overflow on {self.name}")
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def expect_tx(self, nbytes):
        self.tx += nbytes

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        if self.tx < 0:
            raise AssertionError(f"bytes beyond the phase on {self.name}")
        self._maybe_complete()

    def passed(self, parity):
        return (self.done & 1) != parity


class DecodeModel:
    def __init__(self, seed, n_tiles, n_kt, n_ct, stages, dynamic, protocol="kernel"):
        self.r = random.Random(seed)
        self.n_tiles, self.n_kt, self.n_ct, self.S = n_tiles, n_kt, n_ct, stages
        self.n_st = (n_kt + 1) // 2  # two k-tiles per FP4 ring use
        self.n_grp = (n_kt + C - 1) // C
        self.dynamic, self.protocol = dynamic, protocol
        self.events, self.now, self.seq, self.last = [], 0.0, 0, {}
        self.copies_in_flight = 0
        self.cta = [self._cta_state(c) for c in range(C)]

    def _cta_state(self, rank):
        S = self.S
        st = dict(
            full=[Barrier(f"full{rank}.{i}", 1) for i in range(S)],
            empty=[Barrier(f"empty{rank}.{i}", 1) for i in range(S)],
            acc_full=[Barrier(f"acc_full{rank}.{i}", 1) for i in range(2)],
            acc_empty=[Barrier(f"acc_empty{rank}.{i}", 4) for i in range(2)],
            amax=Barrier(f"amax{rank}", 1), rready=Barrier(f"rready{rank}", 1),
            xready=[Barrier(f"xready{rank}.{g}", 1) for g in range(self.n_grp)],
            content=[None] * S, tok=[False] * self.n_kt, res=[False] * self.n_ct,
            parts={rank}, tiles=list(range(rank, self.n_tiles, C)), finished=0)
        # barrier setup (before the CTA's cluster arrival)
        st["amax"].arrive_expect_tx(16 * (C - 1))
        own_ct = sum(1 for ct in range(self.n_ct) if ct % C == rank)
        if self.n_ct > own_ct:
            st["rready"].expect_tx(RES_BYTES * (self.n_ct - own_ct))
        for g in range(self.n_grp):
            in_grp = min(C, self.n_kt - g * C)
            owns = g * C + rank < self.n_kt
            nbytes = KT_BYTES * (in_grp - (1 if owns else 0))
            if self.protocol == "no_expected_bytes":
                nbytes = 0
            if owns:
                st["xready"][g].expect_tx(nbytes)
            else:
                st["xready"][g].arrive_expect_tx(nbytes)
        return st

    # ------------------------------------------------------------ timing --
    def later(self, fn, issuer, lo, hi):
        t = max(self.now + self.r.uniform(lo, hi), self.last.get(issuer, 0.0) + 1e-6)
        self.last[issuer] = t
        self.seq += 1
        self.events.append((t, self.seq, fn))

    def copy(self, src, dst, what, bar, nbytes):
        """A CTA-to-CTA bulk copy: the data lands, then its bytes complete."""
        self.copies_in_flight += 1

        def land():
            what()
            self.copies_in_flight -= 1
            bar.complete_tx(nbytes)
        self.later(land, f"copy{src}->{dst}", 5, 60)

    # ------------------------------------------------------------- roles --
    def producer(self, rank):
        s = self.cta[rank]
        u = 0
        for t in s["tiles"]:
            for i in range(self.n_st + self.n_ct):
                stage, ph = u % self.S, (u // self.S) & 1
                if u >= self.S:
                    yield lambda: s["empty"][stage].passed(ph ^ 1)
                s["full"][stage].arrive_expect_tx(1)

                def land(stage=stage, key=(t, i)):
                    s["content"][stage] = key
                    s["full"][stage].complete_tx(1)
                self.later(land, f"tma{rank}", 10, 80)
                u += 1
        s["finished"] += 1

    def mma(self, rank):
        s = self.cta[rank]
        u, acc, acc_ph = 0, 0, 0
        for n, t in enumerate(s["tiles"]):
            yield lambda: s["acc_empty"][acc].passed(acc_ph ^ 1)
            seen = -1
            for i in range(self.n_st + self.n_ct):
                stage, ph = u % self.S, (u // self.S) & 1
                kts = [k for k in (2 * i, 2 * i + 1) if i < self.n_st and k < self.n_kt]
                if n == 0:
                    for g in sorted({k // C for k in kts}):
                        if g > seen:
                            yield lambda g=g: s["xready"][g].passed(0)
                            seen = g
                    if i == self.n_st:
                        yield lambda: s["rready"].passed(0)
                yield lambda: s["full"][stage].passed(ph)
                assert s["content"][stage] == (t, i), ("MMA", rank, t, i, s["content"][stage])
                for k in kts:
                    assert s["tok"][k], ("token k-tile missing", rank, k)
                if i >= self.n_st:
                    assert s["res"][i - self.n_st], ("residual tile missing", rank, i - self.n_st)

                def consumed(stage=stage):
                    s["content"][stage] = "consumed"
                    s["empty"][stage].arrive()
                self.later(consumed, f"mma{rank}", 5, 40)
                u += 1
            self.later(s["acc_full"][acc].arrive, f"mma{rank}", 5, 40)
            acc ^= 1
            if acc == 0:
                acc_ph ^= 1
        s["finished"] += 1

    def epilogue(self, rank, w):
        s = self.cta[rank]
        acc, acc_ph = 0, 0
        for _ in s["tiles"]:
            yield lambda: s["acc_full"][acc].passed(acc_ph)
            s["acc_empty"][acc].arrive()
            acc ^= 1
            if acc == 0:
                acc_ph ^= 1
        s["finished"] += 1

    def quantize(self, rank):
        s = self.cta[rank]
        yield lambda: all(self.started)  # cluster_wait: every CTA set its barriers up
        if self.dynamic:
            for c in range(C):
                if c != rank:
                    self.copy(rank, c, lambda c=c: self.cta[c]["parts"].add(rank), self.cta[c]["amax"], 16)
            yield lambda: s["amax"].passed(0)
            assert s["parts"] == set(range(C)), ("amax partials", rank, s["parts"])
        for kt in range(rank, self.n_kt, C):
            g = kt // C
            if self.protocol == "arrive_before_write":
                s["xready"][g].arrive()
                self.later(lambda kt=kt: s["tok"].__setitem__(kt, True), f"write{rank}", 0, 30)
            else:
                s["tok"][kt] = True
                s["xready"][g].arrive()
            for c in range(C):
                if c != rank:
                    dst = self.cta[c]
                    self.copy(rank, c, lambda dst=dst, kt=kt: dst["tok"].__setitem__(kt, True),
                              dst["xready"][g], KT_BYTES)
            yield lambda: True
        if self.n_ct:
            for ct in range(rank, self.n_ct, C):
                s["res"][ct] = True
            s["rready"].arrive()
            for ct in range(rank, self.n_ct, C):
                for c in range(C):
                    if c != rank:
                        dst = self.cta[c]
                        self.copy(rank, c, lambda dst=dst, ct=ct: dst["res"].__setitem__(ct, True), dst["rready"],
                                  RES_BYTES)
        if self.protocol != "no_end_wait":
            # every copy into this CTA has landed before it may leave
            for g in range(self.n_grp):
                yield lambda g=g: s["xready"][g].passed(0)
            if self.n_ct:
                yield lambda: s["rready"].passed(0)
            if self.dynamic:
                yield lambda: s["amax"].passed(0)
        s["finished"] += 1

    def roles(self, rank):
        return ([self.producer(rank), self.mma(rank), self.quantize(rank)]
                + [self.epilogue(rank, w) for w in range(4)])

    def run(self):
        self.started = [False] * C
        waiting = {}
        for c in range(C):
            self.started[c] = True  # barrier setup, then the cluster arrival
            for g in self.roles(c):
                waiting[g] = next(g, None)
        waiting = {g: p for g, p in waiting.items() if p is not None}
        n_roles = 3 + 4
        while True:
            if all(s["finished"] == n_roles for s in self.cta) and not waiting:
                # the closing cluster barrier: every CTA is there, so they may leave
                assert self.copies_in_flight == 0, ("bulk copies in flight at exit", self.copies_in_flight)
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
                _, _, fn = self.events.pop(0)
                fn()
            else:
                raise AssertionError(f"deadlock with {len(waiting)} roles waiting")


def _failures(protocol, n):
    bad = 0
    for seed in range(n):
        r = random.Random(1000 + seed)
        n_tiles = r.choice([1, 2, 3, 4, 5, 8, 9])  # clusters where some CTAs have no tile, or two
        n_kt = r.choice([1, 2, 3, 5, 8, 16, 17, 32])
        n_ct = r.choice([0, 1, 2, 4])
        m = DecodeModel(seed, n_tiles, n_kt, n_ct, r.choice([3, 4, 7]), r.random() < 0.5, protocol)
        try:
            m.run()
        except AssertionError:
            bad += 1
    return bad


def test_decode_protocol_holds_under_random_schedules():
    assert _failures("kernel", 600) == 0


@pytest.mark.parametrize("protocol", ["no_end_wait", "no_expected_bytes", "arrive_before_write"])
def test_decode_model_rejects_known_wrong_protocols(protocol):
    assert _failures(protocol, 600) > 0
