"""A model of the decode-attention kernel's page-ring synchronization, checked on
CPU under random schedules: the protocol itself, independent of any device
tool.

What is modelled, as `csrc/ekv_attn_body.cuh` does it for one CTA:
- ns stages (even); page j of the split always goes to stage j mod ns and is
  the (j / ns)-th copy into it; a copy is an mbarrier transaction that lands
  at an arbitrary later time.
- mbarrier phases: one pending arrival per phase (an arrive with an expected
  transaction count), completion when the arrival is in and the transaction
  count is back at zero (it may dip below zero while a copy lands before its
  arrival); `wait(parity)` succeeds once the phase of that parity completed,
  i.e. while the barrier's current phase index has the other parity.
- Static assignment (uniform split, ring of >= two pairs per warp, ns a
  multiple of 2 NW): one barrier per stage pair armed by the even page's
  issuer for both pages; warp w takes pairs w, w + NW, ... and waits on its
  pair barrier directly; it refills the stages of its previous pair right
  after the next pair's wait.
- Dynamic assignment: one barrier per stage, a shared counter hands out
  pairs, a warp first waits for the stage's issue record to show its page,
  then for the barrier, and refills right after computing.  A split with
  mixed page formats runs the same per-stage waits with the static pairs
  when the ring allows them ("static, mixed").
- The first fill (pages 0 .. ns-1, issuing threads in any order) and the
  drain (each stage, or each pair's even stage, waits for its last copy).

Checked: every page is computed exactly once, from a stage holding that
page's landed copy; no stage is refilled before its page was computed; no
wait is left that can never succeed (the drain included); nothing is in
flight at the end.
"""
import random

import pytest


class Barrier:
    def __init__(self):
        self.phase = 0      # completed phases
        self.pending = 1    # arrivals still expected in the current phase
        self.tx = 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = 1

    def arrive_expect(self, nbytes):
        self.tx += nbytes
        self.pending -= 1
        assert self.pending == 0, "two arrivals in one phase"
        self._check()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._check()

    def ready(self, parity):
        return (self.phase & 1) != parity


class Ring:
    BYTES = 1

    def __init__(self, np_, nw, ns, mode, rng):
        assert ns % 2 == 0 and mode in ("static", "static_mixed", "dynamic")
        if mode != "dynamic":
            assert ns % (2 * nw) == 0 and ns >= 4 * nw
        self.np, self.nw, self.ns, self.mode, self.rng = np_, nw, ns, mode, rng
        self.static = mode == "static"
        self.pairb = self.static
        nb = ns // 2 if self.pairb else ns
        self.bars = [Barrier() for _ in range(nb)]
        self.stage = [None] * ns          # page whose copy landed in the stage
        self.stage_busy = [None] * ns     # page issued into the stage, not yet computed
        self.issued = [-1] * ns
        self.flight = []                  # (stage, page, barrier)
        self.computed = []
        self.counter = 0

    def bar_of(self, si):
        return self.bars[si >> 1] if self.pairb else self.bars[si]

    def issue(self, k, si):
        assert si == k % self.ns
        assert self.stage_busy[si] is None, f"stage {si} refilled before page {self.stage_busy[si]} was computed"
        bar = self.bar_of(si)
        if not self.pairb:
            bar.arrive_expect(self.BYTES)
        elif si % 2 == 0:
            bar.arrive_expect(self.BYTES * (2 if k + 1 < self.np else 1))
        self.stage_busy[si] = k
        self.flight.append((si, k, bar))
        self.issued[si] = k

    def land_one(self):
        i = self.rng.randrange(len(self.flight))
        si, k, bar = self.flight.pop(i)
        self.stage[si] = k
        bar.complete_tx(self.BYTES)

    def compute(self, k, si):
        assert self.stage[si] == k, f"page {k} computed from stage {si} holding {self.stage[si]}"
        self.computed.append(k)
        self.stage_busy[si] = None

    # ---- one warp (a generator: yields a condition it waits on) -------------
    def warp(self, w):
        ns, np_ = self.ns, self.np
        if self.static:
            it = 0
            while True:
                k = 2 * (w + self.nw * it)
                if k >= np_:
                    break
                two = k + 1 < np_
                q, si = k // ns, k % ns
                bar = self.bars[si >> 1]
                yield lambda bar=bar, q=q: bar.ready(q & 1)
                if it > 0:                       # refill the previous pair's stages
                    kp = k - 2 * self.nw
                    for lane in (0, 1):
                        j = kp + ns + lane
                        if j < np_:
                            yield None           # lanes issue in either order
                            self.issue(j, (kp % ns) + lane)
                self.compute(k, si)
                if two:
                    self.compute(k + 1, si + 1)
                it += 1
        else:
            it = 0
            while True:
                if self.mode == "static_mixed":
                    k = 2 * (w + self.nw * it)
                    it += 1
                else:
                    k = self.counter
                    self.counter += 2
                if k >= np_:
                    break
                two = k + 1 < np_
                q, si = k // ns, k % ns
                for kk, s in ((k, si), (k + 1, si + 1)) if two else ((k, si),):
                    yield lambda s=s, kk=kk: self.issued[s] == kk
                    bar = self.bars[s]
                    yield lambda bar=bar, q=q: bar.ready(q & 1)
                self.compute(k, si)
                if two:
                    self.compute(k + 1, si + 1)
                for lane in (0, 1) if two else (0,):
                    j = k + ns + lane
                    if j < np_:
                        self.issue(j, si + lane)

    def run(self):
        rng = self.rng
        # the first fill: page p by some thread, in any order
        first = list(range(min(self.ns, self.np)))
        rng.shuffle(first)
        for p in first:
            self.issue(p, p)
            if self.flight and rng.random() < 0.3:
                self.land_one()
        warps = {w: self.warp(w) for w in range(self.nw)}
        waits = {w: None for w in warps}
        while warps:
            runnable = [w for w in warps if waits[w] is None or waits[w]()]
            if not runnable or (self.flight and rng.random() < 0.4):
                assert self.flight, "every warp waits on a phase that can never complete"
                self.land_one()
                continue
            w = rng.choice(runnable)
            try:
                waits[w] = next(warps[w])
            except StopIteration:
                del warps[w], waits[w]
        # the drain: each stage (each pair's even stage) waits for its last copy
        drains = []
        for si in range(self.ns):
            if self.pairb and si % 2:
                continue
            if self.issued[si] >= 0:
                q = self.issued[si] // self.ns
                drains.append((self.bar_of(si), q & 1))
        while self.flight:
            self.land_one()
        for bar, parity in drains:
            assert bar.ready(parity), "a drain wait on a phase that can never complete"
        assert sorted(self.computed) == list(range(self.np))


CASES = [  # (pages, warps, stages)
    (0, 4, 16), (1, 4, 16), (2, 4, 16), (7, 4, 16), (16, 4, 16), (17, 4, 16), (31, 4, 16),
    (32, 4, 16), (33, 4, 16), (100, 4, 16), (101, 4, 24), (431, 16, 64), (350, 16, 64),
    (96, 16, 96), (97, 16, 96), (300, 8, 32),
]


@pytest.mark.parametrize("np_, nw, ns", CASES)
@pytest.mark.parametrize("mode", ["static", "static_mixed", "dynamic"])
def test_ring_protocol_random_schedules(np_, nw, ns, mode):
    if mode != "dynamic" and not (ns % (2 * nw) == 0 and ns >= 4 * nw):
        pytest.skip("static assignment needs a ring of two pairs per warp or more")
    for seed in range(40):
        Ring(np_, nw, ns, mode, random.Random(seed)).run()


def test_drain_of_odd_stage_would_wait_forever():
    """The model catches the drain mistake the kernel once had: with pair
    barriers, the odd stage of a pair may hold an older page than the even one
    (an odd page count), and waiting on that older page's phase parity never
    succeeds once the newer phase has completed."""
    r = Ring(3 * 16 + 1, 4, 16, "static", random.Random(0))   # 49 pages: page 48 alone
    r.run()
    odd = 48 % 16 + 1                 # the odd stage beside page 48
    assert r.issued[odd] == 33        # a round older than page 48
    assert not r.bar_of(odd).ready((r.issued[odd] // 16) & 1)
