"""Host model of the attention kernel's barrier protocol (csrc/sdpa.cu), checked under
random interleavings.

The kernel's roles -- a K copy producer, a V copy producer, a thread that issues the
S = Q K^T MMAs, a thread that issues the P V MMAs, eight row warps (two per TMEM lane
quarter, which take the chunks in turn) -- are modelled as coroutines over mbarriers
with the hardware's parity semantics: a wait for parity P returns as soon as the phase
in progress has the other parity.  Copies land in any order.  Each issuing thread's
MMAs complete in its issue order and its commits arrive behind them, but the two
threads' MMAs may complete in any interleaving (the model assumes nothing about order
across threads).  The two warps of a lane quarter hand the running shift over through
a named barrier per direction (the chooser arrives, the other waits) and meet at a
third at the end; a named barrier completes when both warps have arrived, so a warp
that arrived twice before the other waits would break it.  For every run the model
checks:

* no wait can be satisfied by the wrong phase (its barrier one phase behind) or be
  left waiting for a phase two ahead of the one meant;
* every buffer is written only after its last reader is done and read only after its
  writer is done: the K and V ring slots, the three S buffers (S(j), then P_j written
  over it by the rows in two halves, each read by its own P V MMAs), the shift slots,
  and O (rescaled by the rows before a chunk's P V, read out at the end);
* the shifts are chosen in chunk order: a warp chooses chunk j's after it has taken
  chunk j-1's from the other warp;
* each phase of a P barrier is made of the arrivals of a single chunk; every named
  barrier ends with no arrival left waiting;
* nothing deadlocks.

Planted mistakes must be caught, which is what makes the clean runs mean something:
two P V barriers instead of four (with two, a parity wait for P V(i) can pass while
P V(i-2) is still running), S(t) not waiting for P V(t-3), two P barriers instead of
three, a missing wait before a K slot, a V slot, the O rescale or the upper half's
P V MMAs, P barriers counting all eight warps, one shared shift barrier for both
directions, and the last shift left untaken.  With four P V barriers the read-out
could also wait on the last P V's barrier (the model shows it safe:
`readout_on_pvdone`); the kernel waits on the all-done barrier.
"""
import random

import pytest


class Hazard(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.done = 0          # completed phases; the phase in progress has index `done`
        self.arrived = 0
        self.tags = []
        self.phase_tags = []

    def arrive(self, tag=None):
        self.arrived += 1
        self.tags.append(tag)
        if self.arrived == self.count:
            self.phase_tags.append(self.tags)
            self.tags, self.arrived = [], 0
            self.done += 1

    def ready(self, parity):
        return (self.done & 1) != parity


class NamedBarrier:
    """A hardware named barrier over the two warps of a lane quarter: it completes when
    both have arrived (arrive does not wait, sync does).  An arrival by a warp that
    already arrived in the phase in progress would complete it without the other."""

    def __init__(self, name):
        self.name, self.phase, self.arrived = name, 0, []

    def _add(self, w):
        if w in self.arrived:
            raise Hazard("%s: warp %d arrives twice in one phase" % (self.name, w))
        self.arrived.append(w)
        if len(self.arrived) == 2:
            self.arrived, self.phase = [], self.phase + 1

    def arrive(self, w):
        self._add(w)

    def sync(self, w):
        ph = self.phase
        self._add(w)
        while self.phase == ph:
            yield "blocked"


class Model:
    """One CTA with `n` key chunks; `valid[w]` says whether row warp w holds any valid
    query row (decode: only the rows of one lane quarter).  Row warp w serves lane
    quarter w % 4 and the chunks j with j % 2 == w // 4."""

    def __init__(self, n, valid, rng, n_pvdone=4, n_pfull=3, p_count=4, readout_on_pvdone=False,
                 no_s_wait=False, no_k_slot_wait=False, no_v_slot_wait=False,
                 no_rescale_wait=False, no_phi_wait=False, one_shift_barrier=False,
                 skip_last_receive=False):
        self.n, self.valid, self.rng = n, valid, rng
        self.n_pvdone, self.n_pfull = n_pvdone, n_pfull
        self.readout_on_pvdone, self.no_s_wait = readout_on_pvdone, no_s_wait
        self.no_k_slot_wait, self.no_v_slot_wait = no_k_slot_wait, no_v_slot_wait
        self.no_rescale_wait, self.no_phi_wait = no_rescale_wait, no_phi_wait
        self.skip_last_receive = skip_last_receive
        B = Barrier
        self.bar_q = B("q", 1)
        self.kfull = [B("kfull%d" % i, 1) for i in range(2)]
        self.vfull = [B("vfull%d" % i, 1) for i in range(2)]
        self.sfull = [B("sfull%d" % i, 1) for i in range(3)]
        self.pfull = [B("pfull%d" % i, p_count) for i in range(n_pfull)]
        self.phi = [B("phi%d" % i, p_count) for i in range(n_pfull)]
        self.pvdone = [B("pvdone%d" % i, 1) for i in range(n_pvdone)]
        self.mma_done = B("mma_done", 1)
        # named barriers per lane quarter: the shift chosen by group g, and the end meeting
        self.shift_bar = {}
        for q in range(4):
            b0 = NamedBarrier("shift q%d g0" % q)
            b1 = b0 if one_shift_barrier else NamedBarrier("shift q%d g1" % q)
            self.shift_bar[(q, 0)], self.shift_bar[(q, 1)] = b0, b1
        self.end_bar = [NamedBarrier("end q%d" % q) for q in range(4)]
        self.pending = []                       # copies in flight: (barrier, action)
        self.pipe = {"S": [], "PV": []}         # per issuing thread, in issue order
        # data state
        self.landed = set()                     # ("K", j), ("V", i), "Q"
        self.s_done, self.pv_done = set(), set()
        self.pv_lo_issued, self.pv_lo_done = set(), set()
        self.p_written = {}                     # (j, half) -> row warps that wrote it
        self.rescale = {}
        self.shift_slot = {}                    # (quarter, slot) -> [chunk, taken]
        self.shift_known = {}                   # warp -> last chunk whose shift it holds

    # -- checks ---------------------------------------------------------------------
    def need(self, cond, what):
        if not cond:
            raise Hazard(what)

    def wait(self, bar, parity, k, who):
        """Generator: block until bar is ready for parity; k is the phase meant."""
        while True:
            if bar.done >= k + 2:
                raise Hazard("%s waits for phase %d of %s, which is already at %d" % (who, k, bar.name, bar.done))
            if bar.ready(parity):
                self.need(bar.done >= k + 1, "%s: wait for phase %d of %s passed at %d" % (who, k, bar.name, bar.done))
                return
            yield "blocked"

    def pvbar(self, i):
        return self.pvdone[i % self.n_pvdone], (i // self.n_pvdone) & 1, i // self.n_pvdone

    def pbar(self, bars, j):
        return bars[j % self.n_pfull], (j // self.n_pfull) & 1, j // self.n_pfull

    # -- roles ----------------------------------------------------------------------
    def k_producer(self):
        self.pending.append((self.bar_q, lambda: self.landed.add("Q")))
        self.pending.append((self.kfull[0], lambda: self.landed.add(("K", 0))))
        yield "step"
        for j in range(1, self.n):
            if j >= 2 and not self.no_k_slot_wait:
                yield from self.wait(self.sfull[(j - 2) % 3], ((j - 2) // 3) & 1, (j - 2) // 3, "kprod")
            if j >= 2:
                self.need(j - 2 in self.s_done, "K slot %d refilled before S(%d) read it" % (j % 2, j - 2))
            self.pending.append((self.kfull[j & 1], lambda j=j: self.landed.add(("K", j))))
            yield "step"

    def v_producer(self):
        for i in range(self.n):
            if i >= 2 and not self.no_v_slot_wait:
                bar, par, k = self.pvbar(i - 2)
                yield from self.wait(bar, par, k, "vprod")
            if i >= 2:
                self.need(i - 2 in self.pv_done, "V slot %d refilled before P V(%d) read it" % (i % 2, i - 2))
            self.pending.append((self.vfull[i & 1], lambda i=i: self.landed.add(("V", i))))
            yield "step"

    def s_thread(self):
        yield from self.wait(self.bar_q, 0, 0, "S")
        for t in range(self.n):
            yield from self.wait(self.kfull[t & 1], (t >> 1) & 1, t >> 1, "S")
            if t >= 3 and not self.no_s_wait:
                bar, par, k = self.pvbar(t - 3)
                yield from self.wait(bar, par, k, "S")
            self.need("Q" in self.landed and ("K", t) in self.landed, "S(%d) issued before Q/K landed" % t)
            self.pipe["S"].append(("op", "S", t))
            self.pipe["S"].append(("commit", self.sfull[t % 3]))
            yield "step"

    def writers_needed(self, j):
        return {w for w in range(8) if self.valid[w] and w // 4 == j % 2}

    def pv_thread(self):
        for i in range(self.n):
            yield from self.wait(*self.pbar(self.pfull, i), "PV")
            yield from self.wait(self.vfull[i & 1], (i >> 1) & 1, i >> 1, "PV")
            need, writers = self.writers_needed(i), self.p_written.get((i, 0), set())
            self.need(need <= writers, "P V(%d) lower half issued before warps %s wrote it" % (i, sorted(need - writers)))
            self.need(("V", i) in self.landed, "P V(%d) issued before V_%d landed" % (i, i))
            self.pv_lo_issued.add(i)
            self.pipe["PV"].append(("op", "PVlo", i))
            yield "step"
            if not self.no_phi_wait:
                yield from self.wait(*self.pbar(self.phi, i), "PV")
            writers = self.p_written.get((i, 1), set())
            self.need(need <= writers, "P V(%d) upper half issued before warps %s wrote it" % (i, sorted(need - writers)))
            self.pipe["PV"].append(("op", "PV", i))
            bar, _, _ = self.pvbar(i)
            self.pipe["PV"].append(("commit", bar))
            yield "step"
        self.pipe["PV"].append(("commit", self.mma_done))

    def receive(self, w, jp):
        q, g = w % 4, w // 4
        yield from self.shift_bar[(q, g ^ 1)].sync(w)
        slot = self.shift_slot.get((q, jp & 1))
        self.need(slot is not None and slot[0] == jp, "row %d took the shift of chunk %d from a slot holding %s" % (w, jp, slot))
        slot[1] = True
        self.shift_known[w] = jp

    def row_warp(self, w):
        n, q, grp = self.n, w % 4, w // 4
        self.shift_known[w] = -1
        for j in range(grp, n, 2):
            yield from self.wait(self.sfull[j % 3], (j // 3) & 1, j // 3, "row%d" % w)
            self.need(j in self.s_done, "row %d read S(%d) before it was complete" % (w, j))
            yield "step"
            if j >= 1:
                yield from self.receive(w, j - 1)
            self.need(self.shift_known[w] == j - 1, "row %d chose chunk %d's shift before taking chunk %d's" % (w, j, j - 1))
            old = self.shift_slot.get((q, j & 1))
            self.need(old is None or old[1], "row %d overwrote the shift of chunk %d before it was taken" % (w, old[0] if old else -1))
            self.shift_slot[(q, j & 1)] = [j, False]
            self.shift_known[w] = j
            self.shift_bar[(q, grp)].arrive(w)
            yield "step"
            key = (q, j)
            if key not in self.rescale:
                self.rescale[key] = j >= 1 and self.rng.random() < 0.3
            if self.valid[w] and self.rescale[key]:
                if not self.no_rescale_wait:
                    bar, par, k = self.pvbar(j - 1)
                    yield from self.wait(bar, par, k, "row%d" % w)
                self.need(j - 1 in self.pv_done, "row %d rescaled O before P V(%d) was done" % (w, j - 1))
                self.need(j not in self.pv_lo_issued, "O rescaled for chunk %d after its P V started" % j)
                yield "step"
            for half, bars in ((0, self.pfull), (1, self.phi)):
                if self.valid[w]:
                    # P_j's half over S buffer j % 3, which this warp has read out
                    self.p_written.setdefault((j, half), set()).add(w)
                    yield "step"
                bars[j % self.n_pfull].arrive(j)
                yield "step"
        if n >= 1 and (n - 1) % 2 != grp and not self.skip_last_receive:
            yield from self.receive(w, n - 1)
        yield from self.end_bar[q].sync(w)
        if self.readout_on_pvdone:
            bar, par, k = self.pvbar(n - 1)
            yield from self.wait(bar, par, k, "row%d" % w)
        else:
            yield from self.wait(self.mma_done, 0, 0, "row%d" % w)
        self.need(all(i in self.pv_done for i in range(n)), "row %d read O before every P V was done" % w)
        self.need(self.shift_known[w] == n - 1, "row %d ended without the last chunk's shift" % w)

    # -- asynchronous engines --------------------------------------------------------
    def engine_step(self):
        """Land one copy or advance one issuing thread's MMA stream; False if nothing can."""
        choices = []
        if self.pending:
            choices.append("copy")
        for name in ("S", "PV"):
            if self.pipe[name]:
                choices.append(name)
        if not choices:
            return False
        c = self.rng.choice(choices)
        if c == "copy":
            bar, act = self.pending.pop(self.rng.randrange(len(self.pending)))
            act()
            bar.arrive()
            return True
        kind, *rest = self.pipe[c].pop(0)
        if kind == "op":
            name, idx = rest
            if name == "S":
                # S(t) writes S buffer t % 3: P_{t-3} in it must have been read by P V(t-3)
                if idx >= 3:
                    self.need(idx - 3 in self.pv_done, "S(%d) overwrote P_%d before P V(%d) was done" % (idx, idx - 3, idx - 3))
                self.s_done.add(idx)
            elif name == "PVlo":
                self.pv_lo_done.add(idx)
            else:
                self.pv_done.add(idx)
        else:
            rest[0].arrive()
        return True

    def run(self, max_steps=300000):
        agents = [self.k_producer(), self.v_producer(), self.s_thread(), self.pv_thread()] + \
                 [self.row_warp(w) for w in range(8)]
        live = list(range(len(agents)))
        for _ in range(max_steps):
            if not live:
                break
            if self.rng.random() < 0.3 and self.engine_step():
                continue
            order = live[:]
            self.rng.shuffle(order)
            moved = False
            for a in order:
                try:
                    r = next(agents[a])
                except StopIteration:
                    live.remove(a)
                    moved = True
                    break
                if r != "blocked":
                    moved = True
                    break
            if not moved and not self.engine_step():
                raise Hazard("deadlock with agents %s blocked" % live)
        else:
            raise Hazard("did not finish")
        for b in self.pfull + self.phi:
            for ph, tags in enumerate(b.phase_tags):
                self.need(len(set(tags)) == 1, "%s phase %d mixes chunks %s" % (b.name, ph, sorted(set(tags))))
        for nb in list(self.shift_bar.values()) + self.end_bar:
            self.need(not nb.arrived, "%s ends with warps %s left arrived" % (nb.name, nb.arrived))


PATTERNS = {
    "all rows": [True] * 8,
    "decode (one lane quarter)": [w % 4 == 0 for w in range(8)],
    "two quarters": [w % 4 in (0, 1) for w in range(8)],
}


def run_many(patterns, chunks, seeds, **kw):
    for name, valid in patterns.items():
        for n in chunks:
            for seed in seeds:
                Model(n, valid, random.Random(1000 * n + seed), **kw).run()


@pytest.mark.parametrize("pattern", sorted(PATTERNS))
def test_protocol_holds(pattern):
    run_many({pattern: PATTERNS[pattern]}, range(1, 12), range(40))
    run_many({pattern: PATTERNS[pattern]}, range(1, 12), range(10), readout_on_pvdone=True)


MUTATIONS = {
    "two P V barriers": dict(n_pvdone=2),
    "S without the P V wait": dict(no_s_wait=True),
    "two P barriers": dict(n_pfull=2),
    "no K slot wait": dict(no_k_slot_wait=True),
    "no V slot wait": dict(no_v_slot_wait=True),
    "no rescale wait": dict(no_rescale_wait=True),
    "no wait for the upper half of P": dict(no_phi_wait=True),
    "P barriers counting eight warps": dict(p_count=8),
    "one shift barrier for both directions": dict(one_shift_barrier=True),
    "last shift left untaken": dict(skip_last_receive=True),
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_protocol_mistakes_are_caught(mutation):
    with pytest.raises(Hazard):
        run_many(PATTERNS, range(2, 12), range(60), **MUTATIONS[mutation])
