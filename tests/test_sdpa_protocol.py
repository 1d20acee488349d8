"""Host model of the attention kernel's barrier protocol (csrc/sdpa.cu), checked under
random interleavings.

The kernel's roles -- a K copy producer, a V copy producer, a thread that issues the
S = Q K^T MMAs, a thread that issues the P V MMAs, eight row warps (two per TMEM lane
quarter) -- are modelled as coroutines over mbarriers with the hardware's parity
semantics: a wait for parity P returns as soon as the phase in progress has the other
parity.  Copies land in any order.  Each issuing thread's MMAs complete in its issue
order and its commits arrive behind them, but the two threads' MMAs may complete in
any interleaving (the model assumes nothing about order across threads).  For every
run the model checks:

* no wait can be satisfied by the wrong phase (its barrier one phase behind) or be
  left waiting for a phase two ahead of the one meant;
* every buffer is written only after its last reader is done and read only after its
  writer is done: the K and V ring slots, the three S buffers (S(j), then P_j written
  over it by the rows), and O (rescaled by the rows between two P V MMAs, read out at
  the end);
* each phase of a P barrier is made of the arrivals of a single chunk;
* nothing deadlocks.

Planted mistakes must be caught, which is what makes the clean runs mean something:
two P V barriers instead of four (with two, a parity wait for P V(i) can pass while
P V(i-2) is still running), S(t) not waiting for P V(t-3), two P barriers instead of
three, and a missing wait before a K slot, a V slot or the O rescale.  With four P V
barriers the read-out could also wait on the last P V's barrier (the model shows it
safe: `readout_on_pvdone`); the kernel waits on the all-done barrier.
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


class Model:
    """One CTA with `n` key chunks; `valid[w]` says whether row warp w holds any valid
    query row (decode: only the rows of one lane quarter)."""

    def __init__(self, n, valid, rng, n_pvdone=4, n_pfull=3, readout_on_pvdone=False,
                 no_s_wait=False, no_k_slot_wait=False, no_v_slot_wait=False,
                 no_rescale_wait=False):
        self.n, self.valid, self.rng = n, valid, rng
        self.n_pvdone, self.n_pfull = n_pvdone, n_pfull
        self.readout_on_pvdone, self.no_s_wait = readout_on_pvdone, no_s_wait
        self.no_k_slot_wait, self.no_v_slot_wait = no_k_slot_wait, no_v_slot_wait
        self.no_rescale_wait = no_rescale_wait
        B = Barrier
        self.bar_q = B("q", 1)
        self.kfull = [B("kfull%d" % i, 1) for i in range(2)]
        self.vfull = [B("vfull%d" % i, 1) for i in range(2)]
        self.sfull = [B("sfull%d" % i, 1) for i in range(3)]
        self.pfull = [B("pfull%d" % i, 8) for i in range(n_pfull)]
        self.pvdone = [B("pvdone%d" % i, 1) for i in range(n_pvdone)]
        self.mma_done = B("mma_done", 1)
        self.pending = []                       # copies in flight: (barrier, action)
        self.pipe = {"S": [], "PV": []}         # per issuing thread, in issue order
        # data state
        self.landed = set()                     # ("K", j), ("V", i), "Q"
        self.s_done, self.pv_done = set(), set()
        self.s_read = {}                        # j -> row warps that read S(j)
        self.p_written = {}                     # j -> row warps that wrote P_j
        self.named = {}
        self.rescale = {}

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

    def named_sync(self, quarter):
        gen_waiting = self.named.setdefault(quarter, [0, 0])
        gen = gen_waiting[0]
        gen_waiting[1] += 1
        if gen_waiting[1] == 2:
            gen_waiting[0] += 1
            gen_waiting[1] = 0
            return
        while self.named[quarter][0] == gen:
            yield "blocked"

    def pvbar(self, i):
        return self.pvdone[i % self.n_pvdone], (i // self.n_pvdone) & 1, i // self.n_pvdone

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

    def pv_thread(self):
        for i in range(self.n):
            yield from self.wait(self.pfull[i % self.n_pfull], (i // self.n_pfull) & 1, i // self.n_pfull, "PV")
            yield from self.wait(self.vfull[i & 1], (i >> 1) & 1, i >> 1, "PV")
            need = {w for w in range(8) if self.valid[w]}
            writers = self.p_written.get(i, set())
            self.need(need <= writers, "P V(%d) issued before P_%d was written by warps %s" % (i, i, sorted(need - writers)))
            self.need(("V", i) in self.landed, "P V(%d) issued before V_%d landed" % (i, i))
            self.pipe["PV"].append(("op", "PV", i))
            bar, _, _ = self.pvbar(i)
            self.pipe["PV"].append(("commit", bar))
            yield "step"
        self.pipe["PV"].append(("commit", self.mma_done))

    def row_warp(self, w):
        n, quarter = self.n, w % 4
        for j in range(n):
            yield from self.wait(self.sfull[j % 3], (j // 3) & 1, j // 3, "row%d" % w)
            self.need(j in self.s_done, "row %d read S(%d) before it was complete" % (w, j))
            self.s_read.setdefault(j, set()).add(w)
            yield "step"
            yield from self.named_sync(quarter)
            if self.valid[w]:
                key = (quarter, j)
                if key not in self.rescale:
                    self.rescale[key] = j >= 1 and self.rng.random() < 0.3
                # P_j over S buffer j % 3 (already read by this warp)
                self.p_written.setdefault(j, set()).add(w)
                yield "step"
                if self.rescale[key]:
                    if not self.no_rescale_wait:
                        bar, par, k = self.pvbar(j - 1)
                        yield from self.wait(bar, par, k, "row%d" % w)
                    self.need(j - 1 in self.pv_done, "row %d rescaled O before P V(%d) was done" % (w, j - 1))
                    self.need(j not in self.pv_done, "O rescaled for chunk %d after its P V" % j)
                    yield "step"
            self.pfull[j % self.n_pfull].arrive(j)
            yield "step"
            yield from self.named_sync(quarter)
        if self.readout_on_pvdone:
            bar, par, k = self.pvbar(n - 1)
            yield from self.wait(bar, par, k, "row%d" % w)
        else:
            yield from self.wait(self.mma_done, 0, 0, "row%d" % w)
        self.need(all(i in self.pv_done for i in range(n)), "row %d read O before every P V was done" % w)

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
        for b in self.pfull:
            for ph, tags in enumerate(b.phase_tags):
                self.need(len(set(tags)) == 1, "%s phase %d mixes chunks %s" % (b.name, ph, sorted(set(tags))))


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
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_protocol_mistakes_are_caught(mutation):
    with pytest.raises(Hazard):
        run_many(PATTERNS, range(2, 12), range(60), **MUTATIONS[mutation])
