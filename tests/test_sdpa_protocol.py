"""Host model of the attention kernel's barrier protocol (csrc/sdpa.cu), checked under
random interleavings.

The kernel's roles -- one copy producer, one MMA-issuing thread, eight row warps (two
per TMEM lane quarter) -- are modelled as coroutines over mbarriers with the hardware's
parity semantics: a wait for parity P returns as soon as the phase in progress has the
other parity.  Copies land and MMAs complete asynchronously (MMAs in issue order,
commits behind them).  For every run the model checks:

* no wait can be satisfied by the wrong phase (its barrier one phase behind) or be
  left waiting for a phase two ahead of the one meant;
* every buffer is written only after its last reader is done and read only after its
  writer is done: K and V ring slots, the two S buffers, the two P buffers and O;
* each phase of a P barrier is made of the arrivals of a single chunk;
* nothing deadlocks.

Planted mistakes (one P barrier instead of two, no wait before the O rescale, no
wait before a K or a V slot is refilled) must be caught: that is what makes the clean runs
mean something.  The model also shows that the row warps need no wait before
overwriting P_{j-2}: S(j)'s commit, which they wait for, arrives only after every
MMA issued before it -- P_{j-2} V_{j-2} included -- has completed.
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
    """One CTA of the kernel with `n` key chunks; `valid[w]` says whether row warp w holds
    any valid query row (decode: only the rows of one lane quarter)."""

    def __init__(self, n, valid, rng, single_pfull=False, no_rescale_wait=False, no_v_slot_wait=False,
                 no_k_slot_wait=False):
        self.n, self.valid, self.rng = n, valid, rng
        self.single_pfull = single_pfull
        self.no_rescale_wait, self.no_v_slot_wait = no_rescale_wait, no_v_slot_wait
        self.no_k_slot_wait = no_k_slot_wait
        B = Barrier
        self.bar_q = B("q", 1)
        self.kfull = [B("kfull0", 1), B("kfull1", 1)]
        self.vfull = [B("vfull0", 1), B("vfull1", 1)]
        self.sfull = [B("sfull0", 1), B("sfull1", 1)]
        self.pfull = [B("pfull0", 8)] if single_pfull else [B("pfull0", 8), B("pfull1", 8)]
        self.pvdone = [B("pvdone0", 1), B("pvdone1", 1)]
        self.mma_done = B("mma_done", 1)
        self.pending = []      # copies in flight: (barrier, action)
        self.pipe = []         # tensor pipe FIFO: ("op", name, on_done) or ("commit", barrier)
        # data state
        self.landed = set()    # ("K", j), ("V", i), "Q"
        self.s_done = set()    # S(j) complete
        self.pv_done = set()   # P_i V_i complete
        self.s_read = {}       # j -> row warps that have read S(j)
        self.p_written = {}    # i -> row warps that wrote P_i
        self.named = {}        # quarter -> [generation, waiting]
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

    # -- roles ----------------------------------------------------------------------
    def producer(self):
        n = self.n
        self.pending.append((self.bar_q, lambda: self.landed.add("Q")))
        self.pending.append((self.kfull[0], lambda: self.landed.add(("K", 0))))
        yield "step"
        for j in range(1, n + 1):
            if j < n:
                # K slot j % 2 free: S(j-2) done (a fresh barrier with parity 1 passes at once)
                if not self.no_k_slot_wait:
                    yield from self.wait(self.sfull[j & 1], ((j >> 1) & 1) ^ 1, (j >> 1) - 1, "producer")
                if j >= 2:
                    self.need(j - 2 in self.s_done, "K slot %d refilled before S(%d) read it" % (j % 2, j - 2))
                self.pending.append((self.kfull[j & 1], lambda j=j: self.landed.add(("K", j))))
                yield "step"
            # V slot i % 2 free: P V(i-2) done
            i = j - 1
            if not self.no_v_slot_wait:
                yield from self.wait(self.pvdone[i & 1], ((i >> 1) & 1) ^ 1, (i >> 1) - 1, "producer")
            if i >= 2:
                self.need(i - 2 in self.pv_done, "V slot %d refilled before P V(%d) read it" % (i % 2, i - 2))
            self.pending.append((self.vfull[i & 1], lambda i=i: self.landed.add(("V", i))))
            yield "step"

    def mma(self):
        n = self.n
        yield from self.wait(self.bar_q, 0, 0, "mma")
        for j in range(n + 1):
            if j < n:
                yield from self.wait(self.kfull[j & 1], (j >> 1) & 1, j >> 1, "mma")
                self.need("Q" in self.landed and ("K", j) in self.landed, "S(%d) issued before Q/K landed" % j)
                if j >= 2:
                    self.need(len(self.s_read.get(j - 2, ())) == 8, "S(%d) overwrites S(%d) before all rows read it" % (j, j - 2))
                self.pipe.append(("op", "S", j))
                self.pipe.append(("commit", self.sfull[j & 1]))
                yield "step"
            if j >= 1:
                i = j - 1
                if self.single_pfull:
                    yield from self.wait(self.pfull[0], i & 1, i, "mma")
                else:
                    yield from self.wait(self.pfull[i & 1], (i >> 1) & 1, i >> 1, "mma")
                yield from self.wait(self.vfull[i & 1], (i >> 1) & 1, i >> 1, "mma")
                writers = self.p_written.get(i, set())
                need = {w for w in range(8) if self.valid[w]}
                self.need(need <= writers, "P V(%d) issued before P_%d was written by warps %s" % (i, i, sorted(need - writers)))
                self.need(("V", i) in self.landed, "P V(%d) issued before V_%d landed" % (i, i))
                self.pipe.append(("op", "PV", i))
                self.pipe.append(("commit", self.pvdone[i & 1]))
                yield "step"
        self.pipe.append(("commit", self.mma_done))
        yield from self.wait(self.mma_done, 0, 0, "mma")

    def row_warp(self, w):
        n, quarter = self.n, w % 4
        for j in range(n):
            yield from self.wait(self.sfull[j & 1], (j >> 1) & 1, j >> 1, "row%d" % w)
            self.need(j in self.s_done, "row %d read S(%d) before it was complete" % (w, j))
            self.s_read.setdefault(j, set()).add(w)
            yield "step"
            yield from self.named_sync(quarter)
            # P_j overwrites P_{j-2}: no wait of its own, S(j)'s commit came after P V(j-2)
            if self.valid[w]:
                if j >= 2:
                    self.need(j - 2 in self.pv_done, "row %d wrote P_%d over P_%d before P V(%d) was done" % (w, j, j - 2, j - 2))
                self.p_written.setdefault(j, set()).add(w)
                yield "step"
                key = (quarter, j)
                if key not in self.rescale:
                    self.rescale[key] = j >= 1 and self.rng.random() < 0.3
                if self.rescale[key]:
                    if not self.no_rescale_wait:
                        yield from self.wait(self.pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1, (j - 1) >> 1,
                                             "row%d" % w)
                    self.need(j - 1 in self.pv_done, "row %d rescaled O before P V(%d) was done" % (w, j - 1))
                    yield "step"
            bar = self.pfull[0] if self.single_pfull else self.pfull[j & 1]
            bar.arrive(j)
            yield "step"
            yield from self.named_sync(quarter)
        yield from self.wait(self.pvdone[(n - 1) & 1], ((n - 1) >> 1) & 1, (n - 1) >> 1, "row%d" % w)
        self.need(n - 1 in self.pv_done, "row %d read O before the last P V" % w)

    # -- asynchronous engines --------------------------------------------------------
    def engine_step(self):
        """Advance one copy or the tensor pipe; False if neither can move."""
        choices = []
        if self.pending:
            choices.append("copy")
        if self.pipe:
            choices.append("pipe")
        if not choices:
            return False
        if self.rng.choice(choices) == "copy":
            bar, act = self.pending.pop(self.rng.randrange(len(self.pending)))
            act()
            bar.arrive()
        else:
            kind, *rest = self.pipe.pop(0)
            if kind == "op":
                name, idx = rest
                (self.s_done if name == "S" else self.pv_done).add(idx)
            else:
                rest[0].arrive()
        return True

    def run(self, max_steps=200000):
        agents = [self.producer(), self.mma()] + [self.row_warp(w) for w in range(8)]
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
    run_many({pattern: PATTERNS[pattern]}, range(1, 11), range(40))


@pytest.mark.parametrize("mutation", ["single_pfull", "no_rescale_wait", "no_v_slot_wait", "no_k_slot_wait"])
def test_planted_protocol_mistakes_are_caught(mutation):
    with pytest.raises(Hazard):
        run_many(PATTERNS, range(2, 11), range(40), **{mutation: True})
