"""A discrete-event model of the split-K barrier protocol at D = 64 (separate P columns, one
MMA issuer), paired and unpaired (host only, no GPU).

The roles follow the kernel's loops: the TMA producer (Q tiles, then K/V positions in ring
order), the MMA warp (S and PV issue, ring releases, the O1 hand-over between accumulations),
the two softmax warpgroups (S read, P write, warpgroup 1's own store of b, the (m, l) hand-off
and warpgroup 0's merge), the tensor pipe (operations and commits complete in issue order)
and the copy engine (loads land in any order). Random interleavings of many unit sequences
must finish (no deadlock), every parity wait must find its barrier at the phase it waits for
or the one before (never two behind, never past it), and every buffer must hold what its
reader expects: the ring slot's tile, the Q tile of the query tile, the S and P of the tile,
and each accumulator's tiles, never overwritten before its reader is done; and when a
warpgroup writes a tile's P (where the in-place O rescale runs), every earlier PV of its
accumulation has completed.

A unit is (na, nb): one query tile with na K/V tiles (nb = 0: unpaired, tiles alternate
between the warpgroups) or a pair, where warpgroup 0 takes a's first ceil((na + nb) / 2)
tiles, warpgroup 1 all nb tiles of b and then the rest of a. In the kernel a paired CTA runs
one unit; sequences of units here also cover the unpaired CTAs that run several.
"""

from __future__ import annotations

import random

import pytest


class Barrier:
    def __init__(self, name):
        self.name, self.done = name, 0

    def complete(self):
        self.done += 1


class Model:
    def __init__(self, units, stages, seed):
        self.units, self.stages = units, stages
        self.rnd = random.Random(seed)
        self.B = {}
        for n in ["QF", "QE", "ST", "O1Free", "O1Self", "OFB"]:
            self.B[n] = Barrier(n)
        for s in range(stages):
            self.B[("KF", s)], self.B[("KE", s)] = Barrier(("KF", s)), Barrier(("KE", s))
        for w in range(2):
            for n in ["SF", "SFree", "PF", "PVD", "OF"]:
                self.B[(n, w)] = Barrier((n, w))
        self.pipe = []   # tensor pipe: operations and commits, in issue order
        self.tma = []    # copies in flight: (barrier, buffer, value)
        self.q = {}      # Q buffer -> (unit, item)
        self.slot = {}   # ring stage -> (unit, kind, position)
        self.S = {0: None, 1: None}
        self.P = {0: None, 1: None}
        self.O = {0: None, 1: None}  # accumulator: dict(tag, n, read)
        self.stats = None

    # ---- helpers
    def ready(self, name, c):
        """Parity wait for completion c (1-based): satisfied when done == c. A barrier two
        phases behind would satisfy it by parity alone, one past would hide it: both fail."""
        d = self.B[name].done
        assert c - 1 <= d <= c, ("phase", name, "waits for", c, "done", d)
        return d == c

    @staticmethod
    def split(na, nb):
        nk = na + nb
        return nk, (nk + 1) // 2, nk // 2

    @staticmethod
    def tile(na, nb, w, u):
        """(item, K/V tile) of warpgroup w's u-th position (the kernel's unit_tile)."""
        n0 = (na + nb + 1) // 2
        if nb == 0:
            return "a", 2 * u + w
        if w == 0:
            return "a", u
        return ("b", u) if u < nb else ("a", n0 + (u - nb))

    @staticmethod
    def ring(nk):
        seq = [("K", 0)] + ([("K", 1)] if nk > 1 else [])
        for t2 in range(0, nk, 2):
            if t2 + 2 < nk:
                seq.append(("K", t2 + 2))
            if t2 + 3 < nk:
                seq.append(("K", t2 + 3))
            seq.append(("V", t2))
            if t2 + 1 < nk:
                seq.append(("V", t2 + 1))
        return seq

    # ---- roles (generators: each yield is a point where another role may run)
    def producer(self):
        pos = 0
        for k, (na, nb) in enumerate(self.units):
            nk = na + nb
            while not (k == 0 or self.ready("QE", k)):
                yield
            self.tma.append(("QF", ("q", 0), (k, "a")))
            if nb > 0:
                self.tma.append(("QF", ("q", 1), (k, "b")))
            self.q_pending = 2 if nb > 0 else 1
            yield
            for kind, j in self.ring(nk):
                s = pos % self.stages
                while not (pos < self.stages or self.ready(("KE", s), pos // self.stages)):
                    yield
                self.tma.append((("KF", s), ("slot", s), (k, kind, j)))
                pos += 1
                yield

    def mma(self):
        pos = 0
        merges = selfs = 0
        reader = 0  # of the last accumulation into O1: 1 merge, 2 warpgroup 1's own store
        pc = [0, 0]
        tiles = [0, 0]
        for k, (na, nb) in enumerate(self.units):
            nk, n0, n1 = self.split(na, nb)
            while not self.ready("QF", k + 1):
                yield
            s_left = [nk]

            def q_of(w, u):
                return 1 if (w == 1 and u < nb) else 0

            def issue_s(w, u, s, j):
                self.pipe.append(("S", (k, w, u, s, j, q_of(w, u))))
                self.pipe.append(("commit", ("SF", w)))
                s_left[0] -= 1
                if s_left[0] == 0:
                    self.pipe.append(("commit", "QE"))
                self.pipe.append(("commit", ("KE", s)))

            for j in range(min(nk, 2)):  # S_0 of position 0, S_1 of position 1
                s = pos % self.stages
                while not self.ready(("KF", s), pos // self.stages + 1):
                    yield
                issue_s(j, 0, s, j)
                pos += 1
                yield
            for t2 in range(0, nk, 2):
                u = t2 >> 1
                for w in range(2):
                    if t2 + 2 + w < nk:
                        while not self.ready(("SFree", w), tiles[w] + u + 1):
                            yield
                        s = pos % self.stages
                        while not self.ready(("KF", s), pos // self.stages + 1):
                            yield
                        issue_s(w, u + 1, s, t2 + 2 + w)
                        pos += 1
                        yield
                for w in range(2):
                    if t2 + w < nk:
                        s = pos % self.stages
                        while not self.ready(("KF", s), pos // self.stages + 1):
                            yield
                        b_end = w == 1 and u == nb - 1
                        start = u == 0 or (w == 1 and nb > 0 and u == nb)
                        if w == 1 and start:
                            if reader == 1:
                                while not self.ready("O1Free", merges):
                                    yield
                            if reader == 2:
                                while not self.ready("O1Self", selfs):
                                    yield
                            if u < nb:
                                selfs, reader = selfs + 1, 2
                            else:
                                merges, reader = merges + 1, 1
                        while not self.ready(("PF", w), pc[w] + 1):
                            yield
                        pc[w] += 1
                        tag = (k, w, "b" if (w == 1 and u < nb) else "a")
                        self.pipe.append(("PV", (k, w, u, s, t2 + w, not start, tag)))
                        self.pipe.append(("commit", ("PVD", w)))
                        if b_end:
                            self.pipe.append(("commit", "OFB"))
                        elif u == (n1 if w else n0) - 1:
                            self.pipe.append(("commit", ("OF", w)))
                        self.pipe.append(("commit", ("KE", s)))
                        pos += 1
                        yield
            tiles[0] += n0
            tiles[1] += n1

    def softmax(self, w):
        scnt = p_sent = 0
        ocnt = o1cnt = mcnt = 0
        for k, (na, nb) in enumerate(self.units):
            nk, n0, n1 = self.split(na, nb)
            n_mine = n1 if w else n0
            if n_mine == 0:
                continue
            two = w == 1 and nb > 0
            segs = [(True, 0, nb)] + ([(False, nb, n1)] if n1 > nb else []) if two else [(False, 0, n_mine)]
            for own_b, u0, u1 in segs:
                for u in range(u0, u1):
                    while not self.ready(("SF", w), scnt + 1):
                        yield
                    scnt += 1
                    assert self.S[w] == ("S", k, w, u), ("S", self.S[w], (k, w, u))
                    self.S[w] = ("read", k, w, u)
                    self.B[("SFree", w)].complete()
                    yield
                    if p_sent > 0:
                        while not self.ready(("PVD", w), p_sent):
                            yield
                    if u > u0:
                        # the in-place O rescale may run here: every earlier PV of the
                        # accumulation has completed
                        o = self.O[w]
                        tag = (k, w, "b" if own_b else "a")
                        assert o is not None and o["tag"] == tag and o["n"] == u - u0, ("rescale", o, tag, u)
                    assert self.P[w] is None or self.P[w][0] == "used", ("P overwritten", self.P[w], (k, w, u))
                    self.P[w] = ("P", k, w, u)
                    self.B[("PF", w)].complete()
                    p_sent += 1
                    yield
                if w == 1 and not own_b:
                    # (m, l) of warpgroup 1's part of a, for warpgroup 0's merge
                    if mcnt > 0:
                        while not self.ready("O1Free", mcnt):
                            yield
                    mcnt += 1
                    self.stats = k
                    self.B["ST"].complete()
                    yield
                    continue
                # epilogue: warpgroup 0 for a (merging warpgroup 1's part), or warpgroup 1 for b
                done = "OFB" if own_b else ("OF", w)
                while not self.ready(done, ocnt + 1):
                    yield
                ocnt += 1
                merge = w == 0 and n1 > nb
                if merge:
                    while not self.ready(("OF", 1), o1cnt + 1):
                        yield
                    while not self.ready("ST", mcnt + 1):
                        yield
                    o1cnt += 1
                    mcnt += 1
                    assert self.stats == k, ("stats", self.stats, k)
                    o1 = self.O[1]
                    assert o1["tag"] == (k, 1, "a") and o1["n"] == n1 - nb, ("O1 for the merge", o1, k)
                own = self.O[w]
                want = (k, w, "b") if own_b else (k, w, "a")
                assert own["tag"] == want and own["n"] == (nb if own_b else n_mine - (nb if w else 0)), (own, want)
                yield
                own["read"] = True
                if merge:
                    self.O[1]["read"] = True
                    self.B["O1Free"].complete()
                if own_b:
                    self.B["O1Self"].complete()
                yield

    def tensor_pipe(self):
        while True:
            if not self.pipe:
                yield
                continue
            op, x = self.pipe.pop(0)
            if op == "commit":
                self.B[x].complete()
            elif op == "S":
                k, w, u, s, j, qb = x
                assert self.slot.get(s) == (k, "K", j), ("K slot", self.slot.get(s), x)
                na, nb = self.units[k]
                item, _ = self.tile(na, nb, w, u)
                assert self.q.get(qb) == (k, item), ("Q", self.q.get(qb), (k, item), x)
                assert self.S[w] is None or self.S[w][0] == "read", ("S overwritten before read", self.S[w], x)
                self.S[w] = ("S", k, w, u)
            else:
                k, w, u, s, j, acc, tag = x
                assert self.slot.get(s) == (k, "V", j), ("V slot", self.slot.get(s), x)
                assert self.P[w] == ("P", k, w, u), ("P", self.P[w], x)
                self.P[w] = ("used",)
                o = self.O[w]
                if acc:
                    assert o is not None and o["tag"] == tag and not o["read"], ("accumulate", o, x)
                    o["n"] += 1
                else:
                    assert o is None or o["read"], ("accumulator overwritten before read", o, x)
                    self.O[w] = {"tag": tag, "n": 1, "read": False}
            yield

    def copy_engine(self):
        while True:
            if not self.tma:
                yield
                continue
            i = self.rnd.randrange(len(self.tma))
            bar, (kind, idx), val = self.tma.pop(i)
            if kind == "q":
                self.q[idx] = val
                self.q_pending -= 1
                if self.q_pending == 0:
                    self.B[bar].complete()
            else:
                self.slot[idx] = val
                self.B[bar].complete()
            yield

    def run(self, max_steps=400000):
        roles = {"producer": self.producer(), "mma": self.mma(), "wg0": self.softmax(0), "wg1": self.softmax(1)}
        engines = [self.tensor_pipe(), self.copy_engine()]
        live = dict(roles)
        for _ in range(max_steps):
            if not live and not self.pipe and not self.tma:
                return
            g = self.rnd.choice(list(live.values()) + engines)
            try:
                next(g)
            except StopIteration:
                live = {n: r for n, r in live.items() if r is not g}
        raise AssertionError("deadlock or too slow: still running %s" % sorted(live))


def check_final(m):
    # every accumulator was read by its reader at the end
    for w in range(2):
        assert m.O[w] is None or m.O[w]["read"], ("unread accumulator", w, m.O[w])


def random_units(rnd, pair_prob):
    units = []
    for _ in range(rnd.randint(1, 4)):
        na = rnd.randint(1, 10)
        nb = rnd.randint(1, na) if rnd.random() < pair_prob else 0
        units.append((na, nb))
    return units


@pytest.mark.parametrize("stages", [2, 3, 8, 9])
def test_random_unit_sequences_and_interleavings(stages):
    rnd = random.Random(1000 + stages)
    for trial in range(250):
        units = random_units(rnd, 0.6)
        m = Model(units, stages, seed=rnd.randrange(1 << 30))
        m.run()
        check_final(m)


def test_every_pair_shape_of_the_prefill_workload():
    # all (na, nb) with 1 <= nb <= na <= 12, each alone (one unit per paired CTA) and after an
    # unpaired unit (phase counters that start past zero)
    for na in range(1, 13):
        for nb in range(0, na + 1):
            for units in ([(na, nb)], [(3, 0), (na, nb)], [(na, nb), (na, nb)]):
                for seed in range(3):
                    m = Model(units, 8, seed=na * 1000 + nb * 10 + seed)
                    m.run()
                    check_final(m)


class Dropped(Model):
    """The model with the waits on some barriers removed (they always pass)."""

    drop = ()

    def ready(self, name, c):
        if name in self.drop:
            return True
        return super().ready(name, c)


@pytest.mark.parametrize("drop,units,stages", [
    (("SFree", 0), [(8, 0)], 3),         # the next S would overwrite S before its read
    (("PVD", 1), [(7, 1)], 3),           # P overwritten before its PV read it
    (("KE", 1), [(9, 3)], 3),            # a ring stage refilled before its MMA read it
    ("QE", [(1, 0), (4, 2)], 8),         # the next Q loaded under the previous S (a short unit:
                                         # no ring wait of its own orders the load after its S)
    ("OFB", [(6, 2)], 3),                # b stored before its last PV
    (("OF", 0), [(4, 4)], 3),            # a stored before warpgroup 0's last PV (no merge, whose
                                         # wait for warpgroup 1's later PV would cover it)
    ("ST", [(6, 2)], 3),                 # merged before warpgroup 1's (m, l) arrived
])
def test_model_catches_each_missing_wait(drop, units, stages):
    # the checks have teeth: without any one of these waits some interleaving breaks
    failures = 0
    for seed in range(300):
        m = type("M", (Dropped,), {"drop": (drop,)})(units, stages, seed=seed)
        try:
            m.run()
            check_final(m)
        except AssertionError:
            failures += 1
    assert failures > 0, drop


def test_o1_waits_are_implied_by_the_issue_order():
    # With one MMA issuer, warpgroup 0's PV of a round is issued before warpgroup 1's, and
    # each warpgroup hands over the P of a new accumulation only after its own reads of the
    # previous one (warpgroup 0's merge, warpgroup 1's store of b), so the MMA warp's waits
    # for those reads (kO1Free, kO1Self) never block here. They are kept: an issuer per
    # warpgroup would depend on them.
    for seed in range(150):
        m = type("M", (Dropped,), {"drop": ("O1Free", "O1Self")})([(6, 0), (5, 2), (7, 1), (4, 0)], 3, seed=seed)
        m.run()
        check_final(m)


# ---- the same protocol with one MMA issuer per warpgroup (a form not built: the next step for
# the paired form, whose warpgroup 1 then no longer holds up warpgroup 0's PVs). Both issuers
# walk every ring position in the producer's order and release each (a commit where they used
# it, a plain arrive where not); a stage is free once both released it, and Q once both issued
# their last S. Each issuer has its own in-order tensor queue: a commit covers only the MMAs
# of the warp that issued it.

class CBar:
    """A barrier that completes a phase after `count` arrivals."""

    def __init__(self, name, count):
        self.name, self.count, self.pend, self.done = name, count, 0, 0

    def complete(self):  # one arrival
        self.pend += 1
        assert self.pend <= self.count, self.name
        if self.pend == self.count:
            self.pend = 0
            self.done += 1


class Dual(Model):
    """The protocol with an MMA issuer per warpgroup."""

    def __init__(self, units, stages, seed):
        super().__init__(units, stages, seed)
        for s in range(stages):
            self.B[("KE", s)] = CBar(("KE", s), 2)
        self.B["QE"] = CBar("QE", 2)
        self.pipes = {0: [], 1: []}

    def issuer(self, w):
        pos = 0
        merges = selfs = 0
        reader = 0
        pc = 0
        tiles_w = 0
        for k, (na, nb) in enumerate(self.units):
            nk, n0, n1 = self.split(na, nb)
            n_w = n1 if w else n0
            while not self.ready("QF", k + 1):
                yield
            s_left = [n_w]
            if n_w == 0:
                self.B["QE"].complete()
            pipe = self.pipes[w]
            for kind, j in self.ring(nk):
                s = pos % self.stages
                while not self.ready(("KF", s), pos // self.stages + 1):
                    yield
                pos += 1
                u, mine = j >> 1, (j & 1) == w
                if not mine:
                    self.B[("KE", s)].complete()  # plain arrive
                    yield
                    continue
                if kind == "K":
                    if u > 0:
                        while not self.ready(("SFree", w), tiles_w + u):
                            yield
                    qb = 1 if (w == 1 and u < nb) else 0
                    pipe.append(("S", (k, w, u, s, j, qb)))
                    pipe.append(("commit", ("SF", w)))
                    s_left[0] -= 1
                    if s_left[0] == 0:
                        pipe.append(("commit", "QE"))
                    pipe.append(("commit", ("KE", s)))
                else:
                    start = u == 0 or (w == 1 and nb > 0 and u == nb)
                    if w == 1 and start:
                        if reader == 1:
                            while not self.ready("O1Free", merges):
                                yield
                        if reader == 2:
                            while not self.ready("O1Self", selfs):
                                yield
                        if u < nb:
                            selfs, reader = selfs + 1, 2
                        else:
                            merges, reader = merges + 1, 1
                    while not self.ready(("PF", w), pc + 1):
                        yield
                    pc += 1
                    tag = (k, w, "b" if (w == 1 and u < nb) else "a")
                    pipe.append(("PV", (k, w, u, s, j, not start, tag)))
                    pipe.append(("commit", ("PVD", w)))
                    if w == 1 and u == nb - 1:
                        pipe.append(("commit", "OFB"))
                    elif u == n_w - 1:
                        pipe.append(("commit", ("OF", w)))
                    pipe.append(("commit", ("KE", s)))
                yield
            tiles_w += n_w

    def tensor_pipe_w(self, w):
        while True:
            self.pipe = self.pipes[w]
            if not self.pipe:
                yield
                continue
            g = super().tensor_pipe()
            next(g)  # executes one op of self.pipe
            yield

    def run(self, max_steps=600000):
        roles = {"producer": self.producer(), "mma0": self.issuer(0), "mma1": self.issuer(1),
                 "wg0": self.softmax(0), "wg1": self.softmax(1)}
        engines = [self.tensor_pipe_w(0), self.tensor_pipe_w(1), self.copy_engine()]
        live = dict(roles)
        for _ in range(max_steps):
            if not live and not self.pipes[0] and not self.pipes[1] and not self.tma:
                return
            g = self.rnd.choice(list(live.values()) + engines)
            try:
                next(g)
            except StopIteration:
                live = {n: r for n, r in live.items() if r is not g}
        raise AssertionError("deadlock: %s" % sorted(live))




def test_two_issuer_form_of_the_protocol():
    rnd = random.Random(7)
    for stages in (2, 3, 8):
        for _ in range(120):
            m = Dual(random_units(rnd, 0.7), stages, seed=rnd.randrange(1 << 30))
            m.run()
            check_final(m)


def test_two_issuer_form_needs_the_o1_waits():
    class NoO1(Dual):
        def ready(self, name, c):
            if name in ("O1Free", "O1Self"):
                return True
            return super().ready(name, c)

    failures = 0
    for seed in range(300):
        try:
            m = NoO1([(6, 0), (5, 2), (7, 1)], 8, seed=seed)
            m.run()
            check_final(m)
        except AssertionError:
            failures += 1
    assert failures > 0
