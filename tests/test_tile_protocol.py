"""Discrete-event models of the kernel's other MMA protocols (host only, no GPU): the forms not
covered by the split-K model at D = 64 (test_pair_protocol.py).

* two query tiles per item, D = 128: one MMA issuer, P written over S's TMEM columns, each V
  tile released right after its last PV (not after the S that follows);
* two query tiles per item, D = 64: an MMA issuer per warpgroup, separate P columns, both
  issuers walking every ring position and releasing each (a stage is free once both did);
* one query tile per item, D = 128: one issuer, P over S's columns, tiles alternating between
  the warpgroups and warpgroup 0 merging warpgroup 1's part;
* the fp32-I/O kernel: separate K and V rings, V transposer warps filling transposed-V
  buffers for the PV, and Q copied into TMEM by the MMA warp before the item's S products.

Each model follows the kernel's issue order, ring order and waits. Over random item sequences
and interleavings (copies land in any order; each issuer's tensor queue runs in its order) every
role must finish, every parity wait must find its barrier at the awaited phase or the one
before, and no buffer may be overwritten before its reader is done: ring slots, Q tiles, S, P
(in S's columns or its own), the O accumulators (including the softmax warpgroup's in-place
rescale of O, which needs every earlier PV of the accumulation complete).
"""

from __future__ import annotations

import random

import pytest


class Bar:
    def __init__(self, name, count=1):
        self.name, self.count, self.pend, self.done = name, count, 0, 0

    def arrive(self):
        self.pend += 1
        assert self.pend <= self.count, self.name
        if self.pend == self.count:
            self.pend = 0
            self.done += 1


class Base:
    """Shared state, the copy engine, the tensor queues and the scheduler."""

    issuers = 1
    sep_p = True

    def __init__(self, items, stages, seed):
        self.items, self.stages = items, stages
        self.rnd = random.Random(seed)
        self.B = {}
        for n in ["QF", "ST", "O1Free"]:
            self.B[n] = Bar(n)
        self.B["QE"] = Bar("QE", self.issuers)
        for s in range(stages):
            self.B[("KF", s)], self.B[("KE", s)] = Bar(("KF", s)), Bar(("KE", s), self.issuers)
        for w in range(2):
            for n in ["SF", "SFree", "PF", "PVD", "OF"]:
                self.B[(n, w)] = Bar((n, w))
        self.queues = {i: [] for i in range(self.issuers)}
        self.tma = []
        self.q, self.slot = {}, {}
        self.cols = {0: None, 1: None}   # S, or P written over it (P in S's columns)
        self.P = {0: None, 1: None}      # separate P columns
        self.O = {0: None, 1: None}
        self.stats = None
        self.q_pending = 0

    def ready(self, name, c):
        d = self.B[name].done
        assert c - 1 <= d <= c, ("phase", name, "waits for", c, "done", d)
        return d == c

    def load(self, bar, buf, val):
        self.tma.append((bar, buf, val))

    def copy_engine(self):
        while True:
            if self.tma:
                bar, (kind, idx), val = self.tma.pop(self.rnd.randrange(len(self.tma)))
                if kind == "q":
                    self.q[idx] = val
                    self.q_pending -= 1
                    if self.q_pending == 0:
                        self.B[bar].arrive()
                else:
                    self.slot[idx] = val
                    self.B[bar].arrive()
            yield

    def tensor(self, i):
        while True:
            qu = self.queues[i]
            if qu:
                op, x = qu.pop(0)
                if op == "commit":
                    self.B[x].arrive()
                elif op == "S":
                    self.exec_s(*x)
                else:
                    self.exec_pv(*x)
            yield

    def exec_s(self, k, w, u, s, j, qb, qval):
        assert self.slot.get(s) == (k, "K", j), ("K slot", self.slot.get(s), (k, j))
        assert self.q.get(qb) == qval, ("Q", self.q.get(qb), qval)
        cur = self.cols[w]
        if self.sep_p:
            assert cur is None or cur[0] == "read", ("S overwritten before read", cur)
        else:
            assert cur is None or cur[0] == "P used", ("S over a P not yet read", cur)
        self.cols[w] = ("S", k, w, u)

    def exec_pv(self, k, w, u, s, j, acc, tag):
        assert self.slot.get(s) == (k, "V", j), ("V slot", self.slot.get(s), (k, j))
        if self.sep_p:
            assert self.P[w] == ("P", k, w, u), ("P", self.P[w], (k, w, u))
            self.P[w] = ("used",)
        else:
            assert self.cols[w] == ("P", k, w, u), ("P", self.cols[w], (k, w, u))
            self.cols[w] = ("P used",)
        o = self.O[w]
        if acc:
            assert o is not None and o["tag"] == tag and not o["read"], ("accumulate", o, tag)
            o["n"] += 1
        else:
            assert o is None or o["read"], ("accumulator overwritten before read", o, tag)
            self.O[w] = {"tag": tag, "n": 1, "read": False}

    # softmax helpers
    def read_s(self, w, k, u):
        assert self.cols[w] == ("S", k, w, u), ("S", self.cols[w], (k, w, u))
        self.cols[w] = ("read", k, w, u)

    def write_p(self, w, k, u, tag, first):
        # the in-place O rescale may run here: every earlier PV of the accumulation is complete
        if not first:
            o = self.O[w]
            assert o is not None and o["tag"] == tag and o["n"] == u - first_u(self, w, k, u), ("rescale", o, u)
        if self.sep_p:
            assert self.P[w] is None or self.P[w][0] == "used", ("P overwritten", self.P[w])
            self.P[w] = ("P", k, w, u)
        else:
            assert self.cols[w] == ("read", k, w, u), ("P over S before its read", self.cols[w])
            self.cols[w] = ("P", k, w, u)

    def run(self, max_steps=600000):
        live = {n: g for n, g in self.roles().items()}
        engines = [self.tensor(i) for i in range(self.issuers)] + [self.copy_engine()]
        for _ in range(max_steps):
            if not live and not any(self.queues.values()) and not self.tma:
                for w in range(2):
                    assert self.O[w] is None or self.O[w]["read"], ("unread accumulator", w)
                return
            g = self.rnd.choice(list(live.values()) + engines)
            try:
                next(g)
            except StopIteration:
                live = {n: r for n, r in live.items() if r is not g}
        raise AssertionError("deadlock: %s" % sorted(live))


def first_u(model, w, k, u):
    return 0  # every accumulation in these forms starts at the warpgroup's first tile


# ---------------------------------------------------------------- two query tiles per item
class TwoTile(Base):
    """items: (n0, n1) with n1 in {0, n0, n0 + 1} (n1 = 0: the second query tile is past N)."""

    def producer(self):
        pos = 0
        for k, (n0, n1) in enumerate(self.items):
            nk = max(n0, n1)
            while not (k == 0 or self.ready("QE", k)):
                yield
            nq = 2 if n1 > 0 else 1
            self.q_pending = nq
            for i in range(nq):
                self.load("QF", ("q", i), (k, i))
            yield
            order = [("K", 0)]
            if self.sep_p:   # K0, then per j: K(j+1), V(j)
                for j in range(nk):
                    if j + 1 < nk:
                        order.append(("K", j + 1))
                    order.append(("V", j))
            else:            # K0 V0 K1 V1 ...
                order = []
                for j in range(nk):
                    order += [("K", j), ("V", j)]
            for kind, j in order:
                s = pos % self.stages
                while not (pos < self.stages or self.ready(("KE", s), pos // self.stages)):
                    yield
                self.load(("KF", s), ("slot", s), (k, kind, j))
                pos += 1
                yield


class TwoTileD128(TwoTile):
    """One issuer, P over S's columns; V_j released right after its last PV."""

    sep_p = False

    def roles(self):
        return {"producer": self.producer(), "mma": self.mma(), "wg0": self.softmax(0), "wg1": self.softmax(1)}

    def mma(self):
        pos = 0
        pc = [0, 0]
        qu = self.queues[0]
        for k, (n0, n1) in enumerate(self.items):
            nk = max(n0, n1)
            while not self.ready("QF", k + 1):
                yield
            s_left = [n0 + n1]

            def issue_s(w, u, s):
                qu.append(("S", (k, w, u, s, u, w, (k, w))))
                qu.append(("commit", ("SF", w)))
                s_left[0] -= 1
                if s_left[0] == 0:
                    qu.append(("commit", "QE"))

            def slot():
                nonlocal pos
                s = pos % self.stages
                return s

            s = slot()
            while not self.ready(("KF", s), pos // self.stages + 1):
                yield
            pos += 1
            issue_s(0, 0, s)
            if n1 > 0:
                issue_s(1, 0, s)
            qu.append(("commit", ("KE", s)))
            yield
            for j in range(nk):
                sv = slot()
                while not self.ready(("KF", sv), pos // self.stages + 1):
                    yield
                pos += 1
                k_next, sk = False, None
                for w in range(2):
                    nw = n1 if w else n0
                    if j < nw:
                        while not self.ready(("PF", w), pc[w] + 1):
                            yield
                        pc[w] += 1
                        qu.append(("PV", (k, w, j, sv, j, j > 0, (k, w))))
                        if j == nw - 1:
                            qu.append(("commit", ("OF", w)))
                    if (j < n1) if w == 1 else (j >= n1):
                        qu.append(("commit", ("KE", sv)))  # V_j after its last PV
                    if j + 1 < nw:
                        if not k_next:
                            sk = slot()
                            while not self.ready(("KF", sk), pos // self.stages + 1):
                                yield
                            pos += 1
                            k_next = True
                        issue_s(w, j + 1, sk)
                    yield
                if k_next:
                    qu.append(("commit", ("KE", sk)))

    def softmax(self, w):
        scnt = ocnt = 0
        for k, (n0, n1) in enumerate(self.items):
            nw = n1 if w else n0
            for u in range(nw):
                while not self.ready(("SF", w), scnt + 1):
                    yield
                scnt += 1
                self.read_s(w, k, u)
                yield
                self.write_p(w, k, u, (k, w), u == 0)
                self.B[("PF", w)].arrive()
                yield
            if nw == 0:
                continue
            while not self.ready(("OF", w), ocnt + 1):
                yield
            ocnt += 1
            o = self.O[w]
            assert o["tag"] == (k, w) and o["n"] == nw, ("epilogue", o, (k, w, nw))
            yield
            o["read"] = True


class TwoTileD64Dual(TwoTile):
    """An issuer per warpgroup, separate P; each walks every position and releases each."""

    issuers = 2
    sep_p = True

    def roles(self):
        return {"producer": self.producer(), "mma0": self.issuer(0), "mma1": self.issuer(1),
                "wg0": self.softmax(0), "wg1": self.softmax(1)}

    def issuer(self, w):
        pos = 0
        pc = tiles = 0
        qu = self.queues[w]
        for k, (n0, n1) in enumerate(self.items):
            nk = max(n0, n1)
            nw = n1 if w else n0
            while not self.ready("QF", k + 1):
                yield
            s_left = [nw]
            if nw == 0:
                self.B["QE"].arrive()
            order = [("K", 0)]
            for j in range(nk):
                if j + 1 < nk:
                    order.append(("K", j + 1))
                order.append(("V", j))
            for kind, j in order:
                s = pos % self.stages
                while not self.ready(("KF", s), pos // self.stages + 1):
                    yield
                pos += 1
                if j >= nw:
                    self.B[("KE", s)].arrive()  # a position this warpgroup does not use
                    yield
                    continue
                if kind == "K":
                    if j > 0:
                        while not self.ready(("SFree", w), tiles + j):
                            yield
                    qu.append(("S", (k, w, j, s, j, w, (k, w))))
                    qu.append(("commit", ("SF", w)))
                    s_left[0] -= 1
                    if s_left[0] == 0:
                        qu.append(("commit", "QE"))
                else:
                    while not self.ready(("PF", w), pc + 1):
                        yield
                    pc += 1
                    qu.append(("PV", (k, w, j, s, j, j > 0, (k, w))))
                    qu.append(("commit", ("PVD", w)))
                    if j == nw - 1:
                        qu.append(("commit", ("OF", w)))
                qu.append(("commit", ("KE", s)))
                yield
            tiles += nw

    def softmax(self, w):
        scnt = ocnt = p_sent = 0
        for k, (n0, n1) in enumerate(self.items):
            nw = n1 if w else n0
            for u in range(nw):
                while not self.ready(("SF", w), scnt + 1):
                    yield
                scnt += 1
                self.read_s(w, k, u)
                self.B[("SFree", w)].arrive()
                yield
                if p_sent > 0:
                    while not self.ready(("PVD", w), p_sent):
                        yield
                self.write_p(w, k, u, (k, w), u == 0)
                self.B[("PF", w)].arrive()
                p_sent += 1
                yield
            if nw == 0:
                continue
            while not self.ready(("OF", w), ocnt + 1):
                yield
            ocnt += 1
            o = self.O[w]
            assert o["tag"] == (k, w) and o["n"] == nw, ("epilogue", o, (k, w, nw))
            yield
            o["read"] = True


# ---------------------------------------------------------------- one query tile, D = 128
class SplitKD128(Base):
    """items: nk; tile j belongs to warpgroup j & 1; warpgroup 0 merges."""

    sep_p = False

    def roles(self):
        return {"producer": self.producer(), "mma": self.mma(), "wg0": self.softmax(0), "wg1": self.softmax(1)}

    def producer(self):
        pos = 0
        for k, nk in enumerate(self.items):
            while not (k == 0 or self.ready("QE", k)):
                yield
            self.q_pending = 1
            self.load("QF", ("q", 0), (k, 0))
            yield
            order = [("K", 0)]
            for j in range(nk):
                if j + 1 < nk:
                    order.append(("K", j + 1))
                order.append(("V", j))
            for kind, j in order:
                s = pos % self.stages
                while not (pos < self.stages or self.ready(("KE", s), pos // self.stages)):
                    yield
                self.load(("KF", s), ("slot", s), (k, kind, j))
                pos += 1
                yield

    def mma(self):
        pos = 0
        pc = [0, 0]
        merges = 0
        qu = self.queues[0]
        for k, nk in enumerate(self.items):
            n1 = nk // 2
            while not self.ready("QF", k + 1):
                yield
            s_left = [nk]

            def take():
                nonlocal pos
                s = pos % self.stages
                c = pos // self.stages + 1
                pos += 1
                return s, c

            def issue_s(w, u, s, j):
                qu.append(("S", (k, w, u, s, j, 0, (k, 0))))
                qu.append(("commit", ("SF", w)))
                s_left[0] -= 1
                if s_left[0] == 0:
                    qu.append(("commit", "QE"))
                qu.append(("commit", ("KE", s)))

            for j in range(min(nk, 2)):
                s, c = take()
                while not self.ready(("KF", s), c):
                    yield
                issue_s(j, 0, s, j)
                yield
            for j in range(nk):
                w, u = j & 1, j >> 1
                sv, c = take()
                while not self.ready(("KF", sv), c):
                    yield
                if j == 1 and merges > 0:
                    while not self.ready("O1Free", merges):
                        yield
                while not self.ready(("PF", w), pc[w] + 1):
                    yield
                pc[w] += 1
                qu.append(("PV", (k, w, u, sv, j, j >= 2, (k, w))))
                if j + 2 >= nk:
                    qu.append(("commit", ("OF", w)))
                qu.append(("commit", ("KE", sv)))
                yield
                if j + 2 < nk:
                    sk, c = take()
                    while not self.ready(("KF", sk), c):
                        yield
                    issue_s(w, u + 1, sk, j + 2)
                    yield
            if n1 > 0:
                merges += 1

    def softmax(self, w):
        scnt = ocnt = o1cnt = mcnt = 0
        for k, nk in enumerate(self.items):
            n0, n1 = (nk + 1) // 2, nk // 2
            nw = n1 if w else n0
            if nw == 0:
                continue
            for u in range(nw):
                while not self.ready(("SF", w), scnt + 1):
                    yield
                scnt += 1
                self.read_s(w, k, u)
                yield
                self.write_p(w, k, u, (k, w), u == 0)
                self.B[("PF", w)].arrive()
                yield
            if w == 1:
                if mcnt > 0:
                    while not self.ready("O1Free", mcnt):
                        yield
                for _ in range(self.rnd.randint(0, 3)):  # the warpgroup may be slow to get here
                    yield
                mcnt += 1
                self.stats = k
                self.B["ST"].arrive()
                yield
                continue
            while not self.ready(("OF", 0), ocnt + 1):
                yield
            ocnt += 1
            if n1 > 0:
                while not self.ready(("OF", 1), o1cnt + 1):
                    yield
                while not self.ready("ST", mcnt + 1):
                    yield
                o1cnt += 1
                mcnt += 1
                assert self.stats == k
                assert self.O[1]["tag"] == (k, 1) and self.O[1]["n"] == n1, ("O1 for the merge", self.O[1])
            assert self.O[0]["tag"] == (k, 0) and self.O[0]["n"] == n0, ("O0", self.O[0])
            yield
            self.O[0]["read"] = True
            if n1 > 0:
                self.O[1]["read"] = True
                self.B["O1Free"].arrive()
            yield


def two_tile_items(rnd, causal):
    out = []
    for _ in range(rnd.randint(1, 4)):
        n = rnd.randint(1, 9)
        if causal:
            out.append(rnd.choice([(n, n + 1), (n, 0), (n, n)]))
        else:
            out.append((n, n) if rnd.random() < 0.8 else (n, 0))
    return out


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_two_tile_d128_single_issuer(stages):
    rnd = random.Random(50 + stages)
    for _ in range(200):
        m = TwoTileD128(two_tile_items(rnd, rnd.random() < 0.5), stages, seed=rnd.randrange(1 << 30))
        m.run()


@pytest.mark.parametrize("stages", [2, 3, 8])
def test_two_tile_d64_two_issuers(stages):
    rnd = random.Random(60 + stages)
    for _ in range(200):
        m = TwoTileD64Dual(two_tile_items(rnd, rnd.random() < 0.5), stages, seed=rnd.randrange(1 << 30))
        m.run()


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_split_k_d128_single_issuer(stages):
    rnd = random.Random(70 + stages)
    for _ in range(200):
        items = [rnd.randint(1, 11) for _ in range(rnd.randint(1, 4))]
        m = SplitKD128(items, stages, seed=rnd.randrange(1 << 30))
        m.run()


class _Drop:
    drop = ()

    def ready(self, name, c):
        if name in self.drop:
            return True
        return super().ready(name, c)


@pytest.mark.parametrize("cls,drop,items,stages", [
    (TwoTileD128, ("PF", 1), [(4, 5)], 3),        # PV before its P
    (TwoTileD128, ("KE", 0), [(5, 5), (3, 4)], 2),  # a ring stage refilled under its reader
    (TwoTileD128, ("OF", 0), [(3, 3), (2, 3)], 3),  # O read before its last PV
    (TwoTileD64Dual, ("SFree", 1), [(5, 6)], 3),  # the next S over an unread S
    (TwoTileD64Dual, ("PVD", 0), [(6, 6)], 3),    # P overwritten under its PV
    (TwoTileD64Dual, "QE", [(1, 2), (3, 4)], 8),  # next Q under the previous S
    (SplitKD128, "ST", [4], 3),                   # merge before warpgroup 1's (m, l)
    (SplitKD128, ("OF", 1), [4], 3),              # merge before warpgroup 1's last PV (an even
                                                  # count: warpgroup 1's PV is the item's last)
])
def test_models_catch_each_missing_wait(cls, drop, items, stages):
    M = type("M", (_Drop, cls), {"drop": (drop,)})
    failures = 0
    for seed in range(300):
        try:
            M(items, stages, seed=seed).run()
        except AssertionError:
            failures += 1
    assert failures > 0, (cls.__name__, drop)


def test_split_k_d128_o1_wait_is_implied_by_the_issue_order():
    # As at D = 64: with one issuer, warpgroup 0's first PV of an item precedes warpgroup 1's,
    # and warpgroup 0 hands over that P only after its merge of the previous item has read O1.
    M = type("M", (_Drop, SplitKD128), {"drop": ("O1Free",)})
    for seed in range(150):
        M([4, 5, 3, 6], 3, seed=seed).run()


# ---------------------------------------------------------------- fp32 I/O kernel
class SplitKF32(Base):
    """The fp32 kernel: one query tile per item, 64-key tiles alternating between the
    warpgroups; separate K and V rings; two transposer warps copy each V tile into a
    transposed buffer (Vt) that the PV reads; Q is copied from its shared-memory tile into TMEM
    by the MMA warp (in issue order, after the previous item's last S) and S reads it there."""

    sep_p = False

    def __init__(self, items, stages, seed):
        self.kst, self.vst, self.nvt = stages
        super().__init__(items, self.kst, seed)
        for s in range(self.vst):
            self.B[("VF", s)], self.B[("VE", s)] = Bar(("VF", s)), Bar(("VE", s))
        for b in range(self.nvt):
            self.B[("VtF", b)], self.B[("VtE", b)] = Bar(("VtF", b)), Bar(("VtE", b))
        self.vslot, self.vt = {}, {}
        self.q_tmem = None

    def roles(self):
        return {"producer": self.producer(), "mma": self.mma(), "tr": self.transposer(),
                "wg0": self.softmax(0), "wg1": self.softmax(1)}

    def producer(self):
        kpos = vpos = 0
        for k, nk in enumerate(self.items):
            while not (k == 0 or self.ready("QE", k)):
                yield
            self.q_pending = 1
            self.load("QF", ("q", 0), (k, 0))
            yield
            order = [("K", 0)]
            for j in range(nk):
                if j + 1 < nk:
                    order.append(("K", j + 1))
                order.append(("V", j))
            for kind, j in order:
                if kind == "K":
                    s = kpos % self.kst
                    while not (kpos < self.kst or self.ready(("KE", s), kpos // self.kst)):
                        yield
                    self.load(("KF", s), ("slot", s), (k, "K", j))
                    kpos += 1
                else:
                    s = vpos % self.vst
                    while not (vpos < self.vst or self.ready(("VE", s), vpos // self.vst)):
                        yield
                    self.load(("VF", s), ("vslot", s), (k, "V", j))
                    vpos += 1
                yield

    def copy_engine(self):
        while True:
            if self.tma:
                bar, (kind, idx), val = self.tma.pop(self.rnd.randrange(len(self.tma)))
                if kind == "q":
                    self.q[idx] = val
                    self.q_pending -= 1
                    if self.q_pending == 0:
                        self.B[bar].arrive()
                else:
                    (self.vslot if kind == "vslot" else self.slot)[idx] = val
                    self.B[bar].arrive()
            yield

    def transposer(self):
        vpos = vtc = 0
        for k, nk in enumerate(self.items):
            for j in range(nk):
                s, b = vpos % self.vst, vtc % self.nvt
                while not self.ready(("VF", s), vpos // self.vst + 1):
                    yield
                while not (vtc < self.nvt or self.ready(("VtE", b), vtc // self.nvt)):
                    yield
                vpos += 1
                vtc += 1
                assert self.vslot.get(s) == (k, "V", j), ("V slot", self.vslot.get(s), (k, j))
                assert self.vt.get(b, ("free",))[0] in ("free", "used"), ("Vt overwritten", self.vt.get(b))
                yield
                self.vt[b] = ("Vt", k, j)
                self.B[("VE", s)].arrive()
                self.B[("VtF", b)].arrive()
                yield

    def tensor(self, i):
        while True:
            qu = self.queues[i]
            if qu and qu[0][0] == "CPQ":
                _, k = qu.pop(0)
                assert self.q.get(0) == (k, 0), ("Q tile", self.q.get(0), k)
                self.q_tmem = k
            elif qu and qu[0][0] == "PVT":
                _, (k, w, u, b, j, acc) = qu.pop(0)
                assert self.vt.get(b) == ("Vt", k, j), ("Vt", self.vt.get(b), (k, j))
                self.vt[b] = ("used",)
                self.slot[("vt", b)] = (k, "V", j)
                self.exec_pv(k, w, u, ("vt", b), j, acc, (k, w))
            elif qu and qu[0][0] == "SQ":
                _, (k, w, u, s, j) = qu.pop(0)
                assert self.q_tmem == k, ("Q in TMEM", self.q_tmem, k)
                self.q[("tmem",)] = (k, 0)
                self.exec_s(k, w, u, s, j, ("tmem",), (k, 0))
            elif qu:
                op, x = qu.pop(0)
                assert op == "commit", op
                self.B[x].arrive()
            yield

    def mma(self):
        kpos = vtc = 0
        pc = [0, 0]
        merges = 0
        qu = self.queues[0]
        for k, nk in enumerate(self.items):
            n1 = nk // 2
            while not self.ready("QF", k + 1):
                yield
            qu.append(("CPQ", k))
            qu.append(("commit", "QE"))

            def take_k():
                nonlocal kpos
                s, c = kpos % self.kst, kpos // self.kst + 1
                kpos += 1
                return s, c

            def issue_s(w, u, s, j):
                qu.append(("SQ", (k, w, u, s, j)))
                qu.append(("commit", ("SF", w)))
                qu.append(("commit", ("KE", s)))

            for j in range(min(nk, 2)):
                s, c = take_k()
                while not self.ready(("KF", s), c):
                    yield
                issue_s(j, 0, s, j)
                yield
            for j in range(nk):
                w, u = j & 1, j >> 1
                b, c = vtc % self.nvt, vtc // self.nvt + 1
                while not self.ready(("VtF", b), c):
                    yield
                vtc += 1
                if j == 1 and merges > 0:
                    while not self.ready("O1Free", merges):
                        yield
                while not self.ready(("PF", w), pc[w] + 1):
                    yield
                pc[w] += 1
                qu.append(("PVT", (k, w, u, b, j, j >= 2)))
                qu.append(("commit", ("VtE", b)))
                if j + 2 >= nk:
                    qu.append(("commit", ("OF", w)))
                yield
                if j + 2 < nk:
                    s, c = take_k()
                    while not self.ready(("KF", s), c):
                        yield
                    issue_s(w, u + 1, s, j + 2)
                    yield
            if n1 > 0:
                merges += 1

    softmax = SplitKD128.softmax


@pytest.mark.parametrize("stages", [(4, 2, 2), (2, 1, 1), (3, 2, 3), (2, 2, 1)])
def test_fp32_kernel(stages):
    rnd = random.Random(80 + sum(stages))
    for _ in range(120):
        items = [rnd.randint(1, 11) for _ in range(rnd.randint(1, 4))]
        SplitKF32(items, stages, seed=rnd.randrange(1 << 30)).run()


@pytest.mark.parametrize("drop,items", [
    (("VtE", 0), [6, 5]),      # a transposed buffer rewritten before its PV read it
    (("VE", 0), [6]),          # a V stage refilled before the transposers read it
    (("VtF", 1), [5]),         # PV before its transposed V was written
    ("QE", [1, 4]),            # the next Q tile loaded before the copy into TMEM read it
])
def test_fp32_model_catches_each_missing_wait(drop, items):
    M = type("M", (_Drop, SplitKF32), {"drop": (drop,)})
    failures = 0
    for seed in range(300):
        try:
            M(items, (4, 2, 2), seed=seed).run()
        except AssertionError:
            failures += 1
    assert failures > 0, drop
