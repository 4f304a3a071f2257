"""Model check of the attention backward's synchronisation protocol (CPU, randomised schedules).

The backward kernel's roles are re-stated here as a model:
- the TMA producer: K and V once, then each item's Q, dO and row terms through a 4-stage ring;
- issuer A: S^T and dQ^T, in region pairs;
- issuer B: dP^T, dV and dK, in item order, each item's dV/dK only after issuer A has issued
  that item's dQ^T (a shared counter, an ordering preference the kernel bounds);
- two element-wise groups, one per TMEM region, items alternating between the regions.

The model uses the same mbarriers, arrival counts, parities and wait orders as the kernel. The
tensor core executes each issuer's MMAs and commits in that issuer's order only; the two
streams interleave arbitrarily, and TMA copies land at arbitrary later times.

For every schedule the model checks:
- it terminates;
- no parity wait runs two or more phases behind its barrier;
- every MMA and element-wise pass reads the item it expects from the Q/dO stage, the row
  terms, the TMEM region (S^T, dP^T, P^T, dQ^T) and the dS buffer;
- nothing is overwritten before its last reader has finished;
- dV and dK are read out only after every MMA into them.

Item counts cover the degenerate (0, 1, 2) and ring-wrapping (> 4 stages) cases."""
import random

import pytest

from test_fwd_protocol_model import Barrier

NST = 4


class Model:
    def __init__(self, n, rng):
        self.n, self.rng = n, rng
        B = Barrier
        self.kv_full = B("kv_full", 1)
        self.qd_full = [B("qd_full%d" % i, 1) for i in range(NST)]
        self.qd_empty = [B("qd_empty%d" % i, 1) for i in range(NST)]
        self.s_full = [B("s_full%d" % i, 2) for i in range(2)]   # S^T (A) and dP^T (B)
        self.p_full = [B("p_full%d" % i, 1) for i in range(2)]
        self.dq_full = [B("dq_full%d" % i, 1) for i in range(2)]
        self.dq_free = [B("dq_free%d" % i, 1) for i in range(2)]
        self.acc_done = B("acc_done", 1)
        self.kv = False
        self.qd = [None] * NST           # item whose Q/dO a stage holds
        self.rows = [None] * NST         # item whose row terms a stage holds
        self.s_part = [None, None]       # region's S^T columns: ("S", it) or ("DQ", it)
        self.p_part = [None, None]       # region's dP^T columns: ("DP", it) or ("P", it)
        self.ds = [None, None]           # item whose dS a region's smem buffer holds
        self.executed = set()            # (op, item) done by the tensor core
        self.ew1, self.ew2 = set(), set()   # items whose element-wise passes are done
        self.copies = []
        self.queue = {"A": [], "B": []}
        self.dq_issued = 0               # items whose dQ^T issuer A has queued

    def done(self, op, it):
        return (op, it) in self.executed

    # ------------------------------------------------------------------ tensor core
    def execute(self, who):
        op = self.queue[who].pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, it = op
        X, st = it & 1, it % NST
        assert self.kv, "%s(%d) before K/V landed" % (kind, it)
        if kind == "S":
            assert self.qd[st] == it, "S^T(%d) reads Q of %s" % (it, self.qd[st])
            if it >= 2:
                assert self.s_part[X] == ("DQ", it - 2) and it - 2 in self.ew2, \
                    "S^T(%d) over dQ^T(%d) not yet read out" % (it, it - 2)
            self.s_part[X] = ("S", it)
        elif kind == "DP":
            assert self.qd[st] == it, "dP^T(%d) reads dO of %s" % (it, self.qd[st])
            if it >= 2:
                assert self.p_part[X] == ("P", it - 2) and self.done("DV", it - 2), \
                    "dP^T(%d) over P^T(%d) before dV read it" % (it, it - 2)
            self.p_part[X] = ("DP", it)
        elif kind == "DQ":
            assert self.ds[X] == it and self.s_part[X] == ("S", it) and it in self.ew1, \
                "dQ^T(%d): dS %s, columns %s" % (it, self.ds[X], self.s_part[X])
            self.s_part[X] = ("DQ", it)
        elif kind == "DV":
            assert self.p_part[X] == ("P", it) and self.qd[st] == it, "dV(%d)" % it
        elif kind == "DK":
            assert self.ds[X] == it and self.qd[st] == it, "dK(%d)" % it
        self.executed.add((kind, it))

    # ---------------------------------------------------------------------- agents
    def tma(self):
        self.copies.append(("KV", None, None))
        for it in range(self.n):
            st = it % NST
            if it >= NST:
                while not self.qd_empty[st].done(it // NST - 1):
                    yield
                old = it - NST
                assert old in self.ew1, "row terms of %d overwritten before use" % old
            self.rows[st] = it
            self.copies.append(("QD", st, it))

    def issuer_a(self):
        while not self.kv_full.done(0):
            yield
        q = self.queue["A"]

        def mma_s(it):
            X, st = it & 1, it % NST
            while not self.qd_full[st].done(it // NST):
                yield
            if it >= 2:
                while not self.dq_free[X].done((it - 2) >> 1):
                    yield
            q.append(("S", it))
            q.append(("commit", self.s_full[X]))

        def mma_dq(it):
            X = it & 1
            while not self.p_full[X].done(it >> 1):
                yield
            q.append(("DQ", it))
            q.append(("commit", self.dq_full[X]))
            self.dq_issued = it + 1

        for it in range(min(2, self.n)):
            yield from mma_s(it)
        for it in range(0, self.n, 2):
            yield from mma_dq(it)
            if it + 1 < self.n:
                yield from mma_dq(it + 1)
            if it + 2 < self.n:
                yield from mma_s(it + 2)
            if it + 3 < self.n:
                yield from mma_s(it + 3)

    def issuer_b(self):
        while not self.kv_full.done(0):
            yield
        q = self.queue["B"]

        def mma_dp(it):
            X, st = it & 1, it % NST
            while not self.qd_full[st].done(it // NST):
                yield
            q.append(("DP", it))
            q.append(("commit", self.s_full[X]))

        for it in range(min(2, self.n)):
            yield from mma_dp(it)
        for it in range(self.n):
            X, st = it & 1, it % NST
            while not self.p_full[X].done(it >> 1):
                yield
            while self.dq_issued <= it:
                yield
            q.append(("DV", it))
            q.append(("DK", it))
            q.append(("commit", self.qd_empty[st]))
            if it + 2 < self.n:
                yield from mma_dp(it + 2)
        q.append(("commit", self.acc_done))

    def elementwise(self, X):
        """A region's eight warps: one leader waits, the rest follow through a named barrier,
        so the group acts as one agent with one arrival per hand-off."""
        for it in range(X, self.n, 2):
            u, st = it >> 1, it % NST
            while not self.s_full[X].done(u):
                yield
            assert self.s_part[X] == ("S", it), "EW(%d) reads S^T columns %s" % (it, self.s_part[X])
            assert self.p_part[X] == ("DP", it), "EW(%d) reads dP^T columns %s" % (it, self.p_part[X])
            assert self.rows[st] == it, "EW(%d) reads row terms of %s" % (it, self.rows[st])
            yield
            if it >= 2:
                assert self.done("DQ", it - 2) and self.done("DK", it - 2), \
                    "dS(%d) overwrites dS(%d) before its readers" % (it, it - 2)
            self.ds[X] = it
            self.p_part[X] = ("P", it)
            self.ew1.add(it)
            self.p_full[X].arrive()
            while not self.dq_full[X].done(u):
                yield
            assert self.s_part[X] == ("DQ", it), "EW(%d) reads dQ^T columns %s" % (it, self.s_part[X])
            self.ew2.add(it)
            self.dq_free[X].arrive()
        if self.n > 0:
            while not self.acc_done.done(0):
                yield
            for it in range(self.n):
                assert self.done("DV", it) and self.done("DK", it)

    # ------------------------------------------------------------------- scheduler
    def run(self, max_steps=400000):
        live = [self.tma(), self.issuer_a(), self.issuer_b(), self.elementwise(0),
                self.elementwise(1)]
        for _ in range(max_steps):
            if not live and not self.copies and not any(self.queue.values()):
                return
            moves = [("agent", a) for a in live]
            moves += [("copy", i) for i in range(len(self.copies))]
            moves += [("tc", w) for w in ("A", "B") if self.queue[w]]
            kind, x = self.rng.choice(moves)
            if kind == "agent":
                try:
                    next(x)
                except StopIteration:
                    live.remove(x)
            elif kind == "copy":
                what, st, it = self.copies.pop(x)
                if what == "KV":
                    self.kv = True
                    self.kv_full.arrive()
                else:
                    old = it - NST
                    if old >= 0:
                        for op in ("S", "DP", "DV", "DK"):
                            assert self.done(op, old), "Q/dO of %d overwritten before %s" % (old, op)
                    self.qd[st] = it
                    self.qd_full[st].arrive()
            else:
                self.execute(x)
        raise AssertionError("no progress: deadlock")


@pytest.mark.parametrize("n_items", [0, 1, 2, 3, 4, 5, 8, 9, 13])
def test_backward_protocol_is_safe_and_live(n_items):
    rng = random.Random(n_items)
    for _ in range(120):
        Model(n_items, rng).run()


def test_model_catches_a_broken_protocol():
    """The check has teeth: if S^T's barrier took only issuer A's commit, the element-wise
    pass would read dP^T before issuer B's MMA wrote it."""
    rng = random.Random(3)
    caught = False
    for _ in range(300):
        m = Model(6, rng)
        m.s_full = [Barrier("s_full0", 1), Barrier("s_full1", 1)]
        try:
            m.run()
        except AssertionError:
            caught = True
            break
    assert caught
