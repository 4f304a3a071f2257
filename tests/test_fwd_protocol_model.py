"""Model check of the attention forward's synchronisation protocol (CPU, randomised schedules).

The forward kernel's roles are re-stated here as a model:
- the TMA producer: K_j and V_j into 2-slot rings;
- two MMA-issuing threads, one per 128-row query tile t, taking turns unit by unit;
- two softmax groups.

The model uses the same mbarriers, arrival counts, parities, wait orders and turn counter as
the kernel. The tensor core executes each issuing thread's MMAs and commits in that thread's
order only; the two threads' streams interleave arbitrarily, and TMA copies land at arbitrary
later times.

For every schedule the model checks:
- it terminates (no deadlock);
- no parity wait runs while its barrier is two or more phases ahead (parity aliasing);
- every MMA reads the K/V tile and P it expects, not one already overwritten;
- the softmax reads each S_t(j) before S_t(j + 1) overwrites it;
- the softmax rescales O only after every earlier P V into it has finished.

Cases cover a tile 1 with one more KV step than tile 0 (diagonal blocks), equal counts (a tile 1
past the end of the sequence, or the ring's full blocks), and single-step blocks."""
import random

import pytest


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; a parity wait tests the phase bit."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.completed += 1

    def done(self, phase):
        """Wait for the completion of phase `phase` by its parity, as try_wait.parity does."""
        assert self.completed <= phase + 1, "parity aliasing on %s: waiting for phase %d, %d done" % (
            self.name, phase, self.completed)
        return (self.completed & 1) != (phase & 1)


class Model:
    def __init__(self, n0, n1, full_blk, rng):
        self.n, self.full_blk, self.rng = (n0, n1), full_blk, rng
        B = Barrier
        self.k_full = [B("k_full0", 1), B("k_full1", 1)]
        self.k_empty = [B("k_empty0", 2), B("k_empty1", 2)]
        self.v_full = [B("v_full0", 1), B("v_full1", 1)]
        self.v_empty = [B("v_empty0", 2), B("v_empty1", 2)]
        self.s_full = [B("s_full0", 1), B("s_full1", 1)]
        self.p_full = [B("p_full0", 4), B("p_full1", 4)]
        self.o_done = [B("o_done0", 1), B("o_done1", 1)]
        self.units_done = [0, 0]
        self.k_slot, self.v_slot = [None, None], [None, None]   # tile held by each slot
        self.copies = []              # TMA copies in flight: (kind, slot, tile)
        self.queue = [[], []]         # per issuing thread: MMAs and commits not yet executed
        self.s_cols = [None, None]    # TMEM S_t columns: ("S", j) or ("P", j)
        self.pv_done = [-1, -1]       # last P V executed per tile

    # ------------------------------------------------------------------ tensor core
    def execute(self, t):
        op = self.queue[t].pop(0)
        kind = op[0]
        if kind == "commit":
            op[1].arrive()
        elif kind == "S":
            u = op[1]
            assert self.k_slot[u & 1] == u, "S_%d(%d) reads K slot holding %s" % (t, u, self.k_slot[u & 1])
            assert u == 0 or self.pv_done[t] >= u - 1, "S_%d(%d) overwrites P before P V" % (t, u)
            self.s_cols[t] = ("S", u)
        elif kind == "PV":
            u = op[1]
            assert self.v_slot[u & 1] == u, "P V_%d(%d) reads V slot holding %s" % (t, u, self.v_slot[u & 1])
            assert self.s_cols[t] == ("P", u), "P V_%d(%d) reads %s" % (t, u, self.s_cols[t])
            self.pv_done[t] = u

    # ---------------------------------------------------------------------- agents
    def tma(self):
        n1 = self.n[1]
        for j in range(n1):
            st = j & 1
            if j >= 2:
                while not self.k_empty[st].done((j - 2) >> 1):
                    yield
            self.copies.append(("K", st, j))
            if j >= 2:
                while not self.v_empty[st].done((j - 2) >> 1):
                    yield
            self.copies.append(("V", st, j))

    def mma(self, t):
        nt, n0 = self.n[t], self.n[0]
        for u in range(nt + 1):
            if u >= 1:
                while not self.p_full[t].done(u - 1):
                    yield
                while not self.v_full[(u - 1) & 1].done((u - 1) >> 1):
                    yield
            if u < nt:
                while not self.k_full[u & 1].done(u >> 1):
                    yield
            need = u if t == 0 else min(u + 1, n0 + 1)
            while self.units_done[1 - t] < need:
                yield
            q = self.queue[t]
            if u >= 1:
                q.append(("PV", u - 1))
            if u < nt:
                q.append(("S", u))
            self.units_done[t] = u + 1
            yield
            q.append(("commit", self.s_full[t] if u < nt else self.o_done[t]))
            if u >= 1:
                q.append(("commit", self.v_empty[(u - 1) & 1]))
            if u < nt:
                q.append(("commit", self.k_empty[u & 1]))

    def softmax(self, t, warp):
        """One softmax warp of tile t; warp 0 of the tile does the TMEM bookkeeping."""
        nt = self.n[t]
        for j in range(nt):
            while not self.s_full[t].done(j):
                yield
            if warp == 0:
                assert self.s_cols[t] == ("S", j), "softmax %d reads %s at step %d" % (t, self.s_cols[t], j)
                assert self.pv_done[t] >= j - 1, "softmax %d rescales O before P V(%d)" % (t, j - 1)
            yield
            if warp == 0:
                self.s_cols[t] = ("P", j)
            self.p_full[t].arrive()
            # the next step's wait: the other warps of the tile may still be on this one
        while not self.o_done[t].done(0):
            yield
        assert self.pv_done[t] == nt - 1

    # ------------------------------------------------------------------- scheduler
    def run(self, max_steps=200000):
        agents = [self.tma(), self.mma(0), self.mma(1)]
        agents += [self.softmax(t, w) for t in (0, 1) for w in range(4)]
        live = list(agents)
        for _ in range(max_steps):
            moves = [("agent", a) for a in live]
            moves += [("copy", i) for i in range(len(self.copies))]
            moves += [("tc", t) for t in (0, 1) if self.queue[t]]
            if not live and not self.copies and not any(self.queue):
                return
            kind, x = self.rng.choice(moves)
            if kind == "agent":
                try:
                    next(x)
                except StopIteration:
                    live.remove(x)
            elif kind == "copy":
                what, st, j = self.copies.pop(x)
                if what == "K":
                    self.k_slot[st] = j
                    self.k_full[st].arrive()
                else:
                    self.v_slot[st] = j
                    self.v_full[st].arrive()
            else:
                self.execute(x)
        raise AssertionError("no progress: deadlock (units %s, live agents %d)" % (
            self.units_done, len(live)))


CASES = [(1, 1, False), (1, 2, False), (2, 3, False), (3, 4, False), (6, 7, False),
         (2, 2, False), (5, 5, False), (4, 4, True), (7, 7, True)]


@pytest.mark.parametrize("n0,n1,full_blk", CASES)
def test_forward_protocol_is_safe_and_live(n0, n1, full_blk):
    rng = random.Random(1000 * n0 + 10 * n1 + full_blk)
    for _ in range(150):
        Model(n0, n1, full_blk, rng).run()


def test_model_catches_a_broken_protocol():
    """The check has teeth: with one K slot release instead of two (count 1), a schedule
    reloads a K slot while the other tile's S still needs it."""
    rng = random.Random(7)
    caught = False
    for _ in range(300):
        m = Model(4, 5, False, rng)
        m.k_empty = [Barrier("k_empty0", 1), Barrier("k_empty1", 1)]
        try:
            m.run()
        except AssertionError:
            caught = True
            break
    assert caught
