"""Model check of the mbarrier protocol of the two-query-tile prefill kernel
(paged_kv_attention_gqa_gb300/csrc/prefill_pair.cuh): a discrete-event simulation of its K and V
producer warps, its two MMA-issuing warps (one per query tile) and its two softmax warp groups
(four warps each) under random latencies, with waits that poll by parity exactly as
`mbarrier.try_wait.parity` does.

The kernel's barriers: q_full[2]; kv_full[NS] / kv_empty[NS] (a ring stage landed / the MMAs
reading it completed -- one commit per issuing warp, so two arrivals when both tiles are live);
s_full[2] (S_X(j) done), p_full[2] (group X wrote P_X(j); four arrivals), pv_done[2] (PV_X(j) done),
o_final[2]; turn[2] (the two softmax groups take turns, four arrivals each); v_tail (warp 9 zeroed
the V rows past the row's end on the last tile). A commit makes its barrier arrive once every MMA
its own warp issued before it has completed.

Checked under many random schedules:
  * a parity wait is never ambiguous: a waiter polling for phase k finds the barrier at k or k + 1
    completed phases;
  * no hazard: S_X(j) is issued only after PV_X(j-1) (which reads P_X(j-1) from the same columns)
    completed and K_j landed; a ring stage is refilled only after every MMA that read it (both
    tiles') completed; the softmax reads S_X(j) only after it completed; PV_X(j) is issued only
    after P_X(j) was written and V_j landed (and, on the last tile, after its tail rows were
    zeroed); O_X is rescaled only while no PV_X is in flight; the epilogue reads O_X after all PV_X;
  * the two softmax groups never run their main passes at the same time (the turns hold); with
    the head_dim-64 schedule (the turn passed on once S is loaded) their S loads never overlap;
  * every actor finishes (no deadlock), with one query tile or two.
Planted mistakes -- S issued without waiting for the previous PV, a stage released after one
warp's MMAs only, no turns, warp 10 not waiting for the tail rows -- are caught."""
import heapq
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, 0, 0
        self.waiters = []

    def arrive(self, sim):
        self.pending += 1
        assert self.pending <= self.count, f"{self.name}: too many arrivals"
        if self.pending == self.count:
            self.pending = 0
            self.done += 1
            for w in self.waiters:
                sim.later(sim.rng.randint(0, 30), w)
            self.waiters = []


class Sim:
    NS = 4

    def __init__(self, nt, two, seed, plant=None, tail=True, early_turn=False):
        self.rng = random.Random(seed)
        self.nt, self.two, self.plant, self.tail = nt, two, plant, tail
        self.early_turn = early_turn  # head_dim 64: the turn passes once S is loaded
        self.nq = 2 if two else 1
        self.t, self.seq, self.q = 0, 0, []
        B = Barrier
        release = 1 if plant == "single_release" else self.nq
        self.q_full = [B(f"q_full{x}", 1) for x in range(2)]
        self.kv_full = [B(f"kv_full{s}", 1) for s in range(self.NS)]
        self.kv_empty = [B(f"kv_empty{s}", release) for s in range(self.NS)]
        self.s_full = [B(f"s_full{x}", 1) for x in range(2)]
        self.p_full = [B(f"p_full{x}", 4) for x in range(2)]
        self.pv_done = [B(f"pv_done{x}", 1) for x in range(2)]
        self.o_final = [B(f"o_final{x}", 1) for x in range(2)]
        self.turn = [B(f"turn{x}", 4) for x in range(2)]
        self.v_tail = B("v_tail", 1)
        self.s_cpl = [{}, {}]
        self.pv_cpl = [{}, {}]
        self.land = {}          # ring sequence number -> landing time
        self.readers = {}       # ring sequence number -> completion times of the MMAs reading it
        self.p_written = [{}, {}]
        self.tail_zeroed = None
        self.mma_last_done = [0, 0]
        self.in_main = [0, 0]   # softmax warps of each group inside their main pass
        self.finished = 0

    def later(self, dt, fn):
        self.seq += 1
        heapq.heappush(self.q, (self.t + dt, self.seq, fn))

    def run_actor(self, gen):
        def step(_=None):
            try:
                op = next(gen)
            except StopIteration:
                self.finished += 1
                return
            if op[0] == "delay":
                self.later(op[1], step)
            else:
                self.poll(op[1], op[2], step)
        self.later(0, step)

    def poll(self, bar, k, resume):
        assert bar.done >= k, f"{bar.name}: waiting for phase {k} with phase {k - 1} still open"
        assert bar.done <= k + 1, f"{bar.name}: waiting for phase {k} after phase {k + 1} completed"
        if (bar.done & 1) != (k & 1):
            self.later(self.rng.randint(0, 5), resume)
        else:
            bar.waiters.append(lambda: self.poll(bar, k, resume))

    def commit(self, x, bar):
        # tcgen05.commit: arrives once every MMA issued by this warp so far has completed
        when = max(self.mma_last_done[x], self.t) + self.rng.randint(0, 20)
        self.later(when - self.t, lambda: bar.arrive(self))

    def issue_mma(self, x, reads):
        done = self.t + self.rng.randint(20, 400)
        self.mma_last_done[x] = max(self.mma_last_done[x], done)
        self.readers.setdefault(reads, []).append(done)
        return done

    # ---- producers: warp 8 (K, ring sequence 2j) and warp 11 (V, 2j + 1)
    def producer(self, kv):
        if kv == 0:
            for x in range(self.nq):
                self.q_full[x].arrive(self)
        for j in range(self.nt):
            i = 2 * j + kv
            s, use = i % self.NS, i // self.NS
            if use > 0:
                yield ("wait", self.kv_empty[s], use - 1)
                prev = self.readers.get(i - self.NS, [])
                assert len(prev) == self.nq or self.plant == "single_release", f"stage {s} freed by {len(prev)} warps"
                late = [c for c in prev if c > self.t]
                assert not late, f"ring stage {s} refilled (sequence {i}) while an MMA still reads sequence {i - self.NS}"
                if self.plant == "single_release" and len(prev) < self.nq:
                    raise AssertionError(f"ring stage {s} refilled before every tile's MMAs read it")
            land = self.t + self.rng.randint(10, 2000)

            def fire(i=i, s=s):
                self.land[i] = self.t
                self.kv_full[s].arrive(self)
            self.later(land - self.t, fire)
            yield ("delay", self.rng.randint(0, 60))  # the next tile's page ids

    # ---- MMA warps: warp 9 (x = 0) and warp 10 (x = 1)
    def mma(self, x):
        yield ("wait", self.q_full[x], 0)
        if self.nt > 0:
            yield ("wait", self.kv_full[0], 0)
        for j in range(self.nt):
            ik, iv = 2 * j, 2 * j + 1
            sk, sv = ik % self.NS, iv % self.NS
            if j > 0 and self.plant != "no_pv_wait":
                yield ("wait", self.pv_done[x], j - 1)
            if j > 0 and self.pv_cpl[x][j - 1] > self.t:
                raise AssertionError(f"S{x}({j}) issued before PV{x}({j - 1}) (reading the same columns) done")
            assert ik in self.land and self.land[ik] <= self.t, f"S{x}({j}) before K_{j} landed"
            self.s_cpl[x][j] = self.issue_mma(x, ik)
            self.commit(x, self.s_full[x])
            self.commit(x, self.kv_empty[sk])
            yield ("delay", self.rng.randint(1, 40))
            yield ("wait", self.kv_full[sv], iv // self.NS)
            if self.tail and j == self.nt - 1:
                if x == 0:
                    yield ("delay", self.rng.randint(5, 4000))  # zero the tail rows (the warp may be slow to get here)
                    self.tail_zeroed = self.t
                    if self.two:
                        self.v_tail.arrive(self)
                elif self.plant != "no_tail_wait":
                    yield ("wait", self.v_tail, 0)
            if j + 1 < self.nt:
                yield ("wait", self.kv_full[(ik + 2) % self.NS], (ik + 2) // self.NS)
            yield ("wait", self.p_full[x], j)
            assert j in self.p_written[x] and self.p_written[x][j] <= self.t, f"PV{x}({j}) before P written"
            assert iv in self.land and self.land[iv] <= self.t, f"PV{x}({j}) before V_{j} landed"
            if self.tail and j == self.nt - 1:
                assert self.tail_zeroed is not None and self.tail_zeroed <= self.t, f"PV{x}({j}) before the tail was zeroed"
            self.pv_cpl[x][j] = self.issue_mma(x, iv)
            self.commit(x, self.pv_done[x])
            self.commit(x, self.kv_empty[sv])
            if j == self.nt - 1:
                self.commit(x, self.o_final[x])
            yield ("delay", self.rng.randint(1, 40))
        if self.nt == 0:
            self.commit(x, self.o_final[x])

    # ---- softmax warp groups: warps 0-3 (x = 0), 4-7 (x = 1)
    def softmax(self, x, w):
        turns = self.two and self.plant != "no_turn"
        for j in range(self.nt):
            if turns and (x == 1 or j > 0):
                yield ("wait", self.turn[x], j if x else j - 1)
            yield ("wait", self.s_full[x], j)
            assert self.s_cpl[x][j] <= self.t, f"softmax {x} read S({j}) before it completed"
            self.in_main[x] += 1
            assert self.in_main[1 - x] == 0, f"both softmax groups in their main pass at tile {j}"
            if self.early_turn:
                yield ("delay", self.rng.randint(10, 200))  # the S load
                self.in_main[x] -= 1
                if self.two and self.plant != "no_turn":
                    self.turn[1 - x].arrive(self)
                yield ("delay", self.rng.randint(50, 800))  # max and exp pass
            else:
                yield ("delay", self.rng.randint(50, 900))
                self.in_main[x] -= 1
                if self.two and self.plant != "no_turn":
                    self.turn[1 - x].arrive(self)
            if j > 0 and self.rng.random() < 0.3:  # the running max grew: rescale O_X
                yield ("wait", self.pv_done[x], j - 1)
                inflight = [i for i, t in self.pv_cpl[x].items() if t > self.t]
                assert not inflight, f"O{x} rescaled at tile {j} while PV {inflight} in flight"
                yield ("delay", self.rng.randint(10, 200))
            self.p_written[x][j] = max(self.p_written[x].get(j, 0), self.t)
            self.p_full[x].arrive(self)
        yield ("wait", self.o_final[x], 0)
        assert len(self.pv_cpl[x]) == self.nt and max(self.pv_cpl[x].values(), default=0) <= self.t

    def run(self):
        actors = [self.producer(0), self.producer(1)]
        for x in range(self.nq):
            actors.append(self.mma(x))
            actors += [self.softmax(x, w) for w in range(4)]
        for a in actors:
            self.run_actor(a)
        while self.q:
            self.t, _, fn = heapq.heappop(self.q)
            fn()
        assert self.finished == len(actors), f"deadlock: {self.finished} of {len(actors)} actors finished"


@pytest.mark.parametrize("early_turn", [False, True])
@pytest.mark.parametrize("two", [False, True])
@pytest.mark.parametrize("nt", [0, 1, 2, 3, 4, 5, 8, 13])
def test_pair_barrier_protocol_is_sound(nt, two, early_turn):
    for seed in range(120):
        Sim(nt, two, seed * 1000 + nt, tail=bool(seed & 1), early_turn=early_turn).run()


@pytest.mark.parametrize("early_turn", [False, True])
@pytest.mark.parametrize("plant", ["no_pv_wait", "single_release", "no_turn", "no_tail_wait"])
def test_pair_model_catches_a_broken_protocol(plant, early_turn):
    caught = 0
    for seed in range(200):
        try:
            Sim(8, True, seed, plant=plant, tail=True, early_turn=early_turn).run()
        except AssertionError:
            caught += 1
    assert caught > 0
