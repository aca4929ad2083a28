"""Model check of the mbarrier protocol of the prefill kernel (paged_kv_attention_gqa_gb300/
csrc/prefill_kernel.cuh, TMA path): a discrete-event simulation of its producer thread, MMA
thread and four softmax warps under random latencies, with waits that poll by parity exactly
as `mbarrier.try_wait.parity` does.

The kernel's barriers: k_full[2] / v_full[2] (a K or V tile landed), s_full[2] (S_j done; also
"K slot free"), p_full[2] (the four softmax warps wrote P_j), pv_done[2] (PV_j done; also "V slot
free", "S buffer free", and "O holds P_0..P_j V" for the rescale), o_final (after the last PV).
A commit makes its barrier arrive once every MMA the thread issued before it has completed.

Checked under many random schedules (any issue, load, MMA and wake-up latency):
  * a parity wait is never ambiguous: whenever a waiter polls for phase k, the barrier has
    completed k or k + 1 phases (k - 1 would pass too early, k + 2 would wait a phase too long);
  * no hazard: S_j is issued only after PV_{j-2} (which reads P_{j-2} from the same columns)
    completed; K_j / V_j are loaded into a slot only after S_{j-2} / PV_{j-2} completed; the
    softmax reads S_j only after it completed; PV_j is issued only after P_j was written and
    V_j landed; O is rescaled only while no PV is in flight; the epilogue reads O after all PVs;
  * every actor finishes (no deadlock).
The same holds for the cp.async gather path (pages below 8 slots): four producer warps, each
waiting on both barriers of a slot, copying its share of the tile's K and V rows, and arriving
on k_full / v_full, which then count four arrivals.
A planted mistake (the MMA thread not waiting for PV_{j-2}, or the producer reusing a V slot
on S-done) is caught, so the model can tell a broken protocol from a sound one."""
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
            for w in self.waiters:  # suspended waiters re-poll after a wake-up latency
                sim.later(sim.rng.randint(0, 30), w)
            self.waiters = []


class Sim:
    def __init__(self, nt, seed, plant=None, gather=False):
        self.rng = random.Random(seed)
        self.nt, self.plant, self.gather = nt, plant, gather
        nfull = 4 if gather else 1
        self.t, self.seq, self.q = 0, 0, []
        B = Barrier
        self.q_full = B("q_full", 1)
        self.k_full = [B(f"k_full{s}", nfull) for s in range(2)]
        self.v_full = [B(f"v_full{s}", nfull) for s in range(2)]
        self.s_full = [B(f"s_full{s}", 1) for s in range(2)]
        self.p_full = [B(f"p_full{s}", 4) for s in range(2)]
        self.pv_done = [B(f"pv_done{s}", 1) for s in range(2)]
        self.o_final = B("o_final", 1)
        # event log for the hazard checks: when each MMA group completes (fixed at issue) and
        # when each tile landed / P was written
        self.s_cpl, self.pv_cpl = {}, {}
        self.k_load, self.v_load, self.k_land, self.v_land = {}, {}, {}, {}
        self.p_written = {}
        self.mma_last_done = 0  # completion time of the latest MMA issued so far
        self.finished = 0

    def later(self, dt, fn):
        self.seq += 1
        heapq.heappush(self.q, (self.t + dt, self.seq, fn))

    # ---- actors are generators yielding ("delay", dt) or ("wait", barrier, phase)
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
                _, bar, k = op
                self.poll(bar, k, step)
        self.later(0, step)

    def poll(self, bar, k, resume):
        # the two ways a parity wait goes wrong
        assert bar.done >= k, f"{bar.name}: waiting for phase {k} with phase {k - 1} still open"
        assert bar.done <= k + 1, f"{bar.name}: waiting for phase {k} after phase {k + 1} completed"
        if (bar.done & 1) != (k & 1):  # try_wait.parity(k & 1) succeeds
            self.later(self.rng.randint(0, 5), resume)
        else:
            bar.waiters.append(lambda: self.poll(bar, k, resume))

    def commit(self, bar):
        # arrives once every MMA issued before it has completed
        when = max(self.mma_last_done, self.t) + self.rng.randint(0, 20)
        self.later(when - self.t, lambda: bar.arrive(self))

    def issue_mma(self):
        done = self.t + self.rng.randint(20, 400)
        self.mma_last_done = max(self.mma_last_done, done)
        return done

    def tma(self, bar, log, j):
        land = self.t + self.rng.randint(10, 2000)
        log[j] = self.t

        def fire():
            (self.k_land if bar in self.k_full else self.v_land)[j] = self.t
            bar.arrive(self)
        self.later(land - self.t, fire)

    # ---- the kernel's threads
    def producer(self):
        self.q_full.arrive(self)  # Q lands (modelled as already there)
        for j in range(self.nt):
            s, use = j & 1, j >> 1
            if use > 0:
                yield ("wait", self.s_full[s], use - 1)
            if j >= 2 and self.s_cpl.get(j - 2, float("inf")) > self.t:
                raise AssertionError(f"K slot of tile {j} reused before S_{j - 2} done")
            self.tma(self.k_full[s], self.k_load, j)
            yield ("delay", self.rng.randint(0, 50))  # the next tile's page ids
            if use > 0:
                if self.plant == "v_slot_on_s_done":
                    yield ("wait", self.s_full[s], use - 1)
                else:
                    yield ("wait", self.pv_done[s], use - 1)
            if j >= 2 and self.pv_cpl.get(j - 2, float("inf")) > self.t:
                raise AssertionError(f"V slot of tile {j} reused before PV_{j - 2} done")
            self.tma(self.v_full[s], self.v_load, j)

    def gather_producer(self, w):
        # one of four cp.async producer warps: waits on both barriers of the slot, copies its
        # share of tile j's K and V rows, waits for its copies, arrives on both full barriers
        for j in range(self.nt):
            s, use = j & 1, j >> 1
            if use > 0:
                yield ("wait", self.s_full[s], use - 1)
                if self.plant == "v_slot_on_s_done":
                    yield ("wait", self.s_full[s], use - 1)
                else:
                    yield ("wait", self.pv_done[s], use - 1)
            if j >= 2 and self.s_cpl.get(j - 2, float("inf")) > self.t:
                raise AssertionError(f"K slot of tile {j} overwritten before S_{j - 2} done")
            if j >= 2 and self.pv_cpl.get(j - 2, float("inf")) > self.t:
                raise AssertionError(f"V slot of tile {j} overwritten before PV_{j - 2} done")
            yield ("delay", self.rng.randint(50, 2500))  # issue, then wait for its own copies
            self.k_land[j] = max(self.k_land.get(j, 0), self.t)
            self.v_land[j] = max(self.v_land.get(j, 0), self.t)
            self.k_full[s].arrive(self)
            self.v_full[s].arrive(self)

    def mma(self):
        yield ("wait", self.q_full, 0)

        def issue_pv(i):
            s = i & 1
            yield ("wait", self.p_full[s], i >> 1)
            yield ("wait", self.v_full[s], i >> 1)
            assert i in self.p_written and self.p_written[i] <= self.t, f"PV_{i} before P_{i} written"
            assert i in self.v_land and self.v_land[i] <= self.t, f"PV_{i} before V_{i} landed"
            self.pv_cpl[i] = self.issue_mma()
            self.commit(self.pv_done[s])
            yield ("delay", self.rng.randint(1, 40))

        for j in range(self.nt):
            s = j & 1
            yield ("wait", self.k_full[s], j >> 1)
            if j >= 2 and self.plant != "no_pv_wait":
                yield ("wait", self.pv_done[s], (j - 2) >> 1)
            if j >= 2 and self.pv_cpl.get(j - 2, float("inf")) > self.t:
                raise AssertionError(f"S_{j} issued before PV_{j - 2} (reading the same columns) done")
            assert j in self.k_land and self.k_land[j] <= self.t, f"S_{j} before K_{j} landed"
            self.s_cpl[j] = self.issue_mma()
            self.commit(self.s_full[s])
            yield ("delay", self.rng.randint(1, 40))
            if j >= 1:
                yield from issue_pv(j - 1)
        if self.nt >= 1:
            yield from issue_pv(self.nt - 1)
        self.commit(self.o_final)

    def softmax(self, w):
        for j in range(self.nt):
            s = j & 1
            yield ("wait", self.s_full[s], j >> 1)
            assert self.s_cpl[j] <= self.t, f"softmax read S_{j} before it completed"
            yield ("delay", self.rng.randint(50, 900))
            if j > 0 and self.rng.random() < 0.3:  # the running max grew: rescale O
                yield ("wait", self.pv_done[(j - 1) & 1], (j - 1) >> 1)
                inflight = [i for i, t in self.pv_cpl.items() if t > self.t]
                assert not inflight, f"O rescaled at tile {j} while PV {inflight} in flight"
                yield ("delay", self.rng.randint(10, 200))
            self.p_written[j] = max(self.p_written.get(j, 0), self.t)
            self.p_full[s].arrive(self)
        yield ("wait", self.o_final, 0)
        assert len(self.pv_cpl) == self.nt and max(self.pv_cpl.values(), default=0) <= self.t

    def run(self):
        if self.gather:
            self.q_full.arrive(self)
            producers = [self.gather_producer(w) for w in range(4)]
        else:
            producers = [self.producer()]
        actors = producers + [self.mma()] + [self.softmax(w) for w in range(4)]
        for a in actors:
            self.run_actor(a)
        while self.q:
            self.t, _, fn = heapq.heappop(self.q)
            fn()
        assert self.finished == len(actors), f"deadlock: {self.finished} of {len(actors)} actors finished"


@pytest.mark.parametrize("gather", [False, True])
@pytest.mark.parametrize("nt", [1, 2, 3, 4, 5, 8, 13])
def test_prefill_barrier_protocol_is_sound(nt, gather):
    for seed in range(150):
        Sim(nt, seed * 1000 + nt, gather=gather).run()


# In the gather path the producers already wait for PV_{j-2} before copying K_j, so there the
# MMA thread's own wait for it is redundant and dropping it breaks nothing.
@pytest.mark.parametrize("plant,gather", [("no_pv_wait", False), ("v_slot_on_s_done", False),
                                          ("v_slot_on_s_done", True)])
def test_model_catches_a_broken_protocol(plant, gather):
    caught = 0
    for seed in range(200):
        try:
            Sim(8, seed, plant=plant, gather=gather).run()
        except AssertionError:
            caught += 1
    assert caught > 0
