"""Model check of the mbarrier protocol of the head_dim-256 prefill kernel
(paged_kv_attention_gqa_gb300/csrc/prefill_wide.cuh): a discrete-event simulation of its K and V
producer warps, its two MMA-issuing warps (one for S = Q K^T, one for O += P V) and its four softmax
warps under random latencies, with waits that poll by parity exactly as `mbarrier.try_wait.parity`
does.

The kernel's barriers: q_full; k_full[4] / k_empty[4] (one K stage, filled and released by 64-column
quarter: S(j)'s k-steps read the quarters in turn, so quarter q of K(j+1) is requested as soon as
the MMAs reading quarter q of K(j) completed); v_full[4] / v_empty[4] (one V stage, filled and
released by quarter of 32 keys: PV(j)'s k-steps read the key quarters in turn, so quarter q of
V(j+1) is requested as soon as the MMAs reading quarter q of V(j) completed);
s_full[2] (S(j) done in tensor-memory buffer j % 2), p_full[2] (the four softmax warps wrote P(j)
over that buffer), pv_done[2] (PV(j) done, counted per buffer), o_final. A commit makes its barrier
arrive once every MMA its own warp issued before it has completed.

Checked under many random schedules:
  * a parity wait is never ambiguous: a waiter polling for phase k finds the barrier at k or k + 1
    completed phases;
  * no hazard: S(j) is issued only after K_j landed and after PV(j-2), which reads P(j-2) from the
    same buffer, completed; a stage is refilled only after the MMAs reading it completed; the
    softmax reads S(j) only after it completed; PV(j) is issued only after P(j) was written by all
    four warps, and each key quarter of it only after that quarter of V_j landed (and, on the
    last tile, after its tail rows were zeroed); O is
    rescaled only while no PV is in flight; the epilogue reads O after all PVs;
  * every actor finishes (no deadlock).
Planted mistakes -- S(j) issued without waiting for PV(j-2), one pv_done barrier for both buffers
(waited two phases back), PV issued without waiting for P, the tail rows not zeroed first, every K
quarter refilled on the first quarter's release, every V quarter refilled on the first quarter's
release -- are caught."""
import heapq
import random

import pytest

from test_prefill_pair_protocol import Barrier


class Sim:
    def __init__(self, nt, seed, plant=None, tail=True):
        self.rng = random.Random(seed)
        self.nt, self.plant, self.tail = nt, plant, tail
        self.t, self.seq, self.q = 0, 0, []
        B = Barrier
        self.q_full = B("q_full", 1)
        self.k_full = [B(f"k_full{q}", 1) for q in range(4)]
        self.k_empty = [B(f"k_empty{q}", 1) for q in range(4)]
        self.v_full = [B(f"v_full{q}", 1) for q in range(4)]
        self.v_empty = [B(f"v_empty{q}", 1) for q in range(4)]
        self.s_full = [B(f"s_full{b}", 1) for b in range(2)]
        self.p_full = [B(f"p_full{b}", 4) for b in range(2)]
        self.pv_done = [B(f"pv_done{b}", 1) for b in range(2)]
        self.pv_one = B("pv_done", 1)  # the planted single barrier
        self.o_final = B("o_final", 1)
        self.s_cpl, self.pv_cpl, self.land = {}, {}, {}
        self.readers = {}
        self.p_written = {}
        self.tail_zeroed = None
        self.last_done = {"s": 0, "pv": 0}
        self.finished = 0
        self.spawned = 0

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

    def commit(self, who, bar):
        when = max(self.last_done[who], self.t) + self.rng.randint(0, 20)
        self.later(when - self.t, lambda: bar.arrive(self))

    def issue(self, who, reads):
        done = self.t + self.rng.randint(20, 600)
        self.last_done[who] = max(self.last_done[who], done)
        self.readers.setdefault(reads, []).append(done)
        return done

    def producer(self, kv):
        if kv == 0:
            self.q_full.arrive(self)
        for j in range(self.nt):
            for q in range(4):
                if kv == 0:
                    full, empty = self.k_full[q], self.k_empty[q if self.plant != "k_single_release" else 0]
                else:
                    full, empty = self.v_full[q], self.v_empty[q if self.plant != "v_single_release" else 0]
                key = ("K" if kv == 0 else "V", j, q)
                prev = ("K" if kv == 0 else "V", j - 1, q)
                if j > 0:
                    yield ("wait", empty, j - 1)
                    late = [c for c in self.readers.get(prev, []) if c > self.t]
                    assert not late, f"stage part {key} refilled while an MMA still reads {prev}"

                def fire(key=key, full=full):
                    self.land[key] = self.t
                    full.arrive(self)
                self.later(self.rng.randint(10, 2000), fire)
                yield ("delay", self.rng.randint(0, 60))

    def s_issuer(self):
        yield ("wait", self.q_full, 0)
        for j in range(self.nt):
            for q in range(4):  # the k-steps of quarter q, then its release
                yield ("wait", self.k_full[q], j)
                if q == 0 and j >= 2 and self.plant != "no_buf_wait":
                    if self.plant == "single_pv_barrier":
                        yield ("wait", self.pv_one, j - 2)
                    else:
                        yield ("wait", self.pv_done[j % 2], (j - 2) // 2)
                if q == 0 and j >= 2:
                    assert self.pv_cpl.get(j - 2, 1 << 60) <= self.t, f"S({j}) issued while PV({j - 2}) reads its buffer"
                assert self.land.get(("K", j, q), 1 << 60) <= self.t, f"S({j}) quarter {q} before it landed"
                self.s_cpl[j] = self.issue("s", ("K", j, q))
                self.commit("s", self.k_empty[q])
                yield ("delay", self.rng.randint(1, 40))
            self.commit("s", self.s_full[j % 2])

    def pv_issuer(self):
        for j in range(self.nt):
            if self.plant != "no_p_wait":
                yield ("wait", self.p_full[j % 2], j // 2)
            pw = self.p_written.get(j, [])
            assert len(pw) == 4 and max(pw) <= self.t, f"PV({j}) before P({j}) written"
            done = 0
            for q in range(4):  # the k-steps of key quarter q, then its release
                yield ("wait", self.v_full[q], j)
                if self.tail and j == self.nt - 1 and self.plant != "no_tail":
                    yield ("delay", self.rng.randint(5, 1000))  # zero this quarter's V rows past the row's end
                    self.tail_zeroed = self.t
                assert self.land.get(("V", j, q), 1 << 60) <= self.t, f"PV({j}) quarter {q} before it landed"
                if self.tail and j == self.nt - 1:
                    assert self.tail_zeroed is not None and self.tail_zeroed <= self.t, \
                        f"PV({j}) before the tail was zeroed"
                done = max(done, self.issue("pv", ("V", j, q)))
                self.commit("pv", self.v_empty[q])
                yield ("delay", self.rng.randint(1, 40))
            self.pv_cpl[j] = done
            self.commit("pv", self.pv_done[j % 2])
            if self.plant == "single_pv_barrier":
                self.commit("pv", self.pv_one)
            if j == self.nt - 1:
                self.commit("pv", self.o_final)
            yield ("delay", self.rng.randint(1, 40))
        if self.nt == 0:
            self.commit("pv", self.o_final)

    def softmax(self, w):
        for j in range(self.nt):
            yield ("wait", self.s_full[j % 2], j // 2)
            assert self.s_cpl[j] <= self.t, f"softmax read S({j}) before it completed"
            yield ("delay", self.rng.randint(50, 900))
            if j > 0 and self.rng.random() < 0.3:  # the running max grew: rescale O
                yield ("wait", self.pv_done[(j - 1) % 2], (j - 1) // 2)
                inflight = [i for i, t in self.pv_cpl.items() if t > self.t]
                assert not inflight, f"O rescaled at tile {j} while PV {inflight} in flight"
                yield ("delay", self.rng.randint(10, 200))
            self.p_written.setdefault(j, []).append(self.t)
            self.p_full[j % 2].arrive(self)
        yield ("wait", self.o_final, 0)
        assert len(self.pv_cpl) == self.nt and max(self.pv_cpl.values(), default=0) <= self.t

    def run(self):
        actors = [self.producer(0), self.producer(1), self.s_issuer(), self.pv_issuer()]
        actors += [self.softmax(w) for w in range(4)]
        for a in actors:
            self.run_actor(a)
        while self.q:
            self.t, _, fn = heapq.heappop(self.q)
            fn()
        assert self.finished == len(actors), f"deadlock: {self.finished} of {len(actors)} actors finished"


@pytest.mark.parametrize("nt", [0, 1, 2, 3, 4, 5, 8, 13])
def test_wide_barrier_protocol_is_sound(nt):
    for seed in range(150):
        Sim(nt, seed * 1000 + nt, tail=bool(seed & 1)).run()


@pytest.mark.parametrize("plant", ["no_buf_wait", "single_pv_barrier", "no_p_wait", "no_tail", "k_single_release",
                                   "v_single_release"])
def test_wide_model_catches_a_broken_protocol(plant):
    caught = 0
    for seed in range(200):
        try:
            Sim(8, seed, plant=plant, tail=True).run()
        except AssertionError:
            caught += 1
    assert caught > 0
