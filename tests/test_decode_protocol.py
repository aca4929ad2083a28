"""Model check of the decode kernel's stage ring (paged_kv_attention_gqa_gb300/csrc/decode.cu):
a producer filling `stages` slots in turn (full[s]: one TMA arrival, or one per producer lane
on the cp.async path) and Hc consumer warps that each read every chunk and arrive on empty[s]
(count Hc); before the CTA exits the producer waits, chunk by chunk, for the last `stages`
chunks it issued to be consumed.

Under random latencies (the same parity-polling model as the prefill protocol test):
  * every parity wait finds its barrier k or k + 1 phases on (never ambiguous);
  * no slot is refilled before every consumer released it, no consumer reads a chunk before
    it landed, and the CTA never exits with a chunk in flight;
  * nothing deadlocks.
A ring whose producer skips the empty wait is caught."""
import random

import pytest

from test_prefill_protocol import Barrier, Sim


class RingSim(Sim):
    def __init__(self, chunks, stages, consumers, arrivals, seed, plant=None):
        super().__init__(0, seed, plant=plant)
        self.chunks, self.stages, self.nc = chunks, stages, consumers
        self.full = [Barrier(f"full{s}", arrivals) for s in range(stages)]
        self.empty = [Barrier(f"empty{s}", consumers) for s in range(stages)]
        self.arrivals = arrivals
        self.landed, self.released, self.exit_t = {}, {}, None

    def ring_producer(self):
        for it in range(self.chunks):
            s, use = it % self.stages, it // self.stages
            if use > 0 and self.plant != "no_empty_wait":
                yield ("wait", self.empty[s], use - 1)
            prev = it - self.stages
            if prev >= 0 and len(self.released.get(prev, ())) < self.nc:
                raise AssertionError(f"slot {s} refilled with chunk {it} before chunk {prev} was released")
            for _ in range(self.arrivals):  # TMA transaction, or one cp.async arrival per lane
                self.later(self.rng.randint(10, 1500), self._lander(it, s))
            yield ("delay", self.rng.randint(1, 60))
        for d in range(max(0, self.chunks - self.stages), self.chunks):  # the drain
            yield ("wait", self.empty[d % self.stages], d // self.stages)
        assert all(len(self.released.get(i, ())) == self.nc for i in range(self.chunks)), "exit with chunks in flight"
        self.exit_t = self.t

    def _lander(self, it, s):
        def fire():
            self.landed.setdefault(it, 0)
            self.landed[it] += 1
            self.full[s].arrive(self)
        return fire

    def consumer(self, w):
        for it in range(self.chunks):
            s = it % self.stages
            yield ("wait", self.full[s], it // self.stages)
            assert self.landed.get(it, 0) == self.arrivals, f"chunk {it} read before it landed"
            yield ("delay", self.rng.randint(20, 400))
            self.released.setdefault(it, set()).add(w)
            self.empty[s].arrive(self)

    def run(self):
        actors = [self.ring_producer()] + [self.consumer(w) for w in range(self.nc)]
        for a in actors:
            self.run_actor(a)
        import heapq
        while self.q:
            self.t, _, fn = heapq.heappop(self.q)
            fn()
        assert self.finished == len(actors), f"deadlock: {self.finished} of {len(actors)} finished"


@pytest.mark.parametrize("stages,consumers,arrivals", [(2, 1, 1), (3, 4, 1), (4, 8, 1), (6, 2, 32), (8, 4, 64),
                                                        (16, 1, 1)])
def test_decode_ring_is_sound(stages, consumers, arrivals):
    rng = random.Random(stages * 100 + consumers)
    for seed in range(60):
        RingSim(rng.randint(0, 40), stages, consumers, arrivals, seed).run()


def test_model_catches_a_ring_without_empty_waits():
    caught = 0
    for seed in range(100):
        try:
            RingSim(30, 2, 4, 1, seed, plant="no_empty_wait").run()
        except AssertionError:
            caught += 1
    assert caught > 0

