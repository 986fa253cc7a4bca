"""A model of the throughput kernel's stage ring, checked on the CPU.

The kernel's three roles (stage warp, write-back lane, consumer warps) pass
each shared-memory stage through three mbarriers: full (the stage's bulk
loads landed), empty (every role is done with it) and cdone (consumer warps
stored a chunk that other CTAs wait on).  A parity wait is only sound if the
barrier is exactly one phase from the one being waited for, and an mbarrier
must never receive more arrivals than it expects.  This model runs the
roles' orders of operations under random interleavings (bulk copies
completing at random times) for random mixes of chunk kinds and ring depths
and asserts:

  * no wait passes before the phase it means has completed;
  * no barrier is ever two phases ahead of a waiter;
  * no barrier is over-arrived;
  * a stage is never refilled while a role still reads it;
  * every run finishes (no deadlock).

The planted-mistake test reruns the model with the earlier ordering, in which
roles skipped the chunks they do not handle, and checks that the model
reports it.
"""
import random

import pytest


class ProtocolError(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.phase = 0
        self.pending = count
        self.tx = 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError(f"{self.name}: over-arrived in phase {self.phase}")
        self._maybe_complete()

    def arrive_expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive(1)

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._maybe_complete()

    def test_wait(self, want_phase):
        """The hardware answers from parity alone; the model also checks that
        the answer is the right one for the absolute phase meant."""
        ready = (self.phase & 1) != (want_phase & 1)
        if self.phase >= want_phase + 2:
            raise ProtocolError(f"{self.name}: two phases ahead of a waiter "
                                f"(at {self.phase}, waiting for {want_phase})")
        if ready and self.phase <= want_phase:
            raise ProtocolError(f"{self.name}: parity wait passed early "
                                f"(at {self.phase}, waiting for {want_phase})")
        return ready


def run_model(kinds, S, ncw=2, seed=0, old_order=False, max_steps=200000):
    """kinds[k]: 'copy' (aligned, write-back lane), 'cons' (reduce or shifted
    copy, consumer warps), 'notify' (reduce chunk another CTA waits on)."""
    rng = random.Random(seed)
    full = [Barrier(f"full[{i}]", 1) for i in range(S)]
    empty = [Barrier(f"empty[{i}]", (ncw if old_order else ncw + 1)) for i in range(S)]
    C = S if old_order else 2 * S          # cdone ring entries
    cdone = [Barrier(f"cdone[{i}]", ncw) for i in range(C)]
    slot_chunk = [None] * S          # which chunk's data a stage holds
    readers = [set() for _ in range(S)]
    inflight_loads = []              # (slot, chunk)
    inflight_reads = []              # (group id, slot, chunk) of write-back bulk stores
    n = len(kinds)

    def producer():
        for k in range(n):
            slot = k % S
            if k >= S:
                while not empty[slot].test_wait(k // S - 1):
                    yield
            if readers[slot]:
                raise ProtocolError(f"stage {slot} refilled while read by {readers[slot]}")
            slot_chunk[slot] = ("loading", k)
            full[slot].arrive_expect_tx(16)
            inflight_loads.append((slot, k))
            yield

    def consumer(w):
        for k in range(n):
            slot = k % S
            while not full[slot].test_wait(k // S):
                yield
            if slot_chunk[slot] != k:
                raise ProtocolError(f"consumer {w} saw stage {slot} holding {slot_chunk[slot]}, "
                                    f"expected chunk {k}")
            kind = kinds[k]
            if old_order and kind == "copy":
                continue                      # the earlier ordering skipped these chunks
            if kind == "copy":
                empty[slot].arrive()
                yield
                continue
            readers[slot].add(("c", w))
            yield                             # reading the stage
            if slot_chunk[slot] != k:
                raise ProtocolError(f"stage {slot} changed under consumer {w}")
            readers[slot].discard(("c", w))
            if kind == "notify":
                cdone[k % C].arrive()
                if not old_order:
                    empty[slot].arrive()
            else:
                empty[slot].arrive()
            yield

    def writer():
        owed = None
        group = 0
        cd_phase = [0] * C
        for k in range(n):
            slot = k % S
            kind = kinds[k]
            if kind != "copy":
                if old_order:
                    if kind != "notify":
                        continue
                    while not cdone[slot].test_wait(cd_phase[slot]):
                        yield
                    cd_phase[slot] += 1
                    empty[slot].arrive(ncw)
                    continue
                while inflight_reads:             # settle the owed release first
                    yield
                if owed is not None:
                    empty[owed].arrive()
                    owed = None
                while not full[slot].test_wait(k // S):
                    yield
                empty[slot].arrive()
                if kind == "notify":
                    e = k % C
                    while not cdone[e].test_wait(cd_phase[e]):
                        yield
                    cd_phase[e] += 1
                yield
                continue
            while not full[slot].test_wait(k // S):
                yield
            if slot_chunk[slot] != k:
                raise ProtocolError(f"writer saw stage {slot} holding {slot_chunk[slot]}")
            group += 1
            readers[slot].add(("w", group))
            inflight_reads.append((group, slot, k))
            # wait until at most one group still reads shared memory
            while len(inflight_reads) > 1:
                yield
            if owed is not None:
                empty[owed].arrive(1 if not old_order else ncw)
            owed = slot
            yield
        while inflight_reads:
            yield
        if owed is not None:
            empty[owed].arrive(1 if not old_order else ncw)

    roles = {"producer": producer(), "writer": writer()}
    for w in range(ncw):
        roles[f"consumer{w}"] = consumer(w)
    done = set()
    for step in range(max_steps):
        events = [r for r in roles if r not in done]
        if inflight_loads:
            events.append("tma_load")
        if inflight_reads:
            events.append("tma_read")
        if not events:
            return step
        ev = rng.choice(events)
        if ev == "tma_load":
            slot, k = inflight_loads.pop(rng.randrange(len(inflight_loads)))
            slot_chunk[slot] = k
            full[slot].complete_tx(16)
        elif ev == "tma_read":
            g, slot, k = inflight_reads.pop(0)          # bulk groups complete in order
            if slot_chunk[slot] != k:
                raise ProtocolError(f"stage {slot} changed under a bulk store of chunk {k}")
            readers[slot].discard(("w", g))
        else:
            try:
                next(roles[ev])
            except StopIteration:
                done.add(ev)
    raise ProtocolError("deadlock: no progress within the step budget")


def random_kinds(rng, n):
    pattern = rng.choice(["copy", "cons", "mixed", "composed", "alternate"])
    if pattern == "copy":
        return ["copy"] * n
    if pattern == "cons":
        return ["cons"] * n
    if pattern == "composed":
        m = rng.randrange(n + 1)
        return ["notify"] * m + ["copy"] * (n - m)
    if pattern == "alternate":
        return ["copy" if (k // rng.randrange(1, 4)) % 2 == 0 else "cons" for k in range(n)]
    return [rng.choice(["copy", "cons"]) for _ in range(n)]


@pytest.mark.parametrize("S", [2, 3, 4, 6])
def test_ring_protocol_random_interleavings(S):
    rng = random.Random(S)
    for trial in range(400):
        n = rng.randrange(1, 30)
        kinds = random_kinds(rng, n)
        run_model(kinds, S, ncw=rng.choice([1, 2, 3]), seed=trial)


def test_ring_protocol_catches_the_skipping_order():
    """The earlier ordering (roles skipping chunks they do not handle, and the
    writer holding a release while waiting elsewhere) must be reported."""
    failures = 0
    rng = random.Random(7)
    for trial in range(200):
        kinds = [rng.choice(["copy", "cons"]) for _ in range(rng.randrange(4, 20))]
        try:
            run_model(kinds, 2, ncw=2, seed=trial, old_order=True, max_steps=20000)
        except ProtocolError:
            failures += 1
    assert failures > 0
