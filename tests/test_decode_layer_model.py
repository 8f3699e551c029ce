"""A host model of the decode layer kernel's shared-memory protocol.

csrc/decode_layer.cu runs one producer warp and four consumer warps per block
around a ring of slots. The producer claims units (first fc1, then fc2) and, for
each group of four consecutive 256-wide chunks of a unit, waits until all four
consumers have handed the slot back, writes the slot's unit, first chunk and
unit sequence number, arms the slot's mbarrier with the copies' byte count and
issues the copies, which land later. Consumer warp w multiplies chunk w of
every slot (and hands back a slot with no chunk for it at once). A warp sums its
chunks of a unit, then leaves its sum in the unit's partial slot (one of four,
reused every fourth unit once the unit four earlier has been finished) and
counts itself; the last warp of the unit adds the sums in warp-position order
and frees the partial slot. After the last unit the producer arms one slot
without copies, which stops every consumer.

This test replays the kernel's slot indices, parity waits, arrival counts and
unit bookkeeping with random interleavings and copies that land in random
order, and checks on every wait that the parity selects exactly the phase the
role needs, that no warp reads a slot before its copies land or after its
reuse, that each unit's sum adds exactly its chunks in K order, that no partial
slot is overwritten before it is read, and that every role finishes. Because
every consumer waits on every phase of every slot, a parity wait can never pass
on a phase that is two behind. The ring depth, the consumer count and the
number of partial slots are read from the CUDA source, so the model follows the
kernel's constants.
"""
import random

import pytest

import os
import re

from tests.conftest import ROOT


def _kernel_constant(name):
    src = open(os.path.join(ROOT, "quantized_mixture_experts_route_gb300", "csrc", "decode_layer.cu")).read()
    consts = dict(re.findall(r"constexpr int (kL\w+) = (\w+);", src))
    v = consts[name]
    while not v.isdigit():
        v = consts[v]
    return int(v)


NC = _kernel_constant("kLConsumers")          # consumer warps, chunks per slot
RING = _kernel_constant("kLRing")             # slots per block
UNIT_SLOTS = _kernel_constant("kLUnitSlots")  # partial-sum slots


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count, f"{self.name}: too many arrivals in one phase"
        if self.arrived == self.count:
            self.completed += 1
            self.arrived = 0


def ready(bar, parity, phase_needed):
    """mbarrier try_wait.parity; it must select exactly completion `phase_needed`."""
    ok = (bar.completed & 1) != parity
    if ok:
        assert bar.completed == phase_needed, (
            f"{bar.name}: parity wait passed with {bar.completed} completions, needed {phase_needed}")
    return ok


def simulate(unit_chunks, R, seed):
    """unit_chunks: chunks per unit of the block's stream, in claim order."""
    rnd = random.Random(seed)
    full = [Barrier(f"full{s}", 1) for s in range(R)]
    empty = [Barrier(f"empty{s}", NC) for s in range(R)]
    meta = [None] * R                 # (unit seq, first chunk, chunks) or "end"
    landed = [False] * R
    in_flight = []
    part = {}                         # (partial slot, position) -> (unit seq, chunks summed)
    u_arrive = [0] * UNIT_SLOTS
    u_done = [s - UNIT_SLOTS for s in range(UNIT_SLOTS)]
    finished = {}

    def wait(bar, parity, need):
        while not ready(bar, parity, need):
            yield

    def producer():
        i = 0
        for useq, nst in enumerate(unit_chunks):
            for j0 in range(0, nst, NC):
                slot, ph = i % R, (i // R) & 1
                yield from wait(empty[slot], ph ^ 1, i // R)
                assert i < R or landed[slot], "slot refilled while its copies were in flight"
                meta[slot], landed[slot] = (useq, j0, nst), False
                in_flight.append(slot)
                i += 1
        slot, ph = i % R, (i // R) & 1
        yield from wait(empty[slot], ph ^ 1, i // R)
        meta[slot], landed[slot] = "end", True
        full[slot].arrive()

    def copy_engine():
        while True:
            if in_flight:
                slot = in_flight.pop(rnd.randrange(len(in_flight)))
                landed[slot] = True
                full[slot].arrive()
            yield

    def consumer(w):
        i = 0
        acc = None
        while True:
            slot, ph = i % R, (i // R) & 1
            yield from wait(full[slot], ph, i // R + 1)
            m = meta[slot]
            if m == "end":
                return
            assert landed[slot], f"warp {w} read slot use {i} before its copies landed"
            useq, j0, nst = m
            j = j0 + w
            i += 1
            if j >= nst:
                empty[slot].arrive()
                yield
                continue
            if j < NC:
                acc = []
            acc.append(j)             # this warp's chunks of the unit, in K order
            empty[slot].arrive()
            yield
            if j + NC < nst:
                continue
            us = useq % UNIT_SLOTS
            while u_done[us] != useq - UNIT_SLOTS:
                yield
            assert (us, w) not in part, "partial slot overwritten before it was read"
            part[(us, w)] = (useq, list(acc))
            u_arrive[us] += 1
            if u_arrive[us] != min(nst, NC):
                continue
            sums = []
            for q in range(min(nst, NC)):
                owner, chunks = part.pop((us, q))
                assert owner == useq, "partial sum of another unit"
                sums.append(chunks)
            u_arrive[us] = 0
            u_done[us] = useq
            # warp position q holds chunks q, q + NC, ...: together every chunk once, in order
            assert all(ch == list(range(q, nst, NC)) for q, ch in enumerate(sums))
            finished[useq] = True

    roles = [producer()] + [consumer(w) for w in range(NC)]
    engine = copy_engine()
    live = list(roles)
    steps = 0
    last = None
    while live:
        steps += 1
        assert steps < 5_000_000, "model did not finish"
        r = rnd.choice(live + [engine])
        if r is engine:
            next(engine)
            continue
        try:
            next(r)
        except StopIteration:
            live.remove(r)
            continue
        if steps % 20000 == 0:
            snap = (len(live), [(b.completed, b.arrived) for b in full + empty], len(finished))
            assert snap != last, "deadlock: no role moved in 20000 scheduling steps"
            last = snap
    assert len(finished) == len(unit_chunks), "a unit was not finished"


# chunks per unit: fc1 units of the decode stack (K = 2048: 8 chunks), fc2 units
# (K = 768: 3 chunks), one-chunk units, and a long-K fc1 (K = 8192: 32 chunks)
STREAMS = [
    [8] * 6 + [3] * 9,
    [3] * 20,
    [1, 2, 3, 4, 5, 8, 1, 1, 3],
    [32, 32, 3, 3],
    [],
]


@pytest.mark.parametrize("stream", STREAMS, ids=["fc1_then_fc2", "fc2_only", "mixed", "long_k", "no_units"])
def test_layer_protocol(stream):
    for seed in range(8):
        simulate(stream, R=RING, seed=seed)


@pytest.mark.parametrize("R", [1, 2, 5])
def test_layer_protocol_other_ring_depths(R):
    """The protocol does not depend on the ring depth (every consumer sees every phase)."""
    for seed in range(4):
        simulate([8] * 5 + [3] * 7, R=R, seed=seed)
