"""A host model of the decode layer kernel's scheduling protocol.

csrc/decode_layer.cu runs independent warps. Each warp claims units (an entry's
32-row group of fc1 or fc2, all of K) from one counter, in the order of the
kernel's unit queue: the fc1 units of the first L entries, then rounds of one
entry's fc1 units followed by the fc2 units of the entry L places earlier,
then the fc2 units of the last L entries. A warp streams a unit's K chunks
through its own ring of kLStages stages: it issues a chunk's copies as one
committed group while fewer than kLStages chunks are in flight, claims its next
unit when it issues the copies of the current unit's last two chunks, and
multiplies its oldest chunk after waiting until at most (in flight - 1) of its
groups are pending. The copy engine lands groups in any order. An fc2 chunk's
activations (the entry's SwiGLU outputs) are copied only once every fc1 unit of
the entry has finished; a warp that finds them not finished stops issuing,
multiplies what it has in flight, and only then waits. A block's warps share the
set of entries already seen finished.

This test replays that protocol with random interleavings and random landing
order and checks, at every step, that a chunk is multiplied only after its
copies landed, that no stage is refilled before it was multiplied, that a
unit's chunks are multiplied in K order by the warp that claimed it, that an
fc2 chunk's activations are copied only after all fc1 units of its entry
finished, that every unit is finished exactly once, and that the warps never
deadlock (the wait for an entry always ends). The ring depth and the queue
are read from the CUDA source, so the model follows the kernel.
"""
import os
import random
import re

import pytest

from tests.conftest import ROOT

SRC = open(os.path.join(ROOT, "quantized_mixture_experts_route_gb300", "csrc", "decode_layer.cu")).read()


def _kernel_constant(name):
    consts = dict(re.findall(r"constexpr int (kL\w+) = (\w+);", SRC))
    v = consts[name]
    while not v.isdigit():
        v = consts[v]
    return int(v)


STAGES = _kernel_constant("kLStages")


def unit_queue(entries, a, b, L):
    """The kernel's UnitQueue::decode for every position: (fc1?, entry, row group)."""
    out = []
    p1, p2 = L * a, L * a + (entries - L) * (a + b)
    for q in range(entries * (a + b)):
        if q < p1:
            out.append((True, q // a, q % a))
        elif q < p2:
            r, o = divmod(q - p1, a + b)
            out.append((True, L + r, o) if o < a else (False, r, o - a))
        else:
            r, o = divmod(q - p2, b)
            out.append((False, entries - L + r, o))
    return out


def test_queue_is_a_permutation_with_fc1_first():
    for entries, a, b, L in [(5, 3, 4, 2), (7, 2, 3, 7), (4, 6, 2, 1), (1, 3, 3, 1), (9, 48, 64, 4)]:
        q = unit_queue(entries, a, b, L)
        assert sorted(q) == sorted([(True, e, r) for e in range(entries) for r in range(a)] +
                                   [(False, e, r) for e in range(entries) for r in range(b)])
        last_fc1 = {e: max(i for i, u in enumerate(q) if u[0] and u[1] == e) for e in range(entries)}
        first_fc2 = {e: min(i for i, u in enumerate(q) if not u[0] and u[1] == e) for e in range(entries)}
        assert all(last_fc1[e] < first_fc2[e] for e in range(entries))


def test_kernel_queue_matches_the_model():
    """The model's queue is the kernel's: the same three ranges in the same order."""
    body = SRC[SRC.index("struct UnitQueue"):SRC.index("template <bool BF16S, int FMT>")]
    assert "const int p1 = L * a, p2 = p1 + (entries - L) * (a + b);" in body
    assert "ei = f1 ? L + r : r;" in body and "ei = entries - L + r;" in body


def simulate(entries, a, b, nst1, nst2, warps, per_block, L, seed):
    rnd = random.Random(seed)
    queue = unit_queue(entries, a, b, L)
    nunits = len(queue)
    claim = [0]
    fc1_done = [0] * entries
    finished = {}
    ready = [set() for _ in range((warps + per_block - 1) // per_block)]

    def take():
        q = claim[0]
        claim[0] += 1
        return q

    def warp(w):
        blk = ready[w // per_block]
        ring = [None] * STAGES                 # per stage: (unit, chunk) it holds
        groups = []                            # per issued group: landed?
        issued = computed = 0
        iu = take()
        nxt = nunits
        ij = 0
        chunks_seen = {}
        while True:
            # issue
            while iu < nunits and issued - computed < STAGES:
                f1, ei, _ = queue[iu]
                inst = nst1 if f1 else nst2
                if not f1 and ij == 0 and ei not in blk:
                    if fc1_done[ei] < a:
                        if issued != computed:
                            break              # drain first
                        while fc1_done[ei] < a:
                            yield "wait"
                    blk.add(ei)
                if not f1:
                    assert fc1_done[ei] == a, "fc2 activations copied before the entry's fc1 finished"
                st = issued % STAGES
                assert ring[st] is None, "stage refilled before it was multiplied"
                ring[st] = (iu, ij)
                groups.append(False)
                issued += 1
                if ij == max(inst - 2, 0):
                    nxt = take()
                ij += 1
                if ij == inst:
                    iu, ij = nxt, 0
                yield "issue"
            if issued == computed:
                return
            # wait until at most (in flight - 1) groups are pending: all older ones landed
            while not all(groups[: computed + 1]):
                yield "copy"
            st = computed % STAGES
            u, j = ring[st]
            f1, ei, _ = queue[u]
            inst = nst1 if f1 else nst2
            assert chunks_seen.get(u, 0) == j, "chunks out of K order"
            chunks_seen[u] = j + 1
            ring[st] = None
            computed += 1
            if j + 1 == inst:
                assert u not in finished, "unit finished twice"
                finished[u] = w
                if f1:
                    fc1_done[ei] += 1
            yield "compute"

    roles = {w: warp(w) for w in range(warps)}
    # the copy engine reaches each warp's group list through the generator's frame
    live = list(roles)
    steps = 0
    stalled = 0
    while live:
        steps += 1
        assert steps < 2_000_000, "model did not finish"
        if rnd.random() < 0.3:
            # land one random pending group of one random warp
            cands = [w for w in live if any(not x for x in roles[w].gi_frame.f_locals.get("groups", []))]
            if cands:
                w = rnd.choice(cands)
                gs = roles[w].gi_frame.f_locals["groups"]
                i = rnd.choice([i for i, x in enumerate(gs) if not x])
                gs[i] = True
                stalled = 0
                continue
        w = rnd.choice(live)
        try:
            r = next(roles[w])
        except StopIteration:
            live.remove(w)
            stalled = 0
            continue
        stalled = 0 if r in ("issue", "compute") else stalled + 1
        if stalled > 200_000:
            raise AssertionError("deadlock: no warp issued or multiplied for 200000 steps")
    assert sorted(finished) == list(range(nunits)), "a unit was not finished"


CASES = {
    # entries, fc1 units per entry, fc2 units per entry, fc1 chunks, fc2 chunks, warps, warps per block
    "decode_stack_scaled": (9, 6, 8, 8, 3, 10, 4),
    "few_warps": (5, 3, 4, 8, 3, 2, 2),
    "one_warp": (3, 2, 2, 4, 2, 1, 1),
    "one_chunk_units": (6, 2, 3, 1, 1, 7, 3),
    "many_warps": (4, 2, 2, 3, 2, 16, 4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_protocol(name):
    entries, a, b, nst1, nst2, warps, per_block = CASES[name]
    for seed in range(6):
        # the kernel's lag: one wave of claims (one unit per warp) in fc1-unit lists, plus 2
        L = min(warps // a + 2, entries)
        simulate(entries, a, b, nst1, nst2, warps, per_block, L, seed)


@pytest.mark.parametrize("L", [1, 2, "all"])
def test_layer_protocol_any_lag(L):
    """The wait always ends whatever the lag: fc1 units precede their fc2 units."""
    entries, a, b = 6, 3, 4
    for seed in range(4):
        simulate(entries, a, b, 4, 2, 5, 2, entries if L == "all" else L, seed)


def test_kernel_lag_and_claim_rule_match_the_model():
    assert "int lag = (int)(gridDim.x * kLWarps) / rg1 + 2;" in SRC
    assert "if (ij == (inst > 2 ? inst - 2 : 0)) next = atomicAdd(claim, 1);" in SRC
    assert "if (issued != computed) break;" in SRC
