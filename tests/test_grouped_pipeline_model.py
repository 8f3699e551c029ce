"""A host model of the grouped GEMM's shared-memory pipeline protocol.

The tcgen05 kernel in csrc/grouped.cu runs six roles on one CTA that hand
shared-memory slots to each other through mbarriers: the code producer (code
tiles and, with scales by tensor copy, a two-box scale ring), the activation
producer, the MMA issuer, two dequantisation groups taking alternate stages,
and the epilogue (one or two accumulator buffers). This test replays the same
slot indices, barrier phase parities and arrival counts as the kernel, with a
random interleaving of the roles, and checks on every wait that the parity
test selects exactly the phase the role needs (no phase is skipped or taken
twice), that no slot is overwritten before its consumer is done with it, that
a role never reads a slot whose copy has not landed, and that every role
finishes (no deadlock). Bulk tensor copies land asynchronously: a seventh role,
the copy engine, completes the copies in flight in random order, so a copy can
land after later ones. Configurations cover one and several tiles, K stage
counts below, equal to and above the ring depths, odd stage counts (the
dequantisation groups swap stages between tiles), scale boxes of one stage, and
the INT3 ring depths with double-buffered accumulators, and the
weights-stationary rings, whose code copies hold R stages each (both groups
read every copy; its slot is free after all R stages). The model has to follow
the kernel: change both together.

With an odd code ring (INT4: three slots) a slot's consecutive stages belong
to different dequantisation groups, and a parity wait alone would pass while
the other group's earlier copy into the slot is still in flight; the kernel's
dequantisers therefore first wait until the producer has issued their stage
into the slot (`issued_word`). test_odd_code_ring_needs_the_issued_word shows
the model finding that race without it.
"""
import os
import random

import pytest


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self, n=1):
        self.arrived += n
        assert self.arrived <= self.count, f"{self.name}: too many arrivals in one phase"
        if self.arrived == self.count:
            self.completed += 1
            self.arrived = 0


def ready(bar, parity, phase_needed):
    """mbarrier try_wait.parity: true once the phase of that parity has completed.
    The protocol must make it select exactly completion number `phase_needed`."""
    ok = (bar.completed & 1) != parity
    if ok:
        assert bar.completed == phase_needed, (
            f"{bar.name}: parity wait passed with {bar.completed} completions, needed {phase_needed}")
    return ok


def simulate(ksteps, works, SA, SB, SC, ACC, tsc, span, seed, issued_word=True, R=1):
    assert ksteps % R == 0
    kcopies = ksteps // R                                       # code copies per tile
    rnd = random.Random(seed)
    in_flight = []                                              # copies issued, not landed: (kind, slot, barrier)
    a_landed, c_landed, s_landed = [False] * SA, [False] * SC, [False] * 2
    c_issued = [-1] * SC                                        # the kernel's cfill words
    afull = [Barrier(f"afull{s}", 1) for s in range(SA)]
    aempty = [Barrier(f"aempty{s}", 1) for s in range(SA)]
    cfull = [Barrier(f"cfull{s}", 1) for s in range(SC)]
    cempty = [Barrier(f"cempty{s}", R) for s in range(SC)]      # one group's arrival per stage of the copy
    bready = [Barrier(f"bready{s}", 1) for s in range(SB)]
    bempty = [Barrier(f"bempty{s}", 1) for s in range(SB)]
    accum = [Barrier(f"accum{b}", 1) for b in range(ACC)]
    drained = [Barrier(f"drained{b}", 1) for b in range(ACC)]
    sfull = [Barrier(f"sfull{b}", 1) for b in range(2)]
    sempty = [Barrier(f"sempty{b}", 2) for b in range(2)]       # both groups, or one group twice
    a_slot, b_slot, c_slot, s_box, acc_buf = [None] * SA, [None] * SB, [None] * SC, [None] * 2, [None] * ACC
    a_used, b_used, c_used = [True] * SA, [True] * SB, [True] * SC
    c_left = [0] * SC                                           # stages of the copy not yet dequantised
    nbox = (ksteps + span - 1) // span
    box_left = {}                                               # arrivals still due per scale box

    def wait(bar, parity, need):
        while not ready(bar, parity, need):
            yield

    def code_producer():
        spans = 0
        for j in range(works):
            for ci in range(kcopies):
                ic = j * kcopies + ci
                s = ic % SC
                yield from wait(cempty[s], ((ic // SC) & 1) ^ 1, ic // SC)
                for sub in range(R):
                    i = ci * R + sub
                    if tsc and i % span == 0:
                        m = spans
                        spans += 1
                        if m >= 2:
                            yield from wait(sempty[m & 1], ((m - 2) >> 1) & 1, (m - 2) // 2 + 1)
                            assert box_left[m - 2] == 0, "scale box overwritten before both groups released it"
                        s_box[m & 1] = m
                        s_landed[m & 1] = False
                        span_len = min(span, ksteps - i)
                        box_left[m] = 2 if span_len >= 2 else 1
                        in_flight.append(("s", m & 1, sfull[m & 1]))
                assert c_used[s], "code slot overwritten before it was dequantised"
                c_slot[s], c_used[s], c_landed[s], c_left[s] = ic, False, False, R
                c_issued[s] = ic
                in_flight.append(("c", s, cfull[s]))

    def act_producer():
        for j in range(works):
            for i in range(ksteps):
                it = j * ksteps + i
                s = it % SA
                yield from wait(aempty[s], ((it // SA) & 1) ^ 1, it // SA)
                assert a_used[s], "activation slot overwritten before the MMAs read it"
                a_slot[s], a_used[s], a_landed[s] = it, False, False
                in_flight.append(("a", s, afull[s]))

    def copy_engine():
        while True:
            if in_flight:
                kind, slot, bar = in_flight.pop(rnd.randrange(len(in_flight)))
                {"a": a_landed, "c": c_landed, "s": s_landed}[kind][slot] = True
                bar.arrive()
            yield

    def mma():
        for j in range(works):
            buf = j % ACC
            if j >= ACC:
                yield from wait(drained[buf], (j // ACC - 1) & 1, j // ACC)
            assert acc_buf[buf] is None, "accumulators overwritten before the epilogue read them"
            acc_buf[buf] = ("accumulating", j)
            for i in range(ksteps):
                it = j * ksteps + i
                sa, sb = it % SA, it % SB
                yield from wait(afull[sa], (it // SA) & 1, it // SA + 1)
                yield from wait(bready[sb], (it // SB) & 1, it // SB + 1)
                assert a_slot[sa] == it and b_slot[sb] == it, "MMA read the wrong stage"
                assert a_landed[sa], "MMA read an activation tile still in flight"
                a_used[sa] = b_used[sb] = True
                aempty[sa].arrive()
                bempty[sb].arrive()
            acc_buf[buf] = j
            accum[buf].arrive()

    def dequant(grp):
        box_seen = -1
        for j in range(works):
            for i in range(ksteps):
                it = j * ksteps + i
                if (it & 1) != grp:
                    continue
                ic = j * kcopies + i // R
                cs, bs = ic % SC, it % SB
                if issued_word and R == 1 and SC % 2 == 1:
                    while c_issued[cs] != ic:
                        yield
                yield from wait(cfull[cs], (ic // SC) & 1, ic // SC + 1)
                assert c_slot[cs] == ic, "dequantiser read the wrong code copy"
                assert c_landed[cs], "dequantiser read a code tile still in flight"
                m_cur = j * nbox + i // span
                if tsc and m_cur != box_seen:
                    box_seen = m_cur
                    yield from wait(sfull[m_cur & 1], (m_cur >> 1) & 1, (m_cur >> 1) + 1)
                    assert s_box[m_cur & 1] == m_cur, "dequantiser read the wrong scale box"
                    assert s_landed[m_cur & 1], "dequantiser read a scale box still in flight"
                yield from wait(bempty[bs], ((it // SB) & 1) ^ 1, it // SB)
                assert b_used[bs], "B slot overwritten before the MMAs read it"
                b_slot[bs], b_used[bs] = it, False
                bready[bs].arrive()
                c_left[cs] -= 1
                if c_left[cs] == 0:
                    c_used[cs] = True
                cempty[cs].arrive()
                if tsc:
                    box0 = (i // span) * span
                    box_end = min(box0 + span, ksteps)
                    if i + 2 >= box_end:
                        box_left[m_cur] -= 1            # this group is done with the box
                        sempty[m_cur & 1].arrive(1 if box_end - box0 >= 2 else 2)

    def epilogue():
        for j in range(works):
            buf = j % ACC
            yield from wait(accum[buf], (j // ACC) & 1, j // ACC + 1)
            assert acc_buf[buf] == j, "epilogue read the wrong tile"
            acc_buf[buf] = None
            drained[buf].arrive()

    roles = [code_producer(), act_producer(), mma(), dequant(0), dequant(1), epilogue()]
    live = list(roles)
    engine = copy_engine()
    steps = 0
    last = None
    while live:
        steps += 1
        assert steps < 10_000_000, "model did not finish"
        r = rnd.choice(live + [engine])
        if r is engine:
            next(engine)
            continue
        try:
            next(r)
        except StopIteration:
            live.remove(r)
            continue
        # a role that is blocked yields without progress; detect a global deadlock
        if steps % 20000 == 0:
            bars = afull + aempty + cfull + cempty + bready + bempty + accum + drained + sfull + sempty
            snapshot = (len(live), [(b.completed, b.arrived) for b in bars])
            assert snapshot != last, "deadlock: no role moved in 20000 scheduling steps"
            last = snapshot
    assert all(v == 0 for v in box_left.values()), "a scale box was not released by every group"


# (ksteps, works, SA, SB, SC, ACC, scales by tensor copy, stages per scale box[, stages per code copy])
CONFIGS = [
    (32, 3, 3, 3, 3, 1, True, 4),     # INT4 block 32, fc1 K = 2048
    (12, 4, 3, 3, 3, 1, True, 4),     # INT4 block 32, fc2 K = 768
    (12, 3, 3, 3, 3, 1, True, 16),    # block 128: one box longer than the tile
    (5, 3, 3, 3, 4, 1, False, 4),     # odd stage count, scales loaded by the producer (INT2 ring)
    (5, 3, 3, 3, 3, 1, True, 4),      # odd stage count with a one-stage scale box per tile
    (2, 5, 3, 3, 3, 1, True, 4),      # fewer stages than the B ring
    (1, 6, 3, 3, 3, 1, True, 4),      # one stage per tile
    (16, 4, 2, 2, 2, 2, True, 2),     # INT3 block 32 (K stage 128): double-buffered accumulators
    (3, 5, 2, 2, 2, 2, True, 4),      # INT3, short K
    # weights-stationary: 256-K code copies
    (32, 4, 3, 3, 2, 2, True, 4, 4),  # INT4 block 32, fc1 K = 2048: 4 stages per copy
    (12, 5, 3, 3, 2, 2, False, 4, 4), # INT4 / INT2 fc2 K = 768, scales by the producer
    (16, 4, 2, 2, 4, 2, True, 4, 2),  # INT3 block 64, fc1 K = 2048 (K stage 128): 2 stages per copy
    (6, 5, 2, 2, 4, 2, False, 4, 2),  # INT3 fc2 K = 768
    (4, 6, 3, 3, 2, 2, True, 16, 4),  # one copy per tile, block 128
]


@pytest.mark.parametrize("cfg", CONFIGS)
def test_pipeline_protocol(cfg):
    R = cfg[8] if len(cfg) > 8 else 1
    for seed in range(6):
        simulate(*cfg[:8], seed=seed, R=R)


def test_odd_code_ring_needs_the_issued_word():
    """Without the issued-stage word, some interleaving lets a dequantisation
    group pass its parity wait on a three-slot code ring while the other group's
    copy into that slot is still in flight."""
    failures = 0
    for seed in range(40):
        try:
            simulate(32, 3, 3, 3, 3, 1, True, 4, seed=seed, issued_word=False)
        except AssertionError:
            failures += 1
    assert failures > 0


# ---- ties to the CUDA source: the model's rings are the kernel's

_CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                     "quantized_mixture_experts_route_gb300", "csrc")
_GROUPED = open(os.path.join(_CSRC, "grouped.cu")).read()
_INTERNAL = open(os.path.join(_CSRC, "qmoe_internal.cuh")).read()

# the kernel's ring configuration, restated (the lines below are asserted verbatim)
_CFG_LINES = [
    "static constexpr int BK = BITS == 3 ? 128 : 64;",
    "static constexpr int BN = BITS == 3 ? 128 : 256;",
    "static constexpr int ACC = WS ? 2 : (4 * BN <= 512 ? 2 : 1);",
    "static constexpr int SA = BITS == 3 ? 2 : 3;",
    "static constexpr int SC = WS ? (BITS == 3 ? 4 : 2) : (BITS == 3 ? 2 : (BITS == 4 ? 3 : 4));",
    "static constexpr int SB = BITS == 3 ? 2 : 3;",
    "static constexpr int CK = WS ? kWsCodeK : BK;",
    "static constexpr int R = CK / BK;",
]


def _cfg(bits, ws):
    bk = 128 if bits == 3 else 64
    bn = 128 if bits == 3 else 256
    acc = 2 if ws else (2 if 4 * bn <= 512 else 1)
    sa = 2 if bits == 3 else 3
    sc = (4 if bits == 3 else 2) if ws else (2 if bits == 3 else (3 if bits == 4 else 4))
    sb = 2 if bits == 3 else 3
    r = (256 if ws else bk) // bk
    return sa, sb, sc, acc, r


def test_kernel_rings_are_the_models():
    for line in _CFG_LINES:
        assert line in _GROUPED, line
    assert "constexpr int kWsCodeK = 256;" in _INTERNAL
    covered = {(c[2], c[3], c[4], c[5], c[8] if len(c) > 8 else 1) for c in CONFIGS}
    for bits in (2, 3, 4):
        for ws in (False, True):
            assert _cfg(bits, ws) in covered, (bits, ws, _cfg(bits, ws))


def test_kernel_protocol_lines_are_the_models():
    """The arrival counts, the copy numbering, the issued-stage guard and the
    scale-box release rule that the model replays."""
    for line in ["mbar_init(bar_cempty(s), kDequantThreads * C::R);",
                 "const int ic = j * kcopies + i / C::R;",
                 "if (C::R == 1 && SC % 2 == 1 && !word_wait(cfill + cs, ic, abort_flag, launch_err))",
                 "if (i + 2 >= box_end) mbar_arrive_cnt(bar_sempty(m_cur & 1), box_end - box0 >= 2 ? 1u : 2u);",
                 "mbar_init(bar_sempty(b), 2 * kDequantThreads);",
                 "if ((it & 1) != grp) continue;"]:
        assert line in _GROUPED, line
