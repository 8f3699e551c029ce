"""A host model of the decode kernels' stream-K split (csrc/decode.cu,
decode_int4_tma_kernel).

The flattened range of (work unit, 256-wide K chunk) pairs is cut into equal
pieces of L chunks, one per warp of the persistent grid (L at least 2). A unit
cut between warps is finished by its last arriving part: each part stores its
FP32 partial tile in one of the warp's two slots of the workspace (slot 0 for
the piece's first unit, slot 1 for its last), takes a ticket, and the warp that
sees the ticket reach the part count adds the parts in chunk order, reading
warp w0's tile from slot 1 when w0's piece began before the unit and every
later warp's from slot 0. This test replays that arithmetic for many unit
counts, chunk counts and grid sizes and checks that every chunk is computed
exactly once, that no warp needs a third slot or writes one slot twice, that
the slots the last arriver reads are exactly the slots the parts wrote, in
chunk order, and that every slot index stays inside the workspace the host
sizes (two slots per warp of the grid). The model has to follow the kernel:
change both together.
"""
import itertools

import pytest

K_MIN_PIECE = 2


def split(units, nq, gw):
    cfull = units * nq
    L = max(K_MIN_PIECE, (cfull + gw - 1) // gw)
    nw = (cfull + L - 1) // L
    covered = [0] * cfull
    written = {}                                 # unit -> list of (chunk begin, warp, slot)
    for wg in range(gw):
        if wg >= nw:
            continue
        x_begin = wg * L
        total = min(x_begin + L, cfull) - x_begin
        assert total > 0
        slots_used = set()
        f, first_unit = 0, True
        unit, cic = divmod(x_begin, nq)
        while f < total:
            first_cic = cic
            while True:                          # the chunks of this unit in this piece
                covered[unit * nq + cic] += 1
                cic += 1
                f += 1
                if not (cic < nq and f < total):
                    break
            whole = first_cic == 0 and cic == nq
            if not whole:
                slot = 0 if first_unit else 1
                assert slot not in slots_used, "a warp wrote one partial slot twice"
                slots_used.add(slot)
                assert wg * 2 + slot < 2 * gw, "partial slot outside the workspace"
                written.setdefault(unit, []).append((unit * nq + first_cic, wg, slot))
            if cic == nq:
                cic = 0
                unit += 1
            first_unit = False
    assert all(c == 1 for c in covered), "a chunk is computed zero or several times"
    for unit, parts in written.items():
        ux = unit * nq
        w0, w1 = ux // L, (ux + nq - 1) // L
        assert len(parts) == w1 - w0 + 1, "ticket count differs from the number of parts"
        hs0 = 1 if w0 * L < ux else 0
        read = [(w, hs0 if w == w0 else 0) for w in range(w0, w1 + 1)]
        assert [(w, s) for _, w, s in sorted(parts)] == read, "last arriver reads other slots or order"
    return L, nw


@pytest.mark.parametrize("nq", [1, 3, 4, 8, 32])
def test_split_covers_every_chunk_once(nq):
    for units, gw in itertools.product([1, 2, 3, 7, 16, 52 * 48, 113, 1000], [1, 5, 16, 64, 152 * 16]):
        split(units, nq, gw)


def test_split_of_the_decode_layer():
    # fc1 of the 2048 / 768 / 128-expert layer at T = 8: 52 experts in ~28 decode-table
    # entries x 48 groups of 32 rows x 8 chunks; fc2: 16-row groups x 3 chunks
    L, nw = split(28 * 48, 8, 152 * 16)
    assert L >= K_MIN_PIECE and nw <= 152 * 16
    split(28 * 128, 3, 152 * 16)


def test_model_constant_matches_the_kernel():
    """The minimum piece the model uses is the kernel's."""
    import os
    import re

    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "quantized_mixture_experts_route_gb300", "csrc", "decode.cu")).read()
    assert int(re.search(r"constexpr int kTMinPiece = (\d+);", src).group(1)) == K_MIN_PIECE
