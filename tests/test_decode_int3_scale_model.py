"""A host model of the INT3 / INT2 decode kernel's block-scale staging
(csrc/decode.cu, decode_int23_tma_kernel).

Each warp walks its piece of `total` chunks through a ring of kRing shared-
memory slots. Issuing chunk i (in the prologue for i < kRing - 1, otherwise
at the top of iteration i - kRing + 1) loads its scales into registers and,
first, stores the previously issued chunk's registers into that chunk's slot;
an iteration that issues nothing stores the pending registers instead. After
that the warp computes chunk f from slot f % kRing. The model replays this
order for every piece length and checks that each chunk's scales are stored
exactly once, into its own slot, before the chunk is computed, and that no
slot's scales are overwritten between their store and their use. The model
has to follow the kernel: change both together.
"""
import os
import re

import pytest

SRC = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "quantized_mixture_experts_route_gb300", "csrc", "decode.cu")).read()


def kernel_ring():
    body = SRC[SRC.index("struct T23Cfg {"):SRC.index("struct Tma23Args {")]
    return int(re.search(r"static constexpr int kRing = (\d+);", body).group(1))


def replay(total, ring):
    slot_content = {}                    # slot -> chunk whose scales it holds
    stored = {}                          # chunk -> number of stores
    pending = None                       # chunk whose scales sit in registers
    computed = []

    def store_pending():
        nonlocal pending
        if pending is not None:
            slot_content[pending % ring] = pending
            stored[pending] = stored.get(pending, 0) + 1
        pending = None

    def issue(chunk):
        nonlocal pending
        store_pending()                  # the previous chunk's scales go to its slot
        pending = chunk                  # this chunk's are loaded into registers

    pre = min(total, ring - 1)
    for u in range(pre):
        issue(u)
    for f in range(total):
        if f + ring - 1 < total:
            issue(f + ring - 1)
        else:
            store_pending()
        # compute chunk f from its slot
        assert slot_content.get(f % ring) == f, (total, ring, f, slot_content)
        computed.append(f)
    assert computed == list(range(total))
    assert all(stored.get(i) == 1 for i in range(total)), stored
    assert pending is None


def test_kernel_ring_is_three():
    assert kernel_ring() == 3


@pytest.mark.parametrize("total", list(range(1, 40)))
def test_scales_in_place_before_use(total):
    replay(total, kernel_ring())


def test_the_kernel_follows_the_model():
    """The issue lambda stores before it loads, and an iteration without an issue stores."""
    body = SRC[SRC.index("decode_int23_tma_kernel("):]
    i_store = body.index("    scale_store();\n    if (lane < ROWS) {")
    i_load = body.index("s_pend = __ldg(")
    assert i_store < i_load
    assert "if (f + C::kRing - 1 < total) issue(true, 0);\n    else scale_store();" in body
