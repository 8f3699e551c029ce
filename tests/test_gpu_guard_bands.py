"""Guard bands around the output and the workspace on every matmul kernel family.

The workspace and the output are carved out of larger buffers whose outer 4 KiB
on each side, and the whole workspace itself, are filled with a byte pattern
before the call. After the call the bands must still hold the pattern (no write
outside the caller's buffers), and the output must match the oracle (nothing
read from the workspace before it was written). The shapes leave ragged tails:
route counts that fill no whole 128- or 256-row tile, weight row counts (fc1
2 x inter, fc2 hidden) that are not multiples of the 256-row weight tile, and
decode units of 16 and 32 rows. With compute-sanitizer closed, these bands are
the out-of-bounds evidence for the tile copies and the epilogues' stores.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

R1 = Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02)
TILES, WS, DECODE = 3, 4, 1     # QMOE_PATH_GROUPED_ROUTE_TILES, QMOE_PATH_GROUPED_WS, QMOE_PATH_DECODE
CASES = {
    # 602 routes over 8 experts; fc1 N = 384 and fc2 N = 320 end in part-filled 256-row tiles
    "route_tiles_int4_ragged": (Shape(T=301, H=320, inter=192, E=8, k=2, bits=4, block=32, dtype=BF16),
                                R1, 201, TILES),
    # INT2 with zero points (scales staged by the producer warp); fc1 N = 640, fc2 N = 448
    "route_tiles_int2_zp_ragged": (Shape(T=257, H=448, inter=320, E=6, k=2, bits=2, block=64, dtype=FP16),
                                   dataclasses.replace(R1, explicit_zp=True), 202, TILES),
    # INT3: 128-row weight tiles with double-buffered accumulators
    "route_tiles_int3": (Shape(T=200, H=384, inter=256, E=5, k=2, bits=3, block=128, dtype=FP16), R1, 203, TILES),
    # about 25 routes per expert: N = 32 of 128 route columns
    "weights_stationary_ragged": (Shape(T=133, H=512, inter=256, E=16, k=3, bits=4, block=32, dtype=FP16),
                                  R1, 204, WS),
    # decode tensor-copy kernel: fc1 in 32-row units (K = 1024), fc2 in 16-row units
    "decode_int4_tma": (Shape(T=8, H=1024, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16), R1, 205, DECODE),
    # INT3 decode tensor-copy kernel
    "decode_int3_tma": (Shape(T=4, H=256, inter=256, E=8, k=2, bits=3, block=64, dtype=BF16), R1, 206, DECODE),
    # generic decode kernel (zero points)
    "decode_generic_zp": (Shape(T=5, H=192, inter=96, E=6, k=2, bits=4, block=32, dtype=FP16),
                          dataclasses.replace(R1, explicit_zp=True), 207, DECODE),
}
G = 4096


@pytest.mark.parametrize("name", sorted(CASES))
def test_guard_bands_and_parity(name):
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    shape, recipe, seed, path = CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    p = gu.problem(shape, path)
    n_ws = qm.qmoe_workspace_bytes(p)
    assert n_ws > 0
    n_out = shape.T * shape.H
    ws_big = torch.full((n_ws + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
    out_big = torch.full((n_out + 2 * G,), 0x3C3C, dtype=torch.int16, device="cuda")
    got = gu.gpu_forward(shape, inp, path=path, ws=ws_big[G:G + n_ws],
                         out=out_big[G:G + n_out].view(shape.T, shape.H))
    wb = ws_big.cpu().numpy()
    ob = out_big.cpu().numpy()
    assert (wb[:G] == 0x5A).all() and (wb[G + n_ws:] == 0x5A).all(), f"{name}: write outside the workspace"
    assert (ob[:G] == 0x3C3C).all() and (ob[G + n_out:] == 0x3C3C).all(), f"{name}: write outside the output"
    ref, _ = oracle.forward(oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits,
                                           shape.block, shape.dtype), inp)
    gu.assert_parity(got, ref, shape.dtype, name)
    assert not np.isnan(gu.to_f64(got, shape.dtype)).any(), name
