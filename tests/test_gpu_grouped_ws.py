"""The two grouped tcgen05 kernels on the same problems: route tiles (256 sorted
routes of one expert on the MMA M side, QMOE_PATH_GROUPED_ROUTE_TILES) and
weights-stationary tiles (128 dequantised weight rows on M, up to 128 routes of
one expert on N in steps of 16, QMOE_PATH_GROUPED_WS), each against the oracle
and against each other; QMOE_PATH_GROUPED picks the weights-stationary kernel
while the routes number at most 32 per expert.

Cases cover several 128-route tiles per expert, experts with one or two routes
(N = 16 against 128 weight rows), INT2/INT3/INT4 with and without zero points
(scales by bulk copies or by the producer warp), both dtypes, MXFP4 and NVFP4,
biases with full-softmax weights, and the INT3 Zipf workload at T = 512 in full
(sampled tokens). The weights-stationary kernel reads codes 256 K at a time, so
its cases have hidden and inter multiples of 256.
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
CASES = {
    # ~175 routes per expert: two 128-route tiles each
    "int4_bf16_two_tiles": (Shape(T=700, H=256, inter=256, E=8, k=2, bits=4, block=32, dtype=BF16), R1, 91),
    # zero points (scales and zero points staged by the producer warp)
    "int2_fp16_zp": (Shape(T=300, H=512, inter=256, E=5, k=2, bits=2, block=32, dtype=FP16),
                     dataclasses.replace(R1, explicit_zp=True), 92),
    "int3_b64": (Shape(T=500, H=512, inter=256, E=7, k=2, bits=3, block=64, dtype=BF16), R1, 93),
    "int3_b128_zp": (Shape(T=300, H=256, inter=512, E=4, k=2, bits=3, block=128, dtype=BF16),
                     dataclasses.replace(R1, explicit_zp=True), 94),
    # one or two routes per expert: N = 16 against 128 weight rows
    "int4_fp16_sparse": (Shape(T=40, H=512, inter=256, E=64, k=2, bits=4, block=32, dtype=FP16), R1, 95),
    # block 128 (a scale box spans 16 stages), H and inter multiples of 256
    "int4_b128": (Shape(T=260, H=1024, inter=512, E=16, k=4, bits=4, block=128, dtype=BF16), R1, 96),
}
FP4_CASES = {
    "mxfp4": (Shape(T=200, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16, format=1), 97),
    "nvfp4": (Shape(T=150, H=512, inter=256, E=16, k=4, bits=4, block=16, dtype=FP16, format=2), 98),
}


def oproblem(shape, inp=None, full_softmax=0):
    inp = inp or {}
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype, full_softmax, getattr(shape, "format", 0), inp.get("g1"), inp.get("g2"))


TILES, WS = 3, 4     # QMOE_PATH_GROUPED_ROUTE_TILES, QMOE_PATH_GROUPED_WS


def run(shape, inp, path, full_softmax=0):
    import torch

    import quantized_mixture_experts_route_gb300 as qm

    p = gu.problem(shape, path)
    d = gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward_ex(p, full_softmax, d.get("fc1_b"), d.get("fc2_b"), d["x"], d["logits"], d["fc1_q"],
                       d["fc1_s"], d.get("fc1_zp"), d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out, ws,
                       fc1_global_scale=d.get("g1"), fc2_global_scale=d.get("g2"))
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16).copy()


def both(shape, inp, label, full_softmax=0):
    ref, _ = oracle.forward(oproblem(shape, inp, full_softmax), inp)
    a = run(shape, inp, TILES, full_softmax)
    b = run(shape, inp, WS, full_softmax)
    gu.assert_parity(a, ref, shape.dtype, f"{label} route tiles")
    gu.assert_parity(b, ref, shape.dtype, f"{label} weights-stationary")
    fa, fb = gu.to_f64(a, shape.dtype), gu.to_f64(b, shape.dtype)
    assert np.linalg.norm(fa - fb) / np.linalg.norm(fa) < 2e-3, label


@pytest.mark.parametrize("name", sorted(CASES))
def test_route_tiles_and_weights_stationary(name):
    shape, recipe, seed = CASES[name]
    both(shape, synthetic.make_numpy(shape, recipe, seed), name)


@pytest.mark.parametrize("name", sorted(FP4_CASES))
def test_fp4_on_both_grouped_kernels(name):
    shape, seed = FP4_CASES[name]
    both(shape, synthetic.make_numpy(shape, Recipe(logit_std=1.0), seed), name)


@pytest.mark.parametrize("name", ["int4_fp16_sparse", "int3_b64"])
def test_biases_and_full_softmax_on_both(name):
    shape, recipe, seed = CASES[name]
    inp = synthetic.make_numpy(shape, dataclasses.replace(recipe, bias_std=0.5), seed)
    both(shape, inp, f"{name} with biases", full_softmax=1)


def test_grouped_takes_weights_stationary_for_few_routes_per_expert():
    """QMOE_PATH_GROUPED gives the weights-stationary kernel's output bit for bit at
    32 routes per expert or fewer, and the route tiles' above that."""
    shape, recipe, seed = CASES["int4_fp16_sparse"]          # 80 routes, E = 64
    inp = synthetic.make_numpy(shape, recipe, seed)
    assert np.array_equal(run(shape, inp, 2), run(shape, inp, WS))
    shape, recipe, seed = CASES["int4_bf16_two_tiles"]       # 1400 routes, E = 8
    inp = synthetic.make_numpy(shape, recipe, seed)
    assert np.array_equal(run(shape, inp, 2), run(shape, inp, TILES))


@pytest.mark.parametrize("block", [64, 128])
def test_int3_zipf_T512_route_tiles_sampled(block):
    """The INT3 Zipf workload in full on the route-tile kernel (AUTO, which the
    full-size sampled tests of the parity file use, takes the weights-stationary one)."""
    shape, recipe, seed = synthetic.int3_zipf(512, block)
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = run(shape, inp, TILES)
    rng = np.random.default_rng(block)
    toks = np.unique(np.concatenate([rng.choice(shape.T, size=24, replace=False), [0, shape.T - 1]]))
    ref, _ = oracle.forward(oproblem(shape), inp, tokens=toks)
    gu.assert_parity(got[toks], ref, shape.dtype, f"INT3 Zipf T=512 b{block} route tiles")
