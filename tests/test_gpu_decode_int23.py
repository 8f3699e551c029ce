"""The INT3 / INT2 decode tensor-copy kernel (implicit zero points 4 and 2;
blocks of 32, 64 and 128; hidden and inter multiples of 256) against the oracle.

Cases span both unit heights (16-row units for one or two tokens or short K,
32-row units otherwise), both dtypes, every block size (8, 4 or 2 scales per
256-wide chunk, scale rows that are not a multiple of 16 bytes: K = 768 with
blocks of 64 and 128), decode-table entries with one and two routes, split-K
pieces cut inside a unit, biases with full-softmax weights, the mid-size T
that still runs on the decode path, and the INT3 Zipf workload's shape; the
same for 2-bit codes (the INT2 workload's shape: FP16, Zipf popularity). A
call with explicit zero points takes the generic kernel and must agree too.
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
    "zipf_T1_b64": synthetic.int3_zipf(1, 64),
    "zipf_T8_b64": synthetic.int3_zipf(8, 64),
    "zipf_T8_b128": synthetic.int3_zipf(8, 128),
    "zipf_T2_b128": synthetic.int3_zipf(2, 128),
    "b32_fp16_T4": (Shape(T=4, H=512, inter=512, E=16, k=4, bits=3, block=32, dtype=FP16), R1, 41),
    # few experts: entries with two routes (pairs of MMA column groups)
    "crowded_b64_T8": (Shape(T=8, H=1024, inter=256, E=4, k=2, bits=3, block=64, dtype=BF16), R1, 42),
    # short K for fc2 (one chunk per unit): 16-row units
    "short_k_b128": (Shape(T=6, H=512, inter=256, E=8, k=3, bits=3, block=128, dtype=BF16), R1, 43),
    # mid-size T on the decode path (R < 4 E)
    "mid_T24_b64": (Shape(T=24, H=512, inter=768, E=64, k=4, bits=3, block=64, dtype=FP16), R1, 44),
    # 2-bit codes
    "int2_T8_b32": (Shape(T=8, H=2048, inter=768, E=128, k=8, bits=2, block=32, dtype=FP16),
                    Recipe(x_std=1.0, zipf_s=1.1, scale_lo=0.002, scale_hi=0.01), 45),
    "int2_T1_b64": (Shape(T=1, H=1024, inter=512, E=32, k=4, bits=2, block=64, dtype=BF16), R1, 46),
    "int2_crowded_b128": (Shape(T=6, H=512, inter=256, E=4, k=2, bits=2, block=128, dtype=FP16), R1, 47),
    "int2_mid_T20_b32": (Shape(T=20, H=768, inter=512, E=64, k=4, bits=2, block=32, dtype=BF16), R1, 48),
}


def oproblem(shape, full_softmax=0):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype, full_softmax)


@pytest.mark.parametrize("name", sorted(CASES))
def test_int23_decode_kernel(name):
    shape, recipe, seed = CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = gu.gpu_forward(shape, inp, path=1)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, name)


@pytest.mark.parametrize("name", ["zipf_T8_b64", "crowded_b64_T8", "int2_T8_b32"])
def test_int23_decode_biases_full_softmax(name):
    shape, recipe, seed = CASES[name]
    inp = synthetic.make_numpy(shape, dataclasses.replace(recipe, bias_std=0.5), seed)
    got = gu.gpu_forward_ex(shape, inp, 1, path=1)
    ref, _ = oracle.forward(oproblem(shape, 1), inp)
    gu.assert_parity(got, ref, shape.dtype, f"{name} with biases")


@pytest.mark.parametrize("name", ["zipf_T8_b64", "int2_T8_b32"])
def test_explicit_zero_points_take_the_generic_kernel(name):
    shape, recipe, seed = CASES[name]
    inp = synthetic.make_numpy(shape, dataclasses.replace(recipe, explicit_zp=True), seed)
    got = gu.gpu_forward(shape, inp, path=1)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, "explicit zero points")


def test_int3_decode_deterministic():
    shape, recipe, seed = CASES["zipf_T8_b128"]
    inp = synthetic.make_numpy(shape, recipe, seed)
    a = gu.gpu_forward(shape, inp, path=1)
    b = gu.gpu_forward(shape, inp, path=1)
    assert np.array_equal(a, b)
