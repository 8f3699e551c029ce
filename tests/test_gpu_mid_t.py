"""Mid-size batches (9 <= T <= 512): the decode path's weights-stationary
kernels with an expert's routes on the MMA N side, and the switch to the
grouped GEMM on the route count.

AUTO runs the decode path for T <= 8 and, up to 64 tokens and 512 routes, while
the routes number fewer than 64 or fewer than 4 per expert (the pages switch
from their tensor-core GEMV to the grouped GEMM at num_r >= 64 && num_r >= 4E,
"[CUDA] Enable Tensor-Core INT3/INT4 QMoE offload ..." #33731 text, item 3);
the grouped GEMM above that. On the decode path the generic kernel (INT2, INT3,
other blocks) takes an expert's routes in chunks of up to 8 per MMA N-fragment,
and the INT4 block-32 kernels take them in pairs of block columns; the chunks
and pairs of one expert run side by side, so its weight rows come from HBM
once and from L2 for the others.

Every case compares with the oracle: whole outputs up to T = 64, sampled
tokens at T = 256 and 512 (the oracle computes them one by one), the INT4
decode-stack shape and the INT3 Zipf workload (block 64), both paths forced at
mid T, an expert with many chunks on the generic kernel, the block-scaled INT4
kernel and the decode layer kernel.
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def oproblem(shape):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype)


def check(shape, inp, path=0, n_sample=None, label="", **kw):
    got = gu.gpu_forward(shape, inp, path=path) if not kw else kw["run"](shape, inp)
    if n_sample is None:
        ref, _ = oracle.forward(oproblem(shape), inp)
        gu.assert_parity(got, ref, shape.dtype, label)
        return got
    rng = np.random.default_rng(shape.T)
    toks = np.unique(np.concatenate([rng.choice(shape.T, size=n_sample, replace=False), [0, shape.T - 1]]))
    ref, _ = oracle.forward(oproblem(shape), inp, tokens=toks)
    gu.assert_parity(got[toks], ref, shape.dtype, label)
    return got


@pytest.mark.parametrize("T", [9, 16, 64, 256, 512])
def test_decode_stack_shape_auto(T):
    shape, recipe, seed = synthetic.decode_layer(T)
    inp = synthetic.make_numpy(shape, recipe, seed)
    check(shape, inp, n_sample=None if T <= 64 else 40, label=f"INT4 T={T}")


@pytest.mark.parametrize("T", [9, 16, 64, 256, 512])
def test_int3_zipf_auto(T):
    shape, recipe, seed = synthetic.int3_zipf(T, 64)
    inp = synthetic.make_numpy(shape, recipe, seed)
    check(shape, inp, n_sample=None if T <= 64 else 40, label=f"INT3 Zipf T={T}")


@pytest.mark.parametrize("T", [16, 32, 63])
def test_mid_t_both_paths(T):
    """The same mid-size batch on the decode path and on the grouped path."""
    shape, recipe, seed = synthetic.decode_layer(T)
    inp = synthetic.make_numpy(shape, recipe, seed)
    a = check(shape, inp, path=1, label=f"decode path T={T}")
    b = check(shape, inp, path=2, label=f"grouped path T={T}")
    fa, fb = gu.to_f64(a, shape.dtype), gu.to_f64(b, shape.dtype)
    assert np.linalg.norm(fa - fb) / np.linalg.norm(fb) < 2e-3


# an expert with many routes on the decode path: several 8-route chunks (generic
# kernel) or many route pairs (INT4 kernels)
CROWDED = {
    "int3_chunks": (Shape(T=40, H=384, inter=256, E=4, k=2, bits=3, block=64, dtype=BF16), 81),
    "int2_zp_chunks": (Shape(T=64, H=256, inter=192, E=3, k=2, bits=2, block=32, dtype=FP16), 82),
    "int4_b64_chunks": (Shape(T=33, H=512, inter=256, E=5, k=3, bits=4, block=64, dtype=BF16), 83),
    "int4_tma_pairs": (Shape(T=48, H=512, inter=512, E=6, k=4, bits=4, block=32, dtype=BF16), 84),
    "int4_bs_pairs": (Shape(T=24, H=384, inter=128, E=4, k=2, bits=4, block=32, dtype=FP16), 85),
}


@pytest.mark.parametrize("name", sorted(CROWDED))
def test_crowded_experts_on_the_decode_path(name):
    shape, seed = CROWDED[name]
    recipe = Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=name.startswith("int2"))
    inp = synthetic.make_numpy(shape, recipe, seed)
    check(shape, inp, path=1, label=name)


@pytest.mark.parametrize("T", [16, 40])
def test_decode_layer_kernel_mid_t(T):
    import torch

    import quantized_mixture_experts_route_gb300 as qm

    shape, recipe, seed = synthetic.decode_layer(T)
    inp = synthetic.make_numpy(shape, recipe, seed)

    def run(shape, inp):
        p = gu.problem(shape, 1)
        d = gu.device_inputs(inp)
        ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
        qm.qmoe_forward_ex(p, 0, None, None, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"],
                           d["fc2_s"], None, out, ws, decode_layer_kernel=1)
        torch.cuda.synchronize()
        return out.cpu().numpy().view(np.uint16)

    check(shape, inp, label=f"decode layer kernel T={T}", run=run)
