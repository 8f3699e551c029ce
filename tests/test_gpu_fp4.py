"""MXFP4 and NVFP4 experts (qmoe_problem.format) against the oracle, on the
decode path and on the grouped tcgen05 path.

The E2M1 codes become FP16 pairs through a byte-permute table, times the block
scale in FP16: E4M3 scales are exact in FP16; E8M0 scales are carried relative
to the expert's first one and that power of two, like the NVFP4 global scale,
is applied in FP32 by the epilogue. On the decode path they run on the decode
layer kernel (or the generic kernel through the stage calls); on the grouped
path the dequantisers form the same FP16 pairs for tcgen05.

CPU tests: the host checks of the formats. GPU tests (-m gpu): decode and
mid-size batches, both dtypes, the decode-stack shape, E8M0 scales far from 1
and spread over a few powers of two, NVFP4 with and without global scales.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

qm = pytest.importorskip("quantized_mixture_experts_route_gb300")
from quantized_mixture_experts_route_gb300 import build as qbuild  # noqa: E402

MX, NV = qm.QMOE_FORMAT_MXFP4, qm.QMOE_FORMAT_NVFP4


def P(T=8, fmt=MX, block=None, path=0, bits=4):
    block = block or (32 if fmt == MX else 16)
    return qm.problem(T, 512, 256, 16, 4, bits, block, BF16, path, fmt)


def test_fp4_host_checks():
    qbuild.build()
    L = qm.lib()
    ws = lambda p: L.qmoe_workspace_bytes(ctypes.byref(p))
    assert ws(P(fmt=MX)) > 0 and ws(P(fmt=NV)) > 0
    assert ws(P(fmt=MX, block=16)) == 0 and ws(P(fmt=NV, block=32)) == 0   # the formats fix the block
    assert ws(P(fmt=MX, bits=3)) == 0
    assert ws(P(fmt=MX, path=qm.QMOE_PATH_GROUPED)) > 0                    # both paths
    assert ws(P(T=200, fmt=NV)) > 0
    assert ws(qm.problem(8, 512, 256, 16, 4, 4, 32, BF16, 0, 3)) == 0       # unknown format
    # a zero point with an FP4 format is an argument error, found before any launch
    F = 1 << 20
    args = [F] * 10
    args[2] = F  # fc1_zp
    p = P(fmt=MX)
    assert L.qmoe_forward(ctypes.byref(p), F, F, F, F, F, F, F, None, F, F, 1 << 40, None) == \
        qm.QMOE_ERR_INVALID_ARGUMENT


def oproblem(shape, inp):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype, 0, shape.format, inp.get("g1"), inp.get("g2"))


def fp4_forward(shape, inp, use_global=True):
    import torch

    p = gu.problem(shape)
    d = gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    g1 = d.get("g1") if use_global else None
    g2 = d.get("g2") if use_global else None
    qm.qmoe_forward_ex(p, 0, None, None, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"],
                       d["fc2_s"], None, out, ws, fc1_global_scale=g1, fc2_global_scale=g2)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


CASES = {
    "mx_T8": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16, format=1), 101),
    "mx_T1_fp16": (Shape(T=1, H=256, inter=512, E=8, k=2, bits=4, block=32, dtype=FP16, format=1), 102),
    "mx_T33_mid": (Shape(T=33, H=512, inter=256, E=12, k=3, bits=4, block=32, dtype=BF16, format=1), 103),
    "nv_T8": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=16, dtype=BF16, format=2), 104),
    "nv_T5_fp16": (Shape(T=5, H=384, inter=128, E=6, k=2, bits=4, block=16, dtype=FP16, format=2), 105),
    "nv_T40_mid": (Shape(T=40, H=256, inter=256, E=8, k=2, bits=4, block=16, dtype=BF16, format=2), 106),
    "mx_grouped_T300": (Shape(T=300, H=512, inter=256, E=8, k=2, bits=4, block=32, dtype=BF16, format=1), 109),
    "nv_grouped_T260_fp16": (Shape(T=260, H=256, inter=320, E=6, k=3, bits=4, block=16, dtype=FP16, format=2), 110),
    "mx_decode_stack": (Shape(T=8, H=2048, inter=768, E=128, k=8, bits=4, block=32, dtype=BF16, format=1), 107),
    "nv_decode_stack": (Shape(T=8, H=2048, inter=768, E=128, k=8, bits=4, block=16, dtype=BF16, format=2), 108),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_fp4_parity(name):
    shape, seed = CASES[name]
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0), seed)
    got = fp4_forward(shape, inp)
    ref, _ = oracle.forward(oproblem(shape, inp), inp)
    gu.assert_parity(got, ref, shape.dtype, name)


@pytest.mark.gpu
def test_nvfp4_without_global_scales():
    """NULL global scale pointers mean 1 on both sides."""
    shape, seed = CASES["nv_T8"]
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0), seed)
    got = fp4_forward(shape, inp, use_global=False)
    ref, _ = oracle.forward(oproblem(shape, dict(inp, g1=None, g2=None)), dict(inp, g1=None, g2=None))
    gu.assert_parity(got, ref, shape.dtype, "NVFP4 without global scales")


@pytest.mark.gpu
@pytest.mark.parametrize("lo,hi", [(127 - 40, 127 - 36), (127 + 20, 127 + 24)])
def test_mxfp4_scales_far_from_one(lo, hi):
    """E8M0 scales of 2^-40 .. 2^-36 or 2^20 .. 2^24, spread over four powers of
    two inside an expert (outside the FP16 range as such); activations scaled so
    that the outputs stay finite."""
    shape, seed = CASES["mx_T8"]
    rng = np.random.default_rng(7)
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0, x_std=1.0 if lo < 127 else 2.0 ** -40), seed)
    for key in ("fc1_s", "fc2_s"):
        inp[key] = rng.integers(lo, hi + 1, size=inp[key].shape, dtype=np.uint8)
    got = fp4_forward(shape, inp)
    ref, _ = oracle.forward(oproblem(shape, inp), inp)
    gu.assert_parity(got, ref, shape.dtype, f"MXFP4 scales 2^{lo - 127}..2^{hi - 127}")


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mx_T8", "nv_T8", "mx_T33_mid"])
def test_fp4_generic_kernel_through_stages(name):
    """The stages one by one run the generic decode kernel for fc1 and fc2 (the
    whole call runs the decode layer kernel for these shapes); NVFP4 without
    global scales there (the stage calls take no options)."""
    import torch

    shape, seed = CASES[name]
    inp = dict(synthetic.make_numpy(shape, Recipe(logit_std=1.0), seed), g1=None, g2=None)
    p = gu.problem(shape)
    d = gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    for st in range(4):
        qm.qmoe_forward_stages(p, st, st, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"],
                               d["fc2_s"], None, out, ws)
    torch.cuda.synchronize()
    staged = out.cpu().numpy().view(np.uint16)
    ref, _ = oracle.forward(oproblem(shape, inp), inp)
    gu.assert_parity(staged, ref, shape.dtype, f"{name} (generic kernel)")
    whole = fp4_forward(shape, inp, use_global=False)
    gu.assert_parity(whole, ref, shape.dtype, f"{name} (layer kernel)")


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mx_T8", "nv_T8", "mx_grouped_T300"])
def test_fp4_with_biases_full_softmax_and_router(name):
    """The FP4 formats with the other options: FC1/FC2 biases, full-softmax
    routing weights and router logits computed from a router weight; against
    the oracle on the GPU's own logits (the routing decision taken from the same
    values on both sides)."""
    import torch

    shape, seed = CASES[name]
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0, bias_std=0.5), seed)
    rng = np.random.default_rng(seed + 7)
    w_router = synthetic.float_to_bits(rng.standard_normal((shape.E, shape.H)) * 0.3, shape.dtype)
    p = gu.problem(shape)
    d = gu.device_inputs(inp)
    logits = torch.empty((shape.T, shape.E), dtype=torch.int16, device="cuda")
    qm.qmoe_router_logits(p, d["x"], gu.dev(w_router), logits)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward_ex(p, 1, d["fc1_b"], d["fc2_b"], d["x"], None, d["fc1_q"], d["fc1_s"], None, d["fc2_q"],
                       d["fc2_s"], None, out, ws, router_weight=gu.dev(w_router),
                       fc1_global_scale=d.get("g1"), fc2_global_scale=d.get("g2"))
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    with_logits = dict(inp, logits=logits.cpu().numpy().view(np.uint16))
    op = oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block, shape.dtype, 1,
                        shape.format, inp.get("g1"), inp.get("g2"))
    ref, _ = oracle.forward(op, with_logits)
    gu.assert_parity(got, ref, shape.dtype, f"{name} with options")
