"""Router logits ahead of routing (qmoe_router_logits, qmoe_options.router_weight)
against the oracle.

The router GEMM sums in FP32 on the tensor cores and rounds each logit once;
the oracle sums in double and rounds once, so a logit may differ by one unit in
the last place where the exact sum sits near a rounding boundary. The tests
bound that (every logit within one unit, almost all equal) and take the
routing decision on both sides from the same logits: the forward with a router
weight is compared with the oracle forward on the GPU's logits, and with the
library's own forward on those logits bit for bit.

CPU tests: argument checks on the host. GPU tests (-m gpu): decode and prefill
batch sizes, both dtypes, expert counts that are not multiples of the 32-expert
tile, NaN inputs, both kernel paths.
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

FAKE = 1 << 20


def test_router_logits_host_checks():
    qbuild.build()
    L = qm.lib()
    p = qm.problem(8, 256, 128, 16, 2, 4, 32, BF16)
    assert L.qmoe_router_logits(ctypes.byref(p), None, FAKE, FAKE, None) == qm.QMOE_ERR_INVALID_ARGUMENT
    assert L.qmoe_router_logits(ctypes.byref(p), FAKE, None, FAKE, None) == qm.QMOE_ERR_INVALID_ARGUMENT
    assert L.qmoe_router_logits(ctypes.byref(p), FAKE, FAKE + 2, FAKE, None) == qm.QMOE_ERR_MISALIGNED
    bad = qm.problem(8, 250, 128, 16, 2, 4, 32, BF16)
    assert L.qmoe_router_logits(ctypes.byref(bad), FAKE, FAKE, FAKE, None) == qm.QMOE_ERR_UNSUPPORTED
    empty = qm.problem(0, 256, 128, 16, 2, 4, 32, BF16)
    assert L.qmoe_router_logits(ctypes.byref(empty), None, None, None, None) == qm.QMOE_OK


def router_weight(E, H, dtype, seed, std=0.05):
    rng = np.random.default_rng(seed)
    return synthetic.float_to_bits(rng.standard_normal((E, H)) * std, dtype)


def gpu_router_logits(shape, x_bits, w_bits):
    import torch

    p = gu.problem(shape)
    out = torch.empty((shape.T, shape.E), dtype=torch.int16, device="cuda")
    qm.qmoe_router_logits(p, gu.dev(x_bits), gu.dev(w_bits), out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def ulp_distance(a, b, dtype):
    """Distance in units of the last place between two arrays of finite 16-bit values."""
    def key(v):
        v = v.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)
    return np.abs(key(a) - key(b))


def check_logits(got, ref, x_bits, w_bits, dtype, label):
    """Every logit within one unit in the last place of the oracle's, plus the error
    bound of an FP32 sum of H products (H 2^-24 sum |x_h w_h|, which matters where
    the sum cancels to near zero); almost all of them equal."""
    g, r = oracle.bits_to_double(got, dtype), oracle.bits_to_double(ref, dtype)
    xa = np.abs(oracle.bits_to_double(x_bits, dtype))
    wa = np.abs(oracle.bits_to_double(w_bits, dtype))
    H = xa.shape[1]
    bound = H * 2.0 ** -24 * (xa @ wa.T)
    ulp = np.abs(oracle.bits_to_double((ref.astype(np.int32) + 1).astype(np.uint16), dtype) - r)
    assert (np.abs(g - r) <= ulp + bound).all(), f"{label}: a logit outside one unit plus the FP32 sum bound"
    d = ulp_distance(got, ref, dtype)
    assert (d == 0).mean() >= 0.98, f"{label}: {(d != 0).mean():.3%} of the logits differ"


SHAPES = {
    "decode_T8": (Shape(T=8, H=2048, inter=768, E=128, k=8, bits=4, block=32, dtype=BF16), 91),
    "decode_T1_fp16": (Shape(T=1, H=512, inter=256, E=40, k=4, bits=4, block=32, dtype=FP16), 92),
    "mid_T33_E100": (Shape(T=33, H=1024, inter=256, E=100, k=6, bits=4, block=32, dtype=BF16), 93),
    "prefill_T1000": (Shape(T=1000, H=2048, inter=768, E=128, k=8, bits=4, block=32, dtype=BF16), 94),
    "tiny_E8": (Shape(T=5, H=64, inter=32, E=8, k=2, bits=4, block=32, dtype=FP16), 95),
    # the tiled GEMM with 32-token tiles, H not a multiple of 128
    "gemm_k64_T200": (Shape(T=200, H=320, inter=128, E=64, k=4, bits=4, block=32, dtype=BF16), 96),
    # 64-token tiles, a ragged token tail and E above one 128-expert block
    "gemm_T4100_E160": (Shape(T=4100, H=1024, inter=256, E=160, k=8, bits=4, block=32, dtype=BF16), 98),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_router_logits_match_the_oracle(name):
    shape, seed = SHAPES[name]
    inp = synthetic.make_activations(shape, Recipe(), seed)
    w = router_weight(shape.E, shape.H, shape.dtype, seed + 1)
    got = gpu_router_logits(shape, inp["x"], w)
    p = oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block, shape.dtype)
    ref = oracle.router_logits(p, inp["x"], w)
    check_logits(got, ref, inp["x"], w, shape.dtype, name)


@pytest.mark.gpu
def test_router_logits_at_8k_tokens_sampled():
    """The prefill size, in the launch configuration of the default call; sampled
    tokens against the oracle."""
    shape, recipe, seed = synthetic.prefill_8k()
    inp = synthetic.make_activations(shape, recipe, seed)
    w = router_weight(shape.E, shape.H, shape.dtype, 7)
    got = gpu_router_logits(shape, inp["x"], w)
    rng = np.random.default_rng(3)
    toks = np.unique(np.concatenate([rng.choice(shape.T, 64, replace=False), [0, shape.T - 1]]))
    p = oracle.Problem(len(toks), shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block, shape.dtype)
    ref = oracle.router_logits(p, inp["x"][toks], w)
    check_logits(got[toks], ref, inp["x"][toks], w, shape.dtype, "prefill 8K")


@pytest.mark.gpu
def test_router_logits_nan_stays_in_its_token():
    shape, seed = SHAPES["tiny_E8"]
    inp = synthetic.make_activations(shape, Recipe(), seed)
    x = inp["x"].copy()
    x[2, 7] = 0x7E00   # FP16 NaN
    got = gpu_router_logits(shape, x, router_weight(shape.E, shape.H, shape.dtype, 3))
    nan = ((got & 0x7C00) == 0x7C00) & ((got & 0x3FF) != 0)
    assert nan[2].all() and not np.delete(nan, 2, axis=0).any()


@pytest.mark.gpu
@pytest.mark.parametrize("name,path", [("decode_T8", 0), ("mid_T33_E100", 0), ("prefill_T1000", 0),
                                       ("tiny_E8", 0), ("mid_T33_E100", 2)])
def test_forward_with_router_weight(name, path):
    """forward_ex with a router weight equals the forward on the logits that
    qmoe_router_logits returns (bit for bit), and matches the oracle forward on
    those logits."""
    import torch

    shape, seed = SHAPES[name]
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), seed)
    w = router_weight(shape.E, shape.H, shape.dtype, seed + 1, std=0.3)
    logits = gpu_router_logits(shape, inp["x"], w)
    p = gu.problem(shape, path)
    d = gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward_ex(p, 0, None, None, d["x"], None, d["fc1_q"], d["fc1_s"], None, d["fc2_q"], d["fc2_s"],
                       None, out, ws, router_weight=gu.dev(w))
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    with_logits = dict(inp, logits=logits)
    assert np.array_equal(got, gu.gpu_forward(shape, with_logits, path=path))
    ref, _ = oracle.forward(oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits,
                                           shape.block, shape.dtype), with_logits)
    gu.assert_parity(got, ref, shape.dtype, f"{name} with router weight")
