"""Range edges of the FP16 operand scheme, against the oracle.

The CUDA path forms FP16 operands: BF16 block scales are converted to FP16
(or applied in FP32 after the MMA), each token's activations are scaled by the
power of two sigma_t that puts max|x_t| in [1, 2), and the SwiGLU output is
stored in FP16 times sigma_t^2. These cases feed values at the edges of those
ranges through every kernel family and compare with the oracle (FP64 from the
same bits) at the parity tolerance of the other tests:

* BF16 scales in [2^-15, 2^-13] (FP16 subnormals once converted);
* BF16 scales near 2^12 (with small activations, so that the outputs stay
  finite in BF16);
* activations N(0, 1) with a few entries of +-1e4 per token (LLM outliers);
* fc1 scales chosen so that max |h| * sigma_t^2 over the routes comes within a
  factor of a few of the FP16 maximum (2^14), and far beyond it (2^22).

The SwiGLU output is stored as h * sigma_t^2 * rho_e, rho_e a power of two
from the expert's first fc1 block scale (csrc/qmoe_internal.cuh, h_norm), so
that the FP16 intermediate keeps its magnitude when all block scales move
together; the cases above would otherwise underflow (tiny scales) or overflow
(huge scales, h beyond the FP16 maximum) there.

CPU tests: the input construction (scales and outliers land where intended).
GPU tests (-m gpu): decode kernels (tensor-copy INT4, block-scaled INT4, the
generic INT3 kernel, the decode layer kernel) and the grouped tcgen05 path.
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

FP16_MAX = 65504.0

# (shape, path, decode layer kernel): one entry per kernel family
KERNELS = {
    "decode_int4_tma": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16), 1, 0),
    "decode_int4_bs": (Shape(T=5, H=256, inter=128, E=8, k=3, bits=4, block=32, dtype=BF16), 1, 0),
    "decode_int3": (Shape(T=4, H=384, inter=256, E=6, k=2, bits=3, block=64, dtype=BF16), 1, 0),
    "decode_layer_kernel": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16), 1, 1),
    "grouped_int4": (Shape(T=200, H=256, inter=256, E=6, k=2, bits=4, block=32, dtype=BF16), 2, 0),
    "grouped_int3": (Shape(T=160, H=256, inter=256, E=5, k=2, bits=3, block=32, dtype=BF16), 2, 0),
}


def oproblem(shape):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype)


def set_scales(inp, shape, lo, hi, seed):
    """Block scales drawn log-uniform in [lo, hi], stored in the problem's dtype."""
    rng = np.random.default_rng(seed)
    out = dict(inp)
    for key in ("fc1_s", "fc2_s"):
        v = np.exp2(rng.uniform(np.log2(lo), np.log2(hi), size=inp[key].shape))
        out[key] = synthetic.float_to_bits(v, shape.dtype)
    return out


def add_outliers(inp, shape, n_per_token, magnitude, seed):
    rng = np.random.default_rng(seed)
    x = oracle.bits_to_double(inp["x"], shape.dtype)
    for t in range(shape.T):
        cols = rng.choice(shape.H, size=n_per_token, replace=False)
        x[t, cols] = magnitude * rng.choice([-1.0, 1.0], size=n_per_token)
    return dict(inp, x=synthetic.float_to_bits(x, shape.dtype))


def sigma(x_row):
    """The power of two that puts max|x_row| in [1, 2) (1 for an all-zero row)."""
    m = np.max(np.abs(x_row))
    return 1.0 if m == 0 else 2.0 ** -np.floor(np.log2(m))


def max_h_sigma2(shape, inp):
    """max over routes of |h| * sigma_t^2, from the oracle's expert FFN."""
    p = oproblem(shape)
    idx, _ = oracle.route(p, inp["logits"])
    x = oracle.bits_to_double(inp["x"], shape.dtype)
    best = 0.0
    for t in range(shape.T):
        s2 = sigma(x[t]) ** 2
        for j in range(shape.k):
            _, h, _ = oracle.expert_ffn(p, inp, int(idx[t][j]), x[t])
            best = max(best, float(np.max(np.abs(h))) * s2)
    return best


def base_inputs(shape, seed, x_std=1.0):
    return synthetic.make_numpy(shape, Recipe(x_std=x_std, logit_std=1.0, scale_lo=0.005, scale_hi=0.02), seed)


def case_inputs(case, shape, seed):
    if case == "tiny_scales":
        return set_scales(base_inputs(shape, seed), shape, 2.0 ** -15, 2.0 ** -13, seed + 1)
    if case == "huge_scales":
        # scales up to 2^12 with activations ~N(0, 2^-12): outputs of order one
        return set_scales(base_inputs(shape, seed, x_std=2.0 ** -12), shape, 2.0 ** 11, 2.0 ** 12, seed + 1)
    if case == "outliers":
        return add_outliers(base_inputs(shape, seed), shape, 3, 1.0e4, seed + 1)
    if case in ("h_near_fp16_max", "h_beyond_fp16_max"):
        # scale every fc1 block scale by one factor so that max |h| sigma^2 lands near
        # 2^14 (a quarter of the FP16 maximum) or 2^22
        inp = base_inputs(shape, seed)
        m = max_h_sigma2(shape, inp)
        target = 2.0 ** 14 if case == "h_near_fp16_max" else 2.0 ** 22
        f = np.sqrt(target / m)          # h is quadratic in the weights
        s1 = oracle.bits_to_double(inp["fc1_s"], shape.dtype) * f
        return dict(inp, fc1_s=synthetic.float_to_bits(s1, shape.dtype))
    raise ValueError(case)


CASES = ["tiny_scales", "huge_scales", "outliers", "h_near_fp16_max", "h_beyond_fp16_max"]


@pytest.mark.parametrize("case", CASES)
def test_inputs_reach_the_edges(case):
    """The constructed inputs sit where the case says (checked on the oracle side)."""
    shape = KERNELS["decode_int4_bs"][0]
    inp = case_inputs(case, shape, 11)
    s = oracle.bits_to_double(inp["fc1_s"], shape.dtype)
    x = oracle.bits_to_double(inp["x"], shape.dtype)
    if case == "tiny_scales":
        assert s.min() >= 2.0 ** -15 * 0.99 and s.max() <= 2.0 ** -13
        assert (s < 2.0 ** -14).mean() > 0.3      # many are FP16 subnormals
    elif case == "huge_scales":
        assert s.max() <= 2.0 ** 12 and s.min() >= 2.0 ** 11 * 0.99
    elif case == "outliers":
        assert (np.abs(x) > 9.9e3).sum() == 3 * shape.T      # 1e4 rounds to 9984 in BF16
    elif case == "h_near_fp16_max":
        m = max_h_sigma2(shape, inp)
        assert 2.0 ** 12 < m < FP16_MAX
    else:
        assert max_h_sigma2(shape, inp) > 2.0 ** 20


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("case", CASES)
def test_range_edge_parity(case, kernel):
    import torch

    import quantized_mixture_experts_route_gb300 as qm

    shape, path, layer_kernel = KERNELS[kernel]
    inp = case_inputs(case, shape, 21)
    ref, _ = oracle.forward(oproblem(shape), inp)
    if layer_kernel:
        p = gu.problem(shape, path)
        d = gu.device_inputs(inp)
        ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
        qm.qmoe_forward_ex(p, 0, None, None, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"],
                           d["fc2_s"], None, out, ws, decode_layer_kernel=1)
        torch.cuda.synchronize()
        got = out.cpu().numpy().view(np.uint16)
    else:
        got = gu.gpu_forward(shape, inp, path=path)
    gu.assert_parity(got, ref, shape.dtype, f"{case} / {kernel}")
