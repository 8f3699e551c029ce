"""qmoe_forward_ex: FC1 / FC2 biases and full-softmax routing weights
(normalize_routing_weights = 0), against the oracle with the same options.

CPU tests: the option checks that happen on the host before any launch. GPU
tests (-m gpu): every decode kernel (tensor-copy INT4, block-scaled INT4,
generic INT2/INT3) and the grouped tcgen05 path, within the parity tolerance of
the other GPU tests; and qmoe_forward_ex with zeroed options equals qmoe_forward
bit for bit.
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

# name: (shape, recipe, seed, path, full_softmax)
CASES = {
    # decode, tensor-copy INT4 kernel (K of both matmuls a multiple of 256)
    "tma_bias": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16),
                 Recipe(logit_std=2.0, scale_lo=0.002, scale_hi=0.01, bias_std=0.5), 71, 1, 0),
    "tma_full_softmax": (Shape(T=6, H=512, inter=512, E=12, k=3, bits=4, block=32, dtype=FP16),
                         Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 72, 1, 1),
    # decode, block-scaled INT4 kernel (inter not a multiple of 256)
    "bs_bias_full": (Shape(T=5, H=256, inter=128, E=8, k=3, bits=4, block=32, dtype=FP16),
                     Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, bias_std=0.5), 73, 1, 1),
    # decode, generic kernel (INT3 block 64, INT2 with zero points)
    "gemv_int3_bias_full": (Shape(T=4, H=384, inter=256, E=6, k=2, bits=3, block=64, dtype=BF16),
                            Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, bias_std=0.5), 74, 1, 1),
    "gemv_int2_zp_bias": (Shape(T=6, H=160, inter=224, E=12, k=5, bits=2, block=32, dtype=BF16),
                          Recipe(logit_std=1.0, scale_lo=0.01, scale_hi=0.05, explicit_zp=True,
                                 bias_std=0.5), 75, 1, 0),
    # grouped tcgen05 path
    "grouped_int4_bias": (Shape(T=300, H=256, inter=192, E=8, k=2, bits=4, block=32, dtype=BF16),
                          Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, bias_std=0.5), 76, 2, 0),
    "grouped_int2_bias_full": (Shape(T=200, H=320, inter=256, E=5, k=2, bits=2, block=32, dtype=FP16),
                               Recipe(logit_std=1.0, scale_lo=0.01, scale_hi=0.04, bias_std=0.5), 77, 2, 1),
    "grouped_int3_full": (Shape(T=260, H=256, inter=256, E=5, k=2, bits=3, block=32, dtype=BF16),
                          Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 78, 2, 1),
    # route tiles with fc1 biases: the epilogue takes a tile's biases from the lanes of
    # one per-tile load; fc1 N = 640 and fc2 N = 448 end in part-filled 256-row tiles
    "tiles_int4_bias_fp16_tail": (Shape(T=250, H=448, inter=320, E=6, k=3, bits=4, block=32, dtype=FP16),
                                  Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, bias_std=0.5), 79, 3, 0),
    # INT3 route tiles: 128-row weight tiles (lanes 0-15 hold the tile's biases)
    "tiles_int3_bias_full": (Shape(T=260, H=384, inter=384, E=5, k=2, bits=3, block=128, dtype=BF16),
                             Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, bias_std=0.5), 80, 3, 1),
}


def oproblem(shape, full_softmax):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype, full_softmax)


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qm.lib()


def _call(L, p, full_softmax, b1=None, b2=None):
    opt = qm.qmoe_options(full_softmax, b1, b2)
    return L.qmoe_forward_ex(ctypes.byref(p), ctypes.byref(opt), *([16] * 9), 16, 1 << 30, None)


def test_invalid_full_softmax_rejected_on_host(L):
    p = qm.problem(4, 256, 128, 8, 2, 4, 32, BF16)
    assert _call(L, p, 2) == qm.QMOE_ERR_INVALID_ARGUMENT
    assert _call(L, p, -1) == qm.QMOE_ERR_INVALID_ARGUMENT


def test_misaligned_bias_rejected_on_host(L):
    p = qm.problem(4, 256, 128, 8, 2, 4, 32, BF16)
    assert _call(L, p, 0, b1=18) == qm.QMOE_ERR_MISALIGNED
    assert _call(L, p, 1, b2=34) == qm.QMOE_ERR_MISALIGNED


def test_empty_batch_with_options(L):
    p = qm.problem(0, 256, 128, 8, 2, 4, 32, BF16)
    assert _call(L, p, 1, b1=32, b2=64) == qm.QMOE_OK
    # a null options pointer means the defaults
    assert L.qmoe_forward_ex(ctypes.byref(p), None, *([None] * 10), 0, None) == qm.QMOE_OK


def test_options_struct_layout():
    # int32, two pointers, int32, three pointers: offsets 0, 8, 16, 24, 32, 40, 48; 56 bytes on LP64 hosts
    assert qm.qmoe_options.fc1_bias.offset == 8 and qm.qmoe_options.fc2_bias.offset == 16
    assert qm.qmoe_options.decode_layer_kernel.offset == 24 and qm.qmoe_options.router_weight.offset == 32
    assert qm.qmoe_options.fc1_global_scale.offset == 40 and qm.qmoe_options.fc2_global_scale.offset == 48
    assert ctypes.sizeof(qm.qmoe_options) == 56
    # the problem: int64, nine int32 (the last the weight format)
    assert qm.qmoe_problem.format.offset == 40 and ctypes.sizeof(qm.qmoe_problem) == 48


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_options_parity(name):
    shape, recipe, seed, path, full = CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = gu.gpu_forward_ex(shape, inp, full, path=path)
    ref, _ = oracle.forward(oproblem(shape, full), inp)
    gu.assert_parity(got, ref, shape.dtype, name)


@pytest.mark.gpu
@pytest.mark.parametrize("path", [1, 2])
def test_zero_options_equal_forward(path):
    import torch

    shape = Shape(T=8 if path == 1 else 64, H=512, inter=256, E=8, k=2, bits=4, block=32, dtype=BF16)
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 79)
    a = gu.gpu_forward(shape, inp, path=path)
    b = gu.gpu_forward_ex(shape, inp, 0, path=path)
    assert np.array_equal(a, b)
    # a null options pointer: the same call
    p = gu.problem(shape, path)
    d = gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    args = [d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"], d["fc2_s"], None, out, ws]
    st = qm.lib().qmoe_forward_ex(ctypes.byref(p), None, *[None if t is None else t.data_ptr() for t in args],
                                  ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == qm.QMOE_OK
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), a)


@pytest.mark.gpu
def test_full_softmax_nan_logit_row():
    """A NaN logit (never selected) makes that token's full-softmax weights, and so
    its output row, NaN on both sides; the other tokens stay within parity."""
    shape = Shape(T=4, H=256, inter=128, E=8, k=2, bits=4, block=32, dtype=BF16)
    inp = synthetic.make_numpy(shape, Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 80)
    lg = inp["logits"].copy()
    lg[2, 5] = 0x7FC0
    inp = dict(inp, logits=lg)
    got = gu.gpu_forward_ex(shape, inp, 1, path=1)
    ref, _ = oracle.forward(oproblem(shape, 1), inp)

    def nan(b):
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)

    assert nan(got[2]).all() and nan(ref[2]).all()
    keep = [0, 1, 3]
    gu.assert_parity(got[keep], ref[keep], shape.dtype, "rows without a NaN logit")
