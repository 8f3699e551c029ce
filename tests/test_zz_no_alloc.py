"""qmoe_forward_decode_static: the decode-path forward whose workspace is the
library's own fixed device array (no allocation in the call).

The CPU tests check the host-side rejections, which come before any CUDA call.
The GPU test calls the entry point through the C ABI several times in a row, on
layers of different sizes (T = 8 with 128 experts and top-8, then T = 1 with 4
experts and top-2, then T = 5), with no synchronisation between the calls, so a
value one call leaves in the shared array would reach the next. Each output is
compared with qmoe_forward's on the same inputs bit for bit (the same kernels
run) and with the oracle within the parity tolerance of the other GPU tests.
This file is collected last, so the GPU test also runs after the rest of the
suite has used the library in the same process.
"""
import os

import numpy as np
import pytest

import synthetic
from tests import gpu_util as gu
from tests.conftest import ROOT

qm = pytest.importorskip("quantized_mixture_experts_route_gb300")
from quantized_mixture_experts_route_gb300 import build as qbuild  # noqa: E402


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return qm.lib()


def _status(L, p):
    import ctypes

    return L.qmoe_forward_decode_static(ctypes.byref(p), *([None] * 9), None)


def test_static_limit_rejected_on_host(L):
    # T=8, E=512, top-k=32, H=I=8192 needs more than the 8 MiB array
    p = qm.problem(8, 8192, 8192, 512, 32, 4, 32, gu.BF16, qm.QMOE_PATH_DECODE)
    assert qm.qmoe_workspace_bytes(p) > qm.QMOE_STATIC_WORKSPACE_BYTES
    assert _status(L, p) == qm.QMOE_ERR_WORKSPACE_TOO_SMALL


def test_grouped_path_rejected_on_host(L):
    p = qm.problem(64, 256, 128, 8, 2, 4, 32, gu.BF16, qm.QMOE_PATH_AUTO)
    assert _status(L, p) == qm.QMOE_ERR_UNSUPPORTED
    p = qm.problem(4, 256, 128, 8, 2, 4, 32, gu.BF16, qm.QMOE_PATH_GROUPED)
    assert _status(L, p) == qm.QMOE_ERR_UNSUPPORTED


def test_invalid_problem_and_empty_batch(L):
    p = qm.problem(4, 250, 128, 8, 2, 4, 32, gu.BF16, qm.QMOE_PATH_AUTO)   # H not a block multiple
    assert _status(L, p) == qm.QMOE_ERR_UNSUPPORTED
    p = qm.problem(0, 256, 128, 8, 2, 4, 32, gu.BF16, qm.QMOE_PATH_AUTO)
    assert _status(L, p) == qm.QMOE_OK


def test_source_allocates_nothing():
    src = open(os.path.join(ROOT, "quantized_mixture_experts_route_gb300", "csrc", "noalloc.cu")).read()
    code = "\n".join(line.split("//")[0] for line in src.splitlines())
    for call in ("cudaMalloc", "cudaFree", "cudaMallocAsync", "cudaHostAlloc", "new ", "malloc("):
        assert call not in code, call


@pytest.mark.gpu
def test_static_matches_forward_and_oracle_calls_in_a_row(L):
    import torch

    import oracle
    from synthetic import BF16, FP16, Recipe, Shape

    layers = [synthetic.decode_layer(8, 0),
              (Shape(T=1, H=256, inter=256, E=4, k=2, bits=4, block=32, dtype=BF16),
               Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 91),
              (Shape(T=5, H=512, inter=384, E=16, k=4, bits=4, block=32, dtype=FP16),
               Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 92),
              synthetic.decode_layer(8, 1)]
    cases = []
    for shape, recipe, seed in layers:
        inp = synthetic.make_numpy(shape, recipe, seed)
        d = gu.device_inputs(inp)
        ref = gu.gpu_forward(shape, inp, d=d)
        out = torch.full((shape.T, shape.H), -1, dtype=torch.int16, device="cuda")
        cases.append((shape, inp, d, ref, out))
    torch.cuda.synchronize()
    for shape, _, d, _, out in cases:      # calls in a row, no synchronisation between them
        qm.qmoe_forward_decode_static(gu.problem(shape), d["x"], d["logits"], d["fc1_q"], d["fc1_s"],
                                      d.get("fc1_zp"), d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out)
    torch.cuda.synchronize()
    for i, (shape, inp, _, ref, out) in enumerate(cases):
        got = out.cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ref), f"static call {i} differs from qmoe_forward"
        want, _ = oracle.forward(oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits,
                                                shape.block, shape.dtype), inp)
        gu.assert_parity(got, want, shape.dtype, f"static call {i} against the oracle")
