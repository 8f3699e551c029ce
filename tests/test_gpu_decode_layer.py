"""The decode layer kernel (fc1 + SwiGLU and fc2 in one persistent launch,
qmoe_options.decode_layer_kernel = 1) against the oracle and against the
separate stage kernels (the default); the workspace's failure word and the NaN
output it causes; guard bands.

CPU test: the failure word's offset from the C ABI. GPU tests (-m gpu): the
kernel runs when asked for on a decode-path call with INT4, block 32, no zero
points and hidden, inter multiples of 256; the separate kernels run otherwise.
"""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

qm = pytest.importorskip("quantized_mixture_experts_route_gb300")
from quantized_mixture_experts_route_gb300 import build as qbuild  # noqa: E402


def layer_forward(shape, inp, d=None, ws=None, out=None):
    """qmoe_forward_ex with the decode layer kernel."""
    import torch

    p = gu.problem(shape)
    d = d or gu.device_inputs(inp)
    if ws is None:
        ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    if out is None:
        out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward_ex(p, 0, None, None, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], d.get("fc1_zp"),
                       d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out, ws, decode_layer_kernel=1)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def oproblem(shape):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype)


CASES = {
    "decode_T1": synthetic.decode_layer(1),
    "decode_T3": synthetic.decode_layer(3),
    "decode_T8": synthetic.decode_layer(8),
    # few experts: every expert has several routes, so several decode-table entries
    "crowded_fp16": (Shape(T=8, H=768, inter=512, E=3, k=3, bits=4, block=32, dtype=FP16),
                     Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 52),
    "small_bf16": (Shape(T=3, H=256, inter=256, E=4, k=2, bits=4, block=32, dtype=BF16),
                   Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 51),
    # k = E: every token reaches every expert
    "k_equals_E": (Shape(T=5, H=512, inter=256, E=6, k=6, bits=4, block=32, dtype=BF16),
                   Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 61),
    # long K of fc1 (32 stages per unit) and wide top-k
    "long_k_wide_topk": (Shape(T=2, H=8192, inter=256, E=64, k=32, bits=4, block=32, dtype=BF16),
                         Recipe(logit_std=1.0, scale_lo=0.002, scale_hi=0.01), 62),
}


def test_error_offset_from_the_abi():
    qbuild.build()
    p = gu.problem(CASES["decode_T8"][0])
    off = qm.qmoe_workspace_error_offset(p)
    assert 0 <= off < qm.qmoe_workspace_bytes(p) and off % 4 == 0
    bad = qm.problem(4, 250, 128, 8, 2, 4, 32, BF16)
    assert qm.qmoe_workspace_error_offset(bad) == -1


def staged_forward(shape, inp, d=None):
    """The same layer through the separate stage kernels (one stage per call)."""
    import torch

    p = gu.problem(shape)
    d = d or gu.device_inputs(inp)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    for st in range(4):
        qm.qmoe_forward_stages(p, st, st, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], d.get("fc1_zp"),
                               d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_kernel_parity_and_stage_kernels(name):
    shape, recipe, seed = CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    d = gu.device_inputs(inp)
    fused = layer_forward(shape, inp, d=d)
    staged = staged_forward(shape, inp, d=d)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(fused, ref, shape.dtype, f"{name} (layer kernel)")
    gu.assert_parity(staged, ref, shape.dtype, f"{name} (stage kernels)")
    a, b = gu.to_f64(fused, shape.dtype), gu.to_f64(staged, shape.dtype)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-3


@pytest.mark.gpu
def test_layer_kernel_is_batch_independent():
    """Each route's sums run over all of K in one warp in a fixed order, so a
    token's output does not depend on the batch it is packed into: packed and
    per-sequence calls agree bit for bit, and so do repeated calls."""
    shape, recipe, seed = synthetic.decode_layer(8)
    inp = synthetic.make_numpy(shape, recipe, seed)
    whole = layer_forward(shape, inp)
    assert np.array_equal(whole, layer_forward(shape, inp))
    d = gu.device_inputs(inp)
    parts, start = [], 0
    for L in (3, 1, 4):
        sub_shape = Shape(**{**shape.__dict__, "T": L})
        sub = dict(inp, x=inp["x"][start:start + L], logits=inp["logits"][start:start + L])
        dd = dict(d, x=gu.dev(sub["x"]), logits=gu.dev(sub["logits"]))
        parts.append(layer_forward(sub_shape, sub, d=dd))
        start += L
    assert np.array_equal(np.concatenate(parts), whole)


@pytest.mark.gpu
def test_layer_kernel_zero_weight_route_is_skipped():
    shape = Shape(T=2, H=256, inter=256, E=4, k=2, bits=4, block=32, dtype=FP16)
    inp = synthetic.make_numpy(shape, Recipe(scale_lo=0.01, scale_hi=0.02), 9)
    inp["logits"] = synthetic.float_to_bits(np.array([[0.0, -60000.0, -60000.0, -60000.0],
                                                      [-60000.0, 0.0, -60000.0, -60000.0]]), FP16)
    s = inp["fc2_s"].copy()
    s[2:] = 0x7E00  # NaN scales in the experts that only receive zero-weight routes
    inp["fc2_s"] = s
    got = layer_forward(shape, inp)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, "zero-weight")


def _nan(bits, dtype):
    f = gu.to_f64(bits, dtype)
    return np.isnan(f)


@pytest.mark.gpu
def test_failure_word_turns_the_output_into_nan():
    """No wait is made to run out: the failure word is written from the host
    between the stages, as a kernel that gave up would leave it, and the
    call's last step (the combine kernel, which follows the separate matmul
    kernels and the decode layer kernel alike) must then write NaN everywhere."""
    import torch

    shape, recipe, seed = synthetic.decode_layer(4)
    inp = synthetic.make_numpy(shape, recipe, seed)
    p = gu.problem(shape)
    d = gu.device_inputs(inp)
    ws = torch.zeros(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.zeros((shape.T, shape.H), dtype=torch.int16, device="cuda")
    args = (d["x"], d["logits"], d["fc1_q"], d["fc1_s"], None, d["fc2_q"], d["fc2_s"], None, out, ws)
    off = qm.qmoe_workspace_error_offset(p)
    # a complete call first: the failure word is 0 afterwards
    qm.qmoe_forward(p, *args)
    torch.cuda.synchronize()
    assert int(ws[off:off + 4].view(torch.int32).item()) == 0
    assert not _nan(out.cpu().numpy().view(np.uint16), shape.dtype).any()
    for code in (2, 3):
        for st in range(3):
            qm.qmoe_forward_stages(p, st, st, *args)
        torch.cuda.synchronize()
        ws[off:off + 4].view(torch.int32).fill_(code)
        qm.qmoe_forward_stages(p, 3, 3, *args)
        torch.cuda.synchronize()
        assert _nan(out.cpu().numpy().view(np.uint16), shape.dtype).all()
    # the next complete call resets the word and computes normally again
    qm.qmoe_forward(p, *args)
    torch.cuda.synchronize()
    assert int(ws[off:off + 4].view(torch.int32).item()) == 0
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(out.cpu().numpy().view(np.uint16), ref, shape.dtype, "after the failure")


GUARD_CASES = {
    "tiny_decode": synthetic.tiny(),
    "layer_kernel": (Shape(T=5, H=512, inter=256, E=6, k=3, bits=4, block=32, dtype=BF16),
                     Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 63),
    # grouped tcgen05 path with ragged M (routes per expert) and N tails
    "grouped_ragged": (Shape(T=333, H=320, inter=192, E=6, k=3, bits=4, block=32, dtype=FP16),
                       Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 64),
    "grouped_int3": (Shape(T=150, H=384, inter=256, E=5, k=2, bits=3, block=64, dtype=BF16),
                     Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 65),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(GUARD_CASES))
def test_outputs_stay_inside_their_buffers(name):
    """Guard bands of 64 KB around the output and the workspace (whose grouped
    regions x16s, h16 and y are reached by bulk tensor copies at ragged tails)
    stay untouched, and the result still matches the oracle."""
    import torch

    shape, recipe, seed = GUARD_CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    p = gu.problem(shape)
    n_ws = qm.qmoe_workspace_bytes(p)
    G = 65536
    ws_big = torch.full((n_ws + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
    out_big = torch.full((shape.T * shape.H + G,), 0x3C3C, dtype=torch.int16, device="cuda")
    ws = ws_big[G:G + n_ws]
    out = out_big[G // 2:G // 2 + shape.T * shape.H].view(shape.T, shape.H)
    got = (layer_forward if name == "layer_kernel" else gu.gpu_forward)(shape, inp, ws=ws, out=out)
    wb = ws_big.cpu().numpy()
    ob = out_big.cpu().numpy()
    assert (wb[:G] == 0x5A).all() and (wb[G + n_ws:] == 0x5A).all()
    assert (ob[:G // 2] == 0x3C3C).all() and (ob[G // 2 + shape.T * shape.H:] == 0x3C3C).all()
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, name)
