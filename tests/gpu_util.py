"""Helpers of the GPU parity tests: move seeded inputs to the device, call the
C ABI through the binding, and compare with the oracle's once-rounded output."""
from __future__ import annotations

import numpy as np

BF16, FP16 = 0, 1
REL_L2_MAX = 2e-3          # relative L2 over the whole [T, H] output
MAX_ABS_FRAC = 2.0 ** -7   # max |gpu - ref| <= 2^-7 * max |ref|


def dev(a):
    import torch

    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def problem(shape, path=0):
    import quantized_mixture_experts_route_gb300 as qm

    return qm.problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                      shape.dtype, path, getattr(shape, "format", 0))


def device_inputs(inp):
    return {k: dev(v) for k, v in inp.items()}


def gpu_forward(shape, inp, path=0, d=None, ws=None, out=None):
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    p = problem(shape, path)
    d = d or device_inputs(inp)
    if ws is None:
        ws = torch.empty(max(qm.qmoe_workspace_bytes(p), 1), dtype=torch.uint8, device="cuda")
    if out is None:
        out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward(p, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], d.get("fc1_zp"), d["fc2_q"],
                    d["fc2_s"], d.get("fc2_zp"), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def gpu_forward_ex(shape, inp, full_softmax, path=0):
    """qmoe_forward_ex with the inputs' optional biases (fc1_b, fc2_b) and routing option."""
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    p = problem(shape, path)
    d = device_inputs(inp)
    ws = torch.empty(max(qm.qmoe_workspace_bytes(p), 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((shape.T, shape.H), dtype=torch.int16, device="cuda")
    qm.qmoe_forward_ex(p, full_softmax, d.get("fc1_b"), d.get("fc2_b"), d["x"], d["logits"], d["fc1_q"],
                       d["fc1_s"], d.get("fc1_zp"), d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def gpu_route(shape, logits, path=0):
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    p = problem(shape, path)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    R = shape.T * shape.k
    idx = torch.empty(R, dtype=torch.int32, device="cuda")
    w = torch.empty(R, dtype=torch.float32, device="cuda")
    off = torch.empty(shape.E + 1, dtype=torch.int32, device="cuda")
    srt = torch.empty(R, dtype=torch.int32, device="cuda")
    qm.qmoe_route(p, dev(logits), idx, w, off, srt, ws)
    torch.cuda.synchronize()
    return (idx.cpu().numpy().reshape(shape.T, shape.k), w.cpu().numpy().reshape(shape.T, shape.k),
            off.cpu().numpy(), srt.cpu().numpy())


def to_f64(bits, dtype):
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def parity(got_bits, ref_bits, dtype):
    """(relative L2, max-abs / max|ref|) of the GPU output against the oracle's."""
    g = to_f64(got_bits, dtype)
    r = to_f64(ref_bits, dtype)
    assert np.isfinite(r).all(), "reference has non-finite values"
    assert np.isfinite(g).all(), "GPU output has non-finite values"
    nr = np.linalg.norm(r)
    assert nr > 0, "reference output is all zero"
    rel = float(np.linalg.norm(g - r) / nr)
    mx = float(np.abs(g - r).max() / np.abs(r).max())
    return rel, mx


def assert_parity(got_bits, ref_bits, dtype, label=""):
    rel, mx = parity(got_bits, ref_bits, dtype)
    assert rel <= REL_L2_MAX and mx <= MAX_ABS_FRAC, f"{label}: rel L2 {rel:.3e}, max-abs frac {mx:.3e}"
    return rel, mx
