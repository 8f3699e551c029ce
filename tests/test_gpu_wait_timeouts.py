"""The matmul kernels' bounded waits, made to run out: a copy of the library built
with QMOE_WAIT_LIMIT_NS = 0, whose waits poll without suspending
(`mbarrier.test_wait`) and give up at the first poll that finds the awaited
phase still open.

No GPU fault, trap or endless loop is involved. A warp or CTA that gives up
records its code in the workspace's failure word, waits (bounded) for its own
copies and MMAs in flight, frees its TMEM and returns; the combine kernel then
writes NaN to every output. Each case runs in a child process on the test
build and checks that the call returns OK and synchronises without a CUDA
error, that the failure word holds the kernel's code (1 grouped GEMM, 2
decode matmul, 3 decode layer kernel; the layer kernel's only bounded wait is
for another warp's fc1 units, which may already be done, so 0 is accepted
there when the output then matches the oracle), that the output is NaN
everywhere when the word is set, and that the CUDA context still computes
afterwards.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[2])
import quantized_mixture_experts_route_gb300 as qm
qm.LIB_PATH = sys.argv[1]
import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

R1 = Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02)
cases = {
    "decode_tma": synthetic.decode_layer(8) + (qm.QMOE_PATH_DECODE,),
    "grouped_route_tiles": (Shape(T=300, H=512, inter=256, E=8, k=2, bits=4, block=32, dtype=BF16), R1, 7,
                            qm.QMOE_PATH_GROUPED_ROUTE_TILES),
    "grouped_ws": (Shape(T=300, H=512, inter=256, E=8, k=2, bits=4, block=32, dtype=BF16), R1, 7,
                   qm.QMOE_PATH_GROUPED_WS),
    "layer_kernel_mxfp4": (Shape(T=8, H=512, inter=256, E=16, k=4, bits=4, block=32, dtype=BF16, format=1),
                           Recipe(logit_std=1.0), 8, qm.QMOE_PATH_DECODE),
}
res = {}
for name, (shape, recipe, seed, path) in cases.items():
    inp = synthetic.make_numpy(shape, recipe, seed)
    p = gu.problem(shape, path)
    d = gu.device_inputs(inp)
    ws = torch.zeros(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    out = torch.zeros((shape.T, shape.H), dtype=torch.int16, device="cuda")
    off = qm.qmoe_workspace_error_offset(p)
    qm.qmoe_forward_ex(p, 0, None, None, d["x"], d["logits"], d["fc1_q"], d["fc1_s"], d.get("fc1_zp"),
                       d["fc2_q"], d["fc2_s"], d.get("fc2_zp"), out, ws,
                       fc1_global_scale=d.get("g1"), fc2_global_scale=d.get("g2"))
    torch.cuda.synchronize()
    word = int(ws[off:off + 4].view(torch.int32).item())
    got = out.cpu().numpy().view(np.uint16)
    f = gu.to_f64(got, shape.dtype)
    parity = None
    if word == 0:
        op = oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                            shape.dtype, 0, shape.format, inp.get("g1"), inp.get("g2"))
        ref, _ = oracle.forward(op, inp)
        rel, mx = gu.parity(got, ref, shape.dtype)
        parity = bool(rel <= gu.REL_L2_MAX and mx <= gu.MAX_ABS_FRAC)
    res[name] = {"word": word, "nan_all": bool(np.isnan(f).all()), "parity": parity}
v = torch.arange(1000, device="cuda", dtype=torch.float32)
res["context_ok"] = float((v * 2).sum().item()) == 999000.0
print("RESULT " + json.dumps(res))
"""


def test_waits_run_out_and_are_reported(tmp_path):
    from quantized_mixture_experts_route_gb300 import build as qbuild

    lib = qbuild.build_variant(str(tmp_path / "libqmoe_nowait.so"), {"QMOE_WAIT_LIMIT_NS": "0ull"})
    r = subprocess.run([sys.executable, "-c", CHILD, lib, ROOT], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert res["context_ok"], res
    assert res["decode_tma"]["word"] == 2 and res["decode_tma"]["nan_all"], res
    for name in ("grouped_route_tiles", "grouped_ws"):
        assert res[name]["word"] == 1 and res[name]["nan_all"], res
    lk = res["layer_kernel_mxfp4"]
    assert lk["word"] in (0, 3), res
    assert lk["nan_all"] if lk["word"] == 3 else lk["parity"], res
