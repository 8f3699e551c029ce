"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Routing and grouping bit-exact; outputs within relative L2
2e-3 and max-abs 2^-7 * max|ref| of the oracle's once-rounded output."""
import numpy as np
import pytest

import oracle
import synthetic
from synthetic import BF16, FP16, Recipe, Shape
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    from quantized_mixture_experts_route_gb300 import build

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()


def oproblem(shape):
    return oracle.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                          shape.dtype)


# ------------------------------------------------------------------ routing + grouping

ROUTE_CASES = [
    # T, E, k, dtype, logits
    (1, 128, 8, BF16, "normal"),
    (4, 8, 2, FP16, "normal"),
    (8, 128, 8, BF16, "normal"),
    (64, 128, 8, BF16, "normal"),          # R = 512: one chunk
    (65, 128, 8, BF16, "normal"),          # R = 520: two chunks, ragged
    (300, 16, 4, FP16, "ties"),
    (1000, 6, 3, BF16, "ties"),
    (77, 512, 32, BF16, "normal"),
    (2000, 200, 7, FP16, "normal"),
    (8192, 128, 8, BF16, "normal"),        # prefill 8K
    (32768, 128, 8, FP16, "zipf"),         # INT2 32K workload routing
    (512, 128, 8, BF16, "zipf"),
]


@pytest.mark.parametrize("T,E,k,dt,kind", ROUTE_CASES, ids=[f"T{c[0]}_E{c[1]}_k{c[2]}_{c[4]}" for c in ROUTE_CASES])
@pytest.mark.parametrize("path", [0, 2])
def test_route_group_bit_exact(T, E, k, dt, kind, path):
    if path == 2 and T <= 8:
        path = 0
    rng = np.random.default_rng(T * 7 + E)
    if kind == "ties":
        vals = rng.integers(0, 3, size=(T, E)).astype(np.float64)
    elif kind == "zipf":
        vals = synthetic.zipf_logits(rng, T, E, 1.1)
    else:
        vals = rng.standard_normal((T, E)) * 2.0
    logits = synthetic.float_to_bits(vals, dt)
    shape = Shape(T=T, H=64, inter=64, E=E, k=k, bits=4, block=32, dtype=dt)
    idx, w, off, srt = gu.gpu_route(shape, logits, path)
    op = oproblem(shape)
    oidx, ow = oracle.route(op, logits)
    ooff, osrt, _ = oracle.permute(op, oidx)
    assert np.array_equal(idx, oidx), "top-k indices differ"
    assert np.array_equal(off, ooff), "expert offsets differ"
    assert np.array_equal(srt, osrt), "sorted routes differ"
    np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)


# ------------------------------------------------------------------ full forward

def case(name):
    if name == "tiny":
        return synthetic.tiny()
    if name.startswith("decode_T"):
        return synthetic.decode_layer(int(name[len("decode_T"):]))
    if name.startswith("int3_b"):
        b, T = name[len("int3_b"):].split("_T")
        return synthetic.int3_zipf(int(T), int(b))
    if name == "int2_T8":
        s, r, seed = synthetic.int2_prefill_32k()
        s.T = 8
        return s, r, seed
    if name == "int4_zp_fp16":
        return (Shape(T=5, H=256, inter=128, E=16, k=4, bits=4, block=64, dtype=FP16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 41)
    if name == "int3_zp_small":
        return (Shape(T=7, H=384, inter=96, E=10, k=3, bits=3, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 42)
    if name == "int2_zp_small":
        return (Shape(T=6, H=160, inter=224, E=12, k=5, bits=2, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.01, scale_hi=0.05, explicit_zp=True), 43)
    if name == "dense_E1_k1":
        return (Shape(T=3, H=128, inter=64, E=1, k=1, bits=4, block=32, dtype=BF16),
                Recipe(scale_lo=0.01, scale_hi=0.03), 44)
    if name == "bs_small":
        return (Shape(T=1, H=256, inter=128, E=4, k=2, bits=4, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 46)
    if name == "bs_zp_fp16":
        return (Shape(T=6, H=512, inter=256, E=5, k=3, bits=4, block=32, dtype=FP16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 47)
    if name == "bs_crowded":
        return (Shape(T=8, H=384, inter=256, E=3, k=3, bits=4, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 48)
    # tensor-copy decode kernel (K of both matmuls a multiple of 256)
    if name == "tma_zp_fp16":
        return (Shape(T=6, H=512, inter=512, E=5, k=3, bits=4, block=32, dtype=FP16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 49)
    if name == "tma_zp_bf16":
        return (Shape(T=7, H=1024, inter=512, E=9, k=4, bits=4, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 50)
    if name == "tma_small":
        return (Shape(T=3, H=256, inter=256, E=4, k=2, bits=4, block=32, dtype=BF16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 51)
    if name == "tma_crowded_fp16":
        return (Shape(T=8, H=768, inter=512, E=3, k=3, bits=4, block=32, dtype=FP16),
                Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 52)
    if name == "wide_k":
        return (Shape(T=2, H=256, inter=128, E=64, k=32, bits=4, block=128, dtype=BF16),
                Recipe(logit_std=0.5, scale_lo=0.005, scale_hi=0.02), 45)
    raise KeyError(name)


DECODE_CASES = ["tiny", "decode_T1", "decode_T2", "decode_T4", "decode_T8", "int3_b64_T1",
                "int3_b64_T8", "int3_b128_T8", "int2_T8", "int4_zp_fp16", "int3_zp_small",
                "int2_zp_small", "dense_E1_k1", "wide_k", "bs_small", "bs_zp_fp16", "bs_crowded",
                "tma_zp_fp16", "tma_zp_bf16", "tma_small", "tma_crowded_fp16"]


@pytest.mark.parametrize("name", DECODE_CASES)
def test_forward_parity_decode(name):
    shape, recipe, seed = case(name)
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = gu.gpu_forward(shape, inp)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, name)


def test_deterministic_and_token_permutation():
    shape, recipe, seed = synthetic.decode_layer(8)
    inp = synthetic.make_numpy(shape, recipe, seed)
    a = gu.gpu_forward(shape, inp)
    b = gu.gpu_forward(shape, inp)
    assert np.array_equal(a, b), "two runs differ"
    perm = np.random.default_rng(0).permutation(shape.T)
    inp2 = dict(inp, x=inp["x"][perm], logits=inp["logits"][perm])
    c = gu.gpu_forward(shape, inp2)
    assert np.array_equal(c, a[perm]), "token permutation does not commute with the output"


def test_packed_sequences_equal_separate_calls():
    """Packed concatenation vs per-sequence calls. The split of K between warps
    depends on the batch size, so the FP32 summation order may differ: the two
    agree far inside the parity bar (and bit for bit within one batch shape)."""
    shape, recipe, seed = synthetic.decode_layer(8)
    inp = synthetic.make_numpy(shape, recipe, seed)
    whole = gu.gpu_forward(shape, inp)
    parts, start = [], 0
    d = gu.device_inputs(inp)
    for L in (3, 1, 4):
        sub_shape = Shape(**{**shape.__dict__, "T": L})
        sub = dict(inp, x=inp["x"][start:start + L], logits=inp["logits"][start:start + L])
        dd = dict(d, x=gu.dev(sub["x"]), logits=gu.dev(sub["logits"]))
        parts.append(gu.gpu_forward(sub_shape, sub, d=dd))
        start += L
    a = gu.to_f64(np.concatenate(parts), shape.dtype)
    b = gu.to_f64(whole, shape.dtype)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-4


def test_nan_input_stays_in_its_token():
    shape, recipe, seed = synthetic.decode_layer(4)
    inp = synthetic.make_numpy(shape, recipe, seed)
    x = inp["x"].copy()
    x[2, 100] = 0x7FC0
    inp["x"] = x
    out = gu.gpu_forward(shape, inp)
    f = gu.to_f64(out, shape.dtype)
    assert np.isnan(f[2]).all()
    assert np.isfinite(np.delete(f, 2, axis=0)).all()


def test_zero_weight_route_is_skipped():
    shape = Shape(T=2, H=256, inter=128, E=4, k=2, bits=4, block=32, dtype=FP16)
    inp = synthetic.make_numpy(shape, Recipe(scale_lo=0.01, scale_hi=0.02), 9)
    inp["logits"] = synthetic.float_to_bits(np.array([[0.0, -60000.0, -60000.0, -60000.0],
                                                      [-60000.0, 0.0, -60000.0, -60000.0]]), FP16)
    s = inp["fc2_s"].copy()
    s[2:] = 0x7E00  # NaN scales in the experts that only receive zero-weight routes
    inp["fc2_s"] = s
    got = gu.gpu_forward(shape, inp)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, "zero-weight")


def test_outputs_stay_inside_their_buffers():
    """Guard bands: bytes around the output and the workspace stay untouched."""
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    shape, recipe, seed = synthetic.tiny()
    inp = synthetic.make_numpy(shape, recipe, seed)
    p = gu.problem(shape)
    n_ws = qm.qmoe_workspace_bytes(p)
    G = 4096
    ws_big = torch.full((n_ws + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
    out_big = torch.full((shape.T * shape.H + 2 * G,), 0x3C3C, dtype=torch.int16, device="cuda")
    ws = ws_big[G:G + n_ws]
    out = out_big[G:G + shape.T * shape.H].view(shape.T, shape.H)
    gu.gpu_forward(shape, inp, ws=ws, out=out)
    wb = ws_big.cpu().numpy()
    ob = out_big.cpu().numpy()
    assert (wb[:G] == 0x5A).all() and (wb[G + n_ws:] == 0x5A).all()
    assert (ob[:G] == 0x3C3C).all() and (ob[G + shape.T * shape.H:] == 0x3C3C).all()


def test_empty_batch():
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    shape, recipe, seed = synthetic.tiny()
    p = qm.problem(0, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block, shape.dtype)
    qm.qmoe_forward(p, None, None, None, None, None, None, None, None, None, None)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ grouped (tcgen05) path

GROUPED_CASES = {
    # name: (shape, recipe, seed); several 128-row tiles per expert, ragged M and N tails
    "g_int4_bf16": (Shape(T=700, H=256, inter=192, E=8, k=2, bits=4, block=32, dtype=BF16),
                    Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 51),
    "g_int4_fp16_zp": (Shape(T=333, H=512, inter=128, E=6, k=3, bits=4, block=64, dtype=FP16),
                       Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 52),
    "g_int2_fp16": (Shape(T=400, H=320, inter=256, E=5, k=2, bits=2, block=32, dtype=FP16),
                    Recipe(logit_std=1.0, scale_lo=0.01, scale_hi=0.04), 53),
    "g_int3_b64": (Shape(T=500, H=384, inter=256, E=7, k=2, bits=3, block=64, dtype=BF16),
                   Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 54),
    "g_int3_b128_zp": (Shape(T=300, H=256, inter=384, E=4, k=2, bits=3, block=128, dtype=BF16),
                       Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02, explicit_zp=True), 55),
    "g_small_T_forced": (Shape(T=5, H=256, inter=128, E=4, k=2, bits=4, block=32, dtype=BF16),
                         Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 56),
    # scales by bulk tensor copies with a long scale box (block 128: 16 stages per box)
    "g_int4_b128_fp16": (Shape(T=300, H=1024, inter=1024, E=4, k=2, bits=4, block=128, dtype=FP16),
                         Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 57),
    # ... and a short one (INT3 block 32: 2 stages of K = 128 per box)
    "g_int3_b32": (Shape(T=260, H=256, inter=256, E=5, k=2, bits=3, block=32, dtype=BF16),
                   Recipe(logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 58),
}


@pytest.mark.parametrize("name", sorted(GROUPED_CASES))
def test_forward_parity_grouped(name):
    shape, recipe, seed = GROUPED_CASES[name]
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = gu.gpu_forward(shape, inp, path=2)
    ref, _ = oracle.forward(oproblem(shape), inp)
    gu.assert_parity(got, ref, shape.dtype, name)


def test_grouped_matches_decode_on_small_batch():
    shape, recipe, seed = synthetic.decode_layer(8)
    inp = synthetic.make_numpy(shape, recipe, seed)
    a = gu.to_f64(gu.gpu_forward(shape, inp, path=1), shape.dtype)
    b = gu.to_f64(gu.gpu_forward(shape, inp, path=2), shape.dtype)
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-3


def _sampled(shape, recipe, seed, n_sample, big_weights=True):
    inp = synthetic.make_numpy(shape, recipe, seed)
    got = gu.gpu_forward(shape, inp)
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(shape.T, size=n_sample, replace=False))
    toks = np.unique(np.concatenate([toks, [0, shape.T - 1]]))
    ref, _ = oracle.forward(oproblem(shape), inp, tokens=toks)
    return got[toks], ref


@pytest.mark.parametrize("which", ["prefill_8k", "int2_32k", "int3_b64_T512", "int3_b128_T512", "decode_T64"])
def test_full_size_sampled(which):
    """Full-size workloads in the launch configuration the benchmark times, checked
    on sampled tokens that the oracle computes one by one."""
    if which == "prefill_8k":
        shape, recipe, seed = synthetic.prefill_8k()
    elif which == "int2_32k":
        shape, recipe, seed = synthetic.int2_prefill_32k()
    elif which == "decode_T64":
        shape, recipe, seed = synthetic.decode_layer(64)
    else:
        b = int(which.split("_b")[1].split("_")[0])
        shape, recipe, seed = synthetic.int3_zipf(512, b)
    got, ref = _sampled(shape, recipe, seed, 48)
    gu.assert_parity(got, ref, shape.dtype, which)


# ------------------------------------------------------------------ back-to-back calls

def _chain(cases, path, sync_each):
    """Run the layers in order on one stream, each consuming the previous output,
    with one shared workspace; return every layer's output bits."""
    import torch
    import quantized_mixture_experts_route_gb300 as qm

    shape0 = cases[0][0]
    p = gu.problem(shape0, path)
    ws = torch.empty(qm.qmoe_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    devs = [gu.device_inputs(inp) for _, inp in cases]
    outs = [torch.empty((shape0.T, shape0.H), dtype=torch.int16, device="cuda") for _ in cases]
    x = devs[0]["x"]
    for (shape, _), d, out in zip(cases, devs, outs):
        qm.qmoe_forward(p, x, d["logits"], d["fc1_q"], d["fc1_s"], d.get("fc1_zp"), d["fc2_q"], d["fc2_s"],
                        d.get("fc2_zp"), out, ws)
        if sync_each:
            torch.cuda.synchronize()
        x = out
    torch.cuda.synchronize()
    return [o.cpu().numpy().view(np.uint16) for o in outs]


@pytest.mark.parametrize("path_name", ["decode", "grouped"])
def test_back_to_back_layers_match_synchronised_calls(path_name):
    """Consecutive calls overlap on the GPU (each kernel may start before the
    previous one ends and waits for it before touching its results). Chained
    layers launched back to back must give exactly the results of the same calls
    separated by a device synchronisation, and each layer must match the oracle
    on the input the GPU actually gave it."""
    if path_name == "decode":
        cases = [synthetic.decode_layer(8, l) for l in range(4)]
        path = 0
    else:
        base, recipe, _ = synthetic.decode_layer(8)
        shape = Shape(**{**base.__dict__, "T": 64})
        cases = [(shape, recipe, 2000 + l) for l in range(3)]
        path = 2
    cases = [(s, synthetic.make_numpy(s, r, seed)) for s, r, seed in cases]
    fast = _chain(cases, path, sync_each=False)
    slow = _chain(cases, path, sync_each=True)
    for l, (a, b) in enumerate(zip(fast, slow)):
        assert np.array_equal(a, b), f"layer {l}: back-to-back result differs from synchronised calls"
    prev = cases[0][1]["x"]
    for l, ((shape, inp), got) in enumerate(zip(cases, fast)):
        ref, _ = oracle.forward(oproblem(shape), dict(inp, x=prev))
        gu.assert_parity(got, ref, shape.dtype, f"chained layer {l}")
        prev = got
