"""Seeded synthetic inputs for the QMoE layer forward.

This module only draws random inputs in the operator's storage formats. It
holds none of the operator's arithmetic: no routing, no unpacking of codes, no
dequantisation, no matmul. Packed weight codes are drawn as uniformly random
bytes, which is the same as drawing every 2-, 3- or 4-bit code uniformly and
independently, whatever the packing order, so the packing convention lives only
in the two implementations that read the codes (the CPU oracle and the CUDA
kernels).

Both the CPU oracle (tests, benchmark baseline) and the CUDA path read inputs
made here. Two backends exist:

* ``numpy`` (host arrays, PCG64): used by the parity tests.
* ``torch`` (tensors made on a torch device with a seeded ``torch.Generator``):
  used for the multi-GB benchmark weights, which would take minutes to draw on
  the host. The same seed gives different values on the two backends.

Workload recipes follow the QMoE pages (microsoft/onnxruntime PRs #32522,
#33575, #33731, #33973): packed token-major input [T, H], raw router logits
[T, E], INT4/INT3/INT2 codes with per-block scales along K, fc1 with 2*inter
interleaved gate/up rows.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16 = 0
FP16 = 1
DTYPE_NAMES = {BF16: "bf16", FP16: "fp16"}


@dataclass
class Shape:
    T: int
    H: int
    inter: int
    E: int
    k: int
    bits: int
    block: int
    dtype: int
    format: int = 0   # 0 integer codes, 1 MXFP4 (E8M0 scales, block 32), 2 NVFP4 (E4M3, block 16)

    def code_bytes_per_row(self, K: int) -> int:
        return K * self.bits // 8


@dataclass
class Recipe:
    """How the values of one workload are drawn."""

    x_std: float = 1.0
    logit_std: float = 1.0
    zipf_s: float | None = None       # None: logits ~ N(0, logit_std); else Zipf-biased Gumbel logits
    scale_lo: float = 0.005
    scale_hi: float = 0.02
    explicit_zp: bool = False         # False: zero point is the implicit 2^(bits-1)
    seq_lens: list[int] | None = None  # packed sequence lengths (sum == T), for the packing tests
    bias_std: float | None = None     # FC1 [E, 2I] and FC2 [E, H] biases ~ N(0, bias_std); None: no biases
    extra: dict = field(default_factory=dict)


def float32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the raw 16-bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    nan = np.isnan(a)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    rounded[nan] = 0x7FC0
    return rounded


def float_to_bits(a: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == BF16:
        return float32_to_bf16_bits(a.astype(np.float32))
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


def split_lengths(rng: np.random.Generator, n_seq: int, lo: int, hi: int, total: int) -> list[int]:
    """Draw n_seq lengths ~U[lo, hi] and rescale them to sum to `total` (largest remainder)."""
    raw = rng.integers(lo, hi + 1, size=n_seq).astype(np.float64)
    ideal = raw * (total / raw.sum())
    base = np.floor(ideal).astype(np.int64)
    short = total - int(base.sum())
    order = np.argsort(-(ideal - base), kind="stable")
    base[order[:short]] += 1
    return [int(v) for v in base]


def zipf_logits(rng: np.random.Generator, T: int, E: int, s: float) -> np.ndarray:
    """Router logits whose top-k selection follows Zipf(s) expert popularity.

    ln p_e + Gumbel(0, 1) noise: the top-k of these samples k experts without
    replacement with probability proportional to p_e (Gumbel top-k), and p_e is
    proportional to rank^-s over a seeded permutation of the experts.
    """
    ranks = rng.permutation(E) + 1
    p = ranks.astype(np.float64) ** (-s)
    p /= p.sum()
    g = rng.gumbel(0.0, 1.0, size=(T, E))
    return np.log(p)[None, :] + g


def make_numpy(shape: Shape, recipe: Recipe, seed: int) -> dict:
    """Draw one layer's inputs on the host.

    Returns uint16 bit patterns for x, logits and scales, uint8 packed codes,
    and uint8 zero points (or None for the implicit 2^(bits-1)).
    """
    rng = np.random.default_rng(seed)
    T, H, I, E = shape.T, shape.H, shape.inter, shape.E
    dt = shape.dtype
    x = float_to_bits(rng.standard_normal((T, H)) * recipe.x_std, dt)
    if recipe.zipf_s is None:
        logits = rng.standard_normal((T, E)) * recipe.logit_std
    else:
        logits = zipf_logits(rng, T, E, recipe.zipf_s)
    logits = float_to_bits(logits, dt)

    def codes(rows: int, K: int) -> np.ndarray:
        nbytes = rows * K * shape.bits // 8
        return rng.integers(0, 256, size=nbytes, dtype=np.uint8).reshape(E, rows // E, K * shape.bits // 8)

    def scales(rows: int, K: int) -> np.ndarray:
        size = (E, rows // E, K // shape.block)
        if shape.format == 1:
            # E8M0 bytes 118..122: block scales 2^-9 .. 2^-5
            return rng.integers(118, 123, size=size, dtype=np.uint8)
        if shape.format == 2:
            # E4M3 bytes 0x08..0x1F: exponent fields 1..3 (2^-6 .. 2^-4), any mantissa
            return rng.integers(0x08, 0x20, size=size, dtype=np.uint8)
        v = rng.uniform(recipe.scale_lo, recipe.scale_hi, size=size)
        return float_to_bits(v, dt)

    def zps(rows: int, K: int):
        if not recipe.explicit_zp or shape.format != 0:
            return None
        return rng.integers(0, 1 << shape.bits, size=(E, rows // E, K // shape.block), dtype=np.uint8)

    fc1_q = codes(E * 2 * I, H)
    fc1_s = scales(E * 2 * I, H)
    fc1_zp = zps(E * 2 * I, H)
    fc2_q = codes(E * H, I)
    fc2_s = scales(E * H, I)
    fc2_zp = zps(E * H, I)
    # biases come last, so that the other inputs do not depend on whether they are drawn
    fc1_b = fc2_b = None
    if recipe.bias_std is not None:
        fc1_b = float_to_bits(rng.standard_normal((E, 2 * I)) * recipe.bias_std, dt)
        fc2_b = float_to_bits(rng.standard_normal((E, H)) * recipe.bias_std, dt)
    out = dict(x=x, logits=logits, fc1_q=fc1_q, fc1_s=fc1_s, fc1_zp=fc1_zp,
               fc2_q=fc2_q, fc2_s=fc2_s, fc2_zp=fc2_zp, fc1_b=fc1_b, fc2_b=fc2_b)
    if shape.format == 2:
        # NVFP4 per-expert FP32 global scales of fc1 and fc2, drawn last
        out["g1"] = rng.uniform(0.25, 1.0, size=E).astype(np.float32)
        out["g2"] = rng.uniform(0.25, 1.0, size=E).astype(np.float32)
    return out


def make_torch_weights(shape: Shape, recipe: Recipe, seed: int, device):
    """Draw one layer's packed weights and scales directly on a torch device.

    Used for the multi-GB benchmark stacks. Returns torch tensors in the same
    formats as :func:`make_numpy` (uint8 codes, int16 bit patterns of scales).
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    E, H, I = shape.E, shape.H, shape.inter
    tdt = torch.bfloat16 if shape.dtype == BF16 else torch.float16

    def codes(rows, K):
        n = rows * K * shape.bits // 8
        return torch.randint(0, 256, (n,), generator=g, device=device, dtype=torch.uint8).view(E, rows // E, -1)

    def scales(rows, K):
        size = (E, rows // E, K // shape.block)
        if shape.format == 1:    # E8M0 bytes 118..122
            return torch.randint(118, 123, size, generator=g, device=device, dtype=torch.uint8)
        if shape.format == 2:    # E4M3 bytes 0x08..0x1F
            return torch.randint(0x08, 0x20, size, generator=g, device=device, dtype=torch.uint8)
        v = torch.rand(size, generator=g, device=device, dtype=torch.float32)
        v = v * (recipe.scale_hi - recipe.scale_lo) + recipe.scale_lo
        return v.to(tdt)

    fc1_q = codes(E * 2 * I, H)
    fc1_s = scales(E * 2 * I, H)
    fc2_q = codes(E * H, I)
    fc2_s = scales(E * H, I)
    out = dict(fc1_q=fc1_q, fc1_s=fc1_s, fc1_zp=None, fc2_q=fc2_q, fc2_s=fc2_s, fc2_zp=None)
    if shape.format == 2:
        out["g1"] = torch.rand(E, generator=g, device=device) * 0.75 + 0.25
        out["g2"] = torch.rand(E, generator=g, device=device) * 0.75 + 0.25
    return out


def make_activations(shape: Shape, recipe: Recipe, seed: int) -> dict:
    """Host x and logits only (per-step inputs of the benchmark stacks)."""
    rng = np.random.default_rng(seed)
    T, H, E = shape.T, shape.H, shape.E
    x = float_to_bits(rng.standard_normal((T, H)) * recipe.x_std, shape.dtype)
    if recipe.zipf_s is None:
        logits = rng.standard_normal((T, E)) * recipe.logit_std
    else:
        logits = zipf_logits(rng, T, E, recipe.zipf_s)
    return dict(x=x, logits=float_to_bits(logits, shape.dtype))


# ---------------------------------------------------------------------------
# The five workloads (sizes, distributions and seeds)
# ---------------------------------------------------------------------------

def tiny() -> tuple[Shape, Recipe, int]:
    """T=4, H=64, inter=32, E=8, k=2, INT4 block 32, FP16, logits N(0,1), scales U[0.005,0.02]."""
    return (Shape(T=4, H=64, inter=32, E=8, k=2, bits=4, block=32, dtype=FP16),
            Recipe(x_std=1.0, logit_std=1.0, scale_lo=0.005, scale_hi=0.02), 0)


def decode_layer(T: int, layer: int = 0) -> tuple[Shape, Recipe, int]:
    """One layer of the 48-layer decode stack: H=2048, inter=768, E=128, k=8, INT4 b32, BF16."""
    return (Shape(T=T, H=2048, inter=768, E=128, k=8, bits=4, block=32, dtype=BF16),
            Recipe(x_std=1.0, logit_std=2.0, scale_lo=0.002, scale_hi=0.01), 1000 + layer)


def prefill_8k() -> tuple[Shape, Recipe, int]:
    """T=8192 packed from 16 sequences ~U[128,1024]; logits N(0,2); INT4 b32, BF16."""
    rng = np.random.default_rng(1)
    lens = split_lengths(rng, 16, 128, 1024, 8192)
    return (Shape(T=8192, H=2048, inter=768, E=128, k=8, bits=4, block=32, dtype=BF16),
            Recipe(x_std=1.0, logit_std=2.0, scale_lo=0.002, scale_hi=0.01, seq_lens=lens), 1)


def int3_zipf(T: int, block: int) -> tuple[Shape, Recipe, int]:
    """INT3 (zero point 4), block 64 or 128, BF16, Zipf(1.1) expert popularity."""
    return (Shape(T=T, H=2048, inter=768, E=128, k=8, bits=3, block=block, dtype=BF16),
            Recipe(x_std=1.0, zipf_s=1.1, scale_lo=0.002, scale_hi=0.01), 2)


def int2_prefill_32k() -> tuple[Shape, Recipe, int]:
    """INT2 b32, FP16, T=32768 packed from 32 sequences ~U[512,1536], Zipf(1.1)."""
    rng = np.random.default_rng(3)
    lens = split_lengths(rng, 32, 512, 1536, 32768)
    return (Shape(T=32768, H=2048, inter=768, E=128, k=8, bits=2, block=32, dtype=FP16),
            Recipe(x_std=1.0, zipf_s=1.1, scale_lo=0.002, scale_hi=0.01, seq_lens=lens), 3)
