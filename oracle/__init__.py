"""Python access to the plain CPU oracle of the QMoE layer forward (qmoe_oracle.c).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The CUDA product path never
imports this package and shares no code with it.

Arrays are numpy: 16-bit floats are passed as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16 = 0
FP16 = 1


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library (portable C11, no ISA flags)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
        "-Wall", "-Wextra", "-I", _HERE, "-o", tmp, src, "-lm", "-lpthread"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle library next to its source if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "qmoe_oracle.h"))):
        compile_source(_SRC, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("block", ctypes.c_int32), ("dtype", ctypes.c_int32), ("full_softmax", ctypes.c_int32),
                ("format", ctypes.c_int32), ("g1", ctypes.c_void_p), ("g2", ctypes.c_void_p)]



def _declare(L):
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    L.oracle_bits_to_double.argtypes = [ctypes.c_uint16, ctypes.c_int]
    L.oracle_bits_to_double.restype = ctypes.c_double
    L.oracle_round_to_bits.argtypes = [ctypes.c_double, ctypes.c_int]
    L.oracle_round_to_bits.restype = ctypes.c_uint16
    L.oracle_unpack.argtypes = [vp, ctypes.c_int, ctypes.c_int64, vp]
    L.oracle_unpack.restype = None
    L.oracle_dequant_row.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int64, vp]
    L.oracle_dequant_row.restype = None
    L.oracle_route.argtypes = [P(_Problem), vp, vp, vp]
    L.oracle_route.restype = ctypes.c_int
    L.oracle_permute.argtypes = [P(_Problem), vp, vp, vp, vp]
    L.oracle_permute.restype = ctypes.c_int
    L.oracle_expert_ffn.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp,
                                    vp, vp]
    L.oracle_expert_ffn.restype = None
    L.oracle_expert_ffn_bias.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp,
                                         vp, vp, vp]
    L.oracle_expert_ffn_bias.restype = None
    L.oracle_forward.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                 ctypes.c_int64, vp, vp, ctypes.c_int]
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_forward_bias.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      ctypes.c_int64, vp, vp, ctypes.c_int]
    L.oracle_forward_bias.restype = ctypes.c_int
    for f in ("oracle_e2m1", "oracle_e8m0", "oracle_e4m3"):
        getattr(L, f).argtypes = [ctypes.c_uint]
        getattr(L, f).restype = ctypes.c_double
    L.oracle_router_logits.argtypes = [P(_Problem), vp, vp, vp]
    L.oracle_router_logits.restype = ctypes.c_int
    L.oracle_num_cores.argtypes = []
    L.oracle_num_cores.restype = ctypes.c_int
    return L


@dataclass
class Problem:
    T: int
    H: int
    inter: int
    E: int
    k: int
    bits: int
    block: int
    dtype: int
    full_softmax: int = 0   # 1: normalize_routing_weights = 0 (weights under the softmax over all E)
    format: int = 0         # 0 integer codes, 1 MXFP4, 2 NVFP4 (see qmoe_oracle.h)
    g1: np.ndarray | None = None   # NVFP4 per-expert FP32 global scales of fc1 / fc2, or None (1.0)
    g2: np.ndarray | None = None

    def c(self) -> _Problem:
        self._g = [None if g is None else np.ascontiguousarray(g, dtype=np.float32) for g in (self.g1, self.g2)]
        return _Problem(self.T, self.H, self.inter, self.E, self.k, self.bits, self.block, self.dtype,
                        self.full_softmax, self.format, *[None if g is None else g.ctypes.data for g in self._g])


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _weights(inp):
    c = lambda a, dt: None if a is None else np.ascontiguousarray(a, dtype=dt)
    # block scales: 16-bit floats of the dtype, or the FP4 formats' 8-bit scales (uint8 arrays)
    sc = lambda a: np.ascontiguousarray(a, dtype=np.uint8 if np.asarray(a).dtype == np.uint8 else np.uint16)
    return (c(inp["fc1_q"], np.uint8), sc(inp["fc1_s"]), c(inp.get("fc1_zp"), np.uint8),
            c(inp["fc2_q"], np.uint8), sc(inp["fc2_s"]), c(inp.get("fc2_zp"), np.uint8))


def _biases(inp):
    c = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.uint16)
    return c(inp.get("fc1_b")), c(inp.get("fc2_b"))


class Oracle:
    """One loaded copy of the oracle library (the default build, or a test's mutant)."""

    def __init__(self, path: str):
        self.L = _declare(ctypes.CDLL(path))

    def bits_to_double(self, bits, dtype: int) -> np.ndarray:
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        f = self.L.oracle_bits_to_double
        return np.array([f(int(v), dtype) for v in b.ravel()], dtype=np.float64).reshape(b.shape)

    def round_to_bits(self, v, dtype: int) -> np.ndarray:
        a = np.ascontiguousarray(v, dtype=np.float64)
        f = self.L.oracle_round_to_bits
        return np.array([f(float(x), dtype) for x in a.ravel()], dtype=np.uint16).reshape(a.shape)

    def unpack(self, packed: np.ndarray, bits: int, n: int) -> np.ndarray:
        p = np.ascontiguousarray(packed, dtype=np.uint8)
        out = np.zeros(n, dtype=np.uint8)
        self.L.oracle_unpack(_ptr(p), bits, n, _ptr(out))
        return out

    def dequant_row(self, q, scales, zp, bits, block, dtype, K, row) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.uint8)
        s = np.ascontiguousarray(scales, dtype=np.uint16)
        z = None if zp is None else np.ascontiguousarray(zp, dtype=np.uint8)
        out = np.zeros(K, dtype=np.float64)
        self.L.oracle_dequant_row(_ptr(q), _ptr(s), _ptr(z), bits, block, dtype, K, row, _ptr(out))
        return out

    def route(self, p: Problem, logits: np.ndarray):
        lg = np.ascontiguousarray(logits, dtype=np.uint16)
        idx = np.zeros((p.T, p.k), dtype=np.int32)
        w = np.zeros((p.T, p.k), dtype=np.float64)
        pc = p.c()
        if self.L.oracle_route(ctypes.byref(pc), _ptr(lg), _ptr(idx), _ptr(w)) != 0:
            raise ValueError("oracle_route: invalid problem")
        return idx, w

    def permute(self, p: Problem, topk_idx: np.ndarray):
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        offsets = np.zeros(p.E + 1, dtype=np.int32)
        R = p.T * p.k
        sorted_route = np.zeros(R, dtype=np.int32)
        route_slot = np.zeros(R, dtype=np.int32)
        pc = p.c()
        if self.L.oracle_permute(ctypes.byref(pc), _ptr(idx), _ptr(offsets), _ptr(sorted_route),
                                 _ptr(route_slot)) != 0:
            raise ValueError("oracle_permute: invalid problem")
        return offsets, sorted_route, route_slot

    def expert_ffn(self, p: Problem, inp: dict, expert: int, x_row: np.ndarray):
        q1, s1, z1, q2, s2, z2 = _weights(inp)
        b1, b2 = _biases(inp)
        xr = np.ascontiguousarray(x_row, dtype=np.float64)
        gu = np.zeros(2 * p.inter)
        h = np.zeros(p.inter)
        y = np.zeros(p.H)
        pc = p.c()
        self.L.oracle_expert_ffn_bias(ctypes.byref(pc), *[_ptr(a) for a in (q1, s1, z1, b1, q2, s2, z2, b2)],
                                      expert, _ptr(xr), _ptr(gu), _ptr(h), _ptr(y))
        return gu, h, y

    def forward(self, p: Problem, inp: dict, tokens=None, nthreads: int = 0, want_acc: bool = False):
        """Layer forward. Returns (out_bits [n, H] uint16, acc [n, H] float64 or None)."""
        x = np.ascontiguousarray(inp["x"], dtype=np.uint16)
        lg = np.ascontiguousarray(inp["logits"], dtype=np.uint16)
        w = _weights(inp)
        tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
        n = p.T if tok is None else len(tok)
        out = np.zeros((n, p.H), dtype=np.uint16)
        acc = np.zeros((n, p.H), dtype=np.float64) if want_acc else None
        pc = p.c()
        q1, s1, z1, q2, s2, z2 = w
        b1, b2 = _biases(inp)
        if self.L.oracle_forward_bias(ctypes.byref(pc), _ptr(x), _ptr(lg),
                                      *[_ptr(a) for a in (q1, s1, z1, b1, q2, s2, z2, b2)],
                                      _ptr(tok), n, _ptr(out), _ptr(acc), nthreads) != 0:
            raise ValueError("oracle_forward: invalid arguments")
        return out, acc

    def router_logits(self, p: Problem, x_bits: np.ndarray, w_router_bits: np.ndarray) -> np.ndarray:
        """Router logits [T][E] (dtype bits) = round(x [T][H] . w_router [E][H]^T)."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        w = np.ascontiguousarray(w_router_bits, dtype=np.uint16)
        assert x.shape == (p.T, p.H) and w.shape == (p.E, p.H)
        out = np.zeros((p.T, p.E), dtype=np.uint16)
        pc = p.c()
        if self.L.oracle_router_logits(ctypes.byref(pc), _ptr(x), _ptr(w), _ptr(out)) != 0:
            raise ValueError("oracle_router_logits: invalid arguments")
        return out

    def fp4_tables(self):
        """(E2M1 values of the 16 codes, E8M0 values of the 256 bytes, E4M3 values of the 256 bytes)."""
        return (np.array([self.L.oracle_e2m1(c) for c in range(16)]),
                np.array([self.L.oracle_e8m0(b) for b in range(256)]),
                np.array([self.L.oracle_e4m3(b) for b in range(256)]))

    def num_cores(self) -> int:
        return self.L.oracle_num_cores()


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def bits_to_double(bits, dtype):
    return default().bits_to_double(bits, dtype)


def round_to_bits(v, dtype):
    return default().round_to_bits(v, dtype)


def unpack(packed, bits, n):
    return default().unpack(packed, bits, n)


def dequant_row(q, scales, zp, bits, block, dtype, K, row):
    return default().dequant_row(q, scales, zp, bits, block, dtype, K, row)


def route(p, logits):
    return default().route(p, logits)


def permute(p, topk_idx):
    return default().permute(p, topk_idx)


def expert_ffn(p, inp, expert, x_row):
    return default().expert_ffn(p, inp, expert, x_row)


def forward(p, inp, tokens=None, nthreads=0, want_acc=False):
    return default().forward(p, inp, tokens, nthreads, want_acc)


def router_logits(p, x_bits, w_router_bits):
    return default().router_logits(p, x_bits, w_router_bits)


def fp4_tables():
    return default().fp4_tables()


def num_cores() -> int:
    return default().num_cores()
