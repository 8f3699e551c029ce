"""Checks that pin the CPU oracle to facts outside itself.

Each check takes an oracle instance, so that the same checks also run against
mutated copies of the oracle (tests/test_oracle_mutants.py): a pin set that no
plausible mistake slips through. The references here are library routines
(numpy bit unpacking, numpy float16 conversion, scipy softmax, torch float64
matmul and SiLU), closed forms, brute force over every expert, invariants of
the method, and the hand-written fixtures under tests/golden/.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

import oracle as oracle_mod
import synthetic
from tests.conftest import read_golden

BF16, FP16 = 0, 1
DT = {"bf16": BF16, "fp16": FP16}


# --------------------------------------------------------------------------- helpers

def lsb_first_codes(packed: np.ndarray, bits: int, n: int) -> np.ndarray:
    """Codes of a continuous least-significant-bit-first bit stream (numpy unpackbits)."""
    stream = np.unpackbits(np.ascontiguousarray(packed, dtype=np.uint8).ravel(), bitorder="little")
    stream = stream[: n * bits].reshape(n, bits).astype(np.int64)
    return (stream << np.arange(bits)).sum(axis=1)


def bits_to_f64(bits: np.ndarray, dtype: int) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant_matrix(q, s, zp, bits, block, dtype, rows, K) -> np.ndarray:
    """[rows, K] float64 weights of one expert from library unpacking and format views."""
    codes = lsb_first_codes(q, bits, rows * K).reshape(rows, K).astype(np.float64)
    scale = np.repeat(bits_to_f64(s, dtype).reshape(rows, K // block), block, axis=1)
    if zp is None:
        z = float(1 << (bits - 1))
    else:
        z = np.repeat(np.asarray(zp, dtype=np.float64).reshape(rows, K // block), block, axis=1)
    return (codes - z) * scale


def dense_expert(inp, shape, e, xrow):
    """gu, h, y of expert e for one input row in torch float64 (matmul + library SiLU),
    with the optional biases fc1_b / fc2_b added after each matmul."""
    H, I = shape.H, shape.inter
    W1 = dequant_matrix(inp["fc1_q"][e], inp["fc1_s"][e], None if inp["fc1_zp"] is None else inp["fc1_zp"][e],
                        shape.bits, shape.block, shape.dtype, 2 * I, H)
    W2 = dequant_matrix(inp["fc2_q"][e], inp["fc2_s"][e], None if inp["fc2_zp"] is None else inp["fc2_zp"][e],
                        shape.bits, shape.block, shape.dtype, H, I)
    W1 = torch.from_numpy(W1)
    W2 = torch.from_numpy(W2)
    x = torch.from_numpy(np.asarray(xrow, dtype=np.float64))
    gu = W1 @ x
    if inp.get("fc1_b") is not None:
        gu = gu + torch.from_numpy(bits_to_f64(inp["fc1_b"][e], shape.dtype))
    gate, up = gu[0::2], gu[1::2]
    h = torch.nn.functional.silu(gate) * up
    y = W2 @ h
    if inp.get("fc2_b") is not None:
        y = y + torch.from_numpy(bits_to_f64(inp["fc2_b"][e], shape.dtype))
    return gu.numpy(), h.numpy(), y.numpy()


def problem_of(shape) -> oracle_mod.Problem:
    return oracle_mod.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                              shape.dtype)


def fail(msg):
    raise AssertionError(msg)


# --------------------------------------------------------------------------- pins

def pin_golden_packing(orc):
    for bits, hexbytes, codes in read_golden("packing.txt"):
        bits = int(bits)
        packed = np.frombuffer(bytes.fromhex(hexbytes), dtype=np.uint8)
        want = [int(c) for c in codes.split(",")]
        got = orc.unpack(packed, bits, len(want)).tolist()
        if got != want:
            fail(f"unpack bits={bits} {hexbytes}: {got} != {want}")
        if lsb_first_codes(packed, bits, len(want)).tolist() != want:
            fail("fixture disagrees with the LSB-first bit stream")


def pin_unpack_random(orc):
    rng = np.random.default_rng(11)
    for bits in (2, 3, 4):
        n = 8 * 257
        packed = rng.integers(0, 256, size=n * bits // 8, dtype=np.uint8)
        if not np.array_equal(orc.unpack(packed, bits, n), lsb_first_codes(packed, bits, n)):
            fail(f"unpack bits={bits} differs from the LSB-first bit stream")


def pin_bits_to_double(orc):
    allbits = np.arange(65536, dtype=np.uint16)
    for dt in (FP16, BF16):
        got = orc.bits_to_double(allbits, dt)
        want = bits_to_f64(allbits, dt)
        same = (got == want) | (np.isnan(got) & np.isnan(want))
        if not same.all():
            bad = int(np.flatnonzero(~same)[0])
            fail(f"bits_to_double dtype={dt} bits={bad:#06x}: {got[bad]} != {want[bad]}")
        if not np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)])):
            fail("bits_to_double loses the sign of zero")


def _parse_pow2_sum(text):
    if text == "nan":
        return float("nan")
    total = 0.0
    for term in text.split("+"):
        m, e = term.split("*2^")
        total += math.ldexp(float(m), int(e))
    return total


def pin_golden_rounding(orc):
    for dt, value, want in read_golden("rounding.txt"):
        got = int(orc.round_to_bits(np.array([_parse_pow2_sum(value)]), DT[dt])[0])
        if got != int(want, 16):
            fail(f"round {dt} {value}: {got:#06x} != {want}")


def pin_rounding_fp16_exhaustive(orc):
    """Every finite FP16 value, every midpoint and points just off the midpoints,
    against numpy's float64 -> float16 conversion (round to nearest even)."""
    vals = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    eps = np.abs(mids) * 2.0 ** -30 + 2.0 ** -60
    probe = np.concatenate([vals, mids, mids + eps, mids - eps, [65519.0, 65520.0, 70000.0]])
    probe = np.concatenate([probe, -probe])
    got = orc.round_to_bits(probe, FP16)
    with np.errstate(over="ignore"):
        want = probe.astype(np.float16).view(np.uint16)
    if not np.array_equal(got, want):
        bad = int(np.flatnonzero(got != want)[0])
        fail(f"fp16 rounding of {probe[bad]!r}: {got[bad]:#06x} != {want[bad]:#06x}")


def pin_rounding_bf16(orc):
    """BF16 rounding of values that are exact float32s, against the float32 bit
    formula (no double rounding is possible there), plus values off the midpoints."""
    rng = np.random.default_rng(5)
    f32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),
        np.array([3.3895314e38, -3.3895314e38, 1.0, 0.0], dtype=np.float32),
    ])
    got = orc.round_to_bits(f32.astype(np.float64), BF16)
    want = synthetic.float32_to_bf16_bits(f32)
    if not np.array_equal(got, want):
        bad = int(np.flatnonzero(got != want)[0])
        fail(f"bf16 rounding of {f32[bad]!r}: {got[bad]:#06x} != {want[bad]:#06x}")
    # a value just above a tie must round up and one just below down, even where
    # a float32 intermediate would have landed exactly on the tie
    for base in (1.0, 1.5, 3.0, 2.0 ** -100, -1.25):
        mag = abs(base)
        ulp = 2.0 ** (math.floor(math.log2(mag)) - 7)
        tie = math.copysign(mag + ulp / 2, base)
        nxt = math.copysign(mag + ulp, base)
        above = orc.round_to_bits(np.array([tie * (1 + 2.0 ** -40)]), BF16)[0]
        below = orc.round_to_bits(np.array([tie * (1 - 2.0 ** -40)]), BF16)[0]
        want_above = synthetic.float32_to_bf16_bits(np.array([nxt], dtype=np.float32))[0]
        want_below = synthetic.float32_to_bf16_bits(np.array([base], dtype=np.float32))[0]
        if above != want_above or below != want_below:
            fail(f"bf16 rounding next to the tie above {base}")


def pin_dequant(orc):
    rng = np.random.default_rng(7)
    for bits, block, dt, explicit in ((4, 32, BF16, False), (3, 64, FP16, True), (2, 32, BF16, True),
                                      (3, 128, BF16, False), (4, 64, FP16, True)):
        rows, K = 6, 256
        q = rng.integers(0, 256, size=rows * K * bits // 8, dtype=np.uint8)
        s = synthetic.float_to_bits(rng.uniform(0.001, 0.1, size=(rows, K // block)), dt)
        zp = rng.integers(0, 1 << bits, size=(rows, K // block), dtype=np.uint8) if explicit else None
        want = dequant_matrix(q, s, zp, bits, block, dt, rows, K)
        for r in range(rows):
            got = orc.dequant_row(q, s, zp, bits, block, dt, K, r)
            if not np.array_equal(got, want[r]):
                fail(f"dequant bits={bits} block={block} row {r}")


def _logits_bits(values, dt):
    return synthetic.float_to_bits(np.asarray(values, dtype=np.float64), dt)


def pin_golden_routing(orc):
    for dt, k, logits, idx, w in read_golden("routing.txt"):
        vals = [float(v) for v in logits.split(",")]
        E = len(vals)
        p = oracle_mod.Problem(1, 8, 8, E, int(k), 4, 8, DT[dt])
        gi, gw = orc.route(p, _logits_bits(vals, DT[dt]).reshape(1, E))
        want_i = [int(v) for v in idx.split(",")]
        want_w = [float(v) for v in w.split(",")]
        if gi[0].tolist() != want_i:
            fail(f"route {logits}: {gi[0].tolist()} != {want_i}")
        if not np.allclose(gw[0], want_w, rtol=1e-14, atol=0):
            fail(f"route weights {logits}: {gw[0]} != {want_w}")


def pin_route_bruteforce(orc):
    """Selection against a full stable sort (Python sorted), weights against
    scipy's softmax of the selected logits; integer logits force many ties."""
    rng = np.random.default_rng(3)
    for E, k, dt, kind in ((8, 2, FP16, "ties"), (8, 8, BF16, "ties"), (16, 5, BF16, "normal"),
                           (128, 8, BF16, "normal"), (7, 3, FP16, "ties")):
        T = 300
        vals = rng.integers(0, 3, size=(T, E)).astype(np.float64) if kind == "ties" else rng.standard_normal((T, E)) * 2
        lb = _logits_bits(vals, dt).reshape(T, E)
        lv = bits_to_f64(lb, dt)
        p = oracle_mod.Problem(T, 8, 8, E, k, 4, 8, dt)
        gi, gw = orc.route(p, lb)
        for t in range(T):
            want = sorted(range(E), key=lambda e: (-lv[t, e], e))[:k]
            if gi[t].tolist() != want:
                fail(f"route E={E} k={k} token {t}: {gi[t].tolist()} != {want}")
            ref = scipy.special.softmax(lv[t, want])
            if not np.allclose(gw[t], ref, rtol=1e-12, atol=1e-15):
                fail(f"route weights E={E} k={k} token {t}")
        if not np.allclose(gw.sum(axis=1), 1.0, atol=1e-12):
            fail("routing weights do not sum to 1")
        if (gi < 0).any() or (gi >= E).any():
            fail("expert id out of range")
        if any(len(set(r)) != k for r in gi.tolist()):
            fail("duplicate expert in one token's top-k")
        if k == E:
            full = scipy.special.softmax(lv, axis=1)
            for t in range(T):
                if not np.allclose(gw[t], full[t, gi[t]], rtol=1e-12):
                    fail("k == E weights differ from the full softmax")


def pin_permute(orc):
    rng = np.random.default_rng(9)
    for T, E, k in ((1, 8, 2), (37, 16, 4), (500, 128, 8), (64, 3, 3)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        p = oracle_mod.Problem(T, 8, 8, E, k, 4, 8, BF16)
        off, srt, slot = orc.permute(p, idx)
        flat = idx.ravel()
        want = sorted(range(T * k), key=lambda r: flat[r])  # Python's sort is stable
        if srt.tolist() != want:
            fail(f"sorted_route T={T} E={E} k={k}")
        counts = np.bincount(flat, minlength=E)
        if off.tolist() != [0] + np.cumsum(counts).tolist():
            fail("expert_offsets")
        if not np.array_equal(slot[srt], np.arange(T * k)):
            fail("route_slot is not the inverse of sorted_route")


def _small_inputs(T=5, H=64, I=96, E=6, k=3, bits=4, block=32, dt=BF16, seed=21, explicit_zp=False,
                  bias_std=None):
    shape = synthetic.Shape(T=T, H=H, inter=I, E=E, k=k, bits=bits, block=block, dtype=dt)
    rec = synthetic.Recipe(x_std=1.0, logit_std=1.5, scale_lo=0.01, scale_hi=0.05, explicit_zp=explicit_zp,
                           bias_std=bias_std)
    return shape, synthetic.make_numpy(shape, rec, seed)


def pin_dense_ffn_E1_k1(orc):
    """E = 1, k = 1 is a dense SwiGLU FFN with weight exactly 1."""
    for bits, block, dt in ((4, 32, BF16), (3, 64, FP16), (2, 32, FP16)):
        shape, inp = _small_inputs(T=4, H=128, I=64, E=1, k=1, bits=bits, block=block, dt=dt)
        p = problem_of(shape)
        out, acc = orc.forward(p, inp, nthreads=1, want_acc=True)
        x = bits_to_f64(inp["x"], dt)
        for t in range(shape.T):
            _, _, y = dense_expert(inp, shape, 0, x[t])
            if not np.allclose(acc[t], y, rtol=1e-12, atol=1e-12):
                fail(f"E=1,k=1 bits={bits} token {t} differs from the dense SwiGLU FFN")


def pin_bruteforce_dense_over_experts(orc):
    """Every expert for every token, combined with the top-k softmax weights
    (zero elsewhere), against the grouped oracle."""
    for bits, block, dt, zp, H, I in ((4, 32, BF16, False, 128, 96), (3, 64, BF16, True, 192, 64),
                                      (2, 32, FP16, False, 160, 32)):
        shape, inp = _small_inputs(T=6, H=H, I=I, E=6, k=3, bits=bits, block=block, dt=dt, explicit_zp=zp)
        p = problem_of(shape)
        out, acc = orc.forward(p, inp, nthreads=2, want_acc=True)
        x = bits_to_f64(inp["x"], dt)
        lv = bits_to_f64(inp["logits"], dt)
        for t in range(shape.T):
            order = sorted(range(shape.E), key=lambda e: (-lv[t, e], e))
            sel = order[: shape.k]
            wsel = scipy.special.softmax(lv[t, sel])
            mask = np.zeros(shape.E)
            mask[sel] = wsel
            total = np.zeros(shape.H)
            for e in range(shape.E):
                _, _, y = dense_expert(inp, shape, e, x[t])
                total += mask[e] * y
            if not np.allclose(acc[t], total, rtol=1e-11, atol=1e-12):
                fail(f"dense-over-experts bits={bits} token {t}")
            ref_bits = (total.astype(np.float16).view(np.uint16) if dt == FP16 else None)
            if ref_bits is not None and not np.array_equal(out[t], ref_bits):
                # the double sums agree to ~1e-12; only an exact tie could flip a bit
                if (np.abs(out[t].astype(np.int64) - ref_bits.astype(np.int64)) > 1).any():
                    fail("rounded outputs differ by more than one unit")


def pin_one_hot(orc):
    """x = e_i gives gate/up equal to column i of the dequantised fc1 (closed form)."""
    shape, inp = _small_inputs(T=1, H=64, I=32, E=3, k=1, bits=4, block=32, dt=BF16)
    p = problem_of(shape)
    W1 = dequant_matrix(inp["fc1_q"][2], inp["fc1_s"][2], None, 4, 32, BF16, 64, 64)  # 2I x H
    for i in (0, 17, 63):
        xr = np.zeros(64)
        xr[i] = 1.0
        gu, h, y = orc.expert_ffn(p, inp, 2, xr)
        if not np.array_equal(gu, W1[:, i]):
            fail(f"one-hot column {i}: fc1 output is not the dequantised column")
        g, u = W1[0::2, i], W1[1::2, i]
        if not np.allclose(h, g / (1 + np.exp(-g)) * u, rtol=1e-14, atol=0):
            fail("one-hot SwiGLU")


def pin_token_permutation(orc):
    """Routing is token-local: permuting the packed tokens permutes the output rows
    bit for bit, and the packed concatenation equals per-sequence calls."""
    shape, inp = _small_inputs(T=12, H=64, I=32, E=8, k=2)
    p = problem_of(shape)
    out, _ = orc.forward(p, inp, nthreads=3)
    perm = np.random.default_rng(2).permutation(shape.T)
    inp2 = dict(inp, x=inp["x"][perm], logits=inp["logits"][perm])
    out2, _ = orc.forward(p, inp2, nthreads=1)
    if not np.array_equal(out2, out[perm]):
        fail("token permutation does not commute with the output")
    pieces, start = [], 0
    for L in (5, 1, 6):
        sub = dict(inp, x=inp["x"][start:start + L], logits=inp["logits"][start:start + L])
        ps = oracle_mod.Problem(L, p.H, p.inter, p.E, p.k, p.bits, p.block, p.dtype)
        pieces.append(orc.forward(ps, sub, nthreads=1)[0])
        start += L
    if not np.array_equal(np.concatenate(pieces), out):
        fail("packed concatenation differs from per-sequence calls")


def pin_zero_weights(orc):
    """zero point equal to every code gives all-zero weights, hence exactly zero output."""
    shape, inp = _small_inputs(T=3, H=64, I=32, E=4, k=2, bits=4, block=32, explicit_zp=True)
    inp = dict(inp)
    for name, zpn in (("fc1_q", "fc1_zp"), ("fc2_q", "fc2_zp")):
        inp[name] = np.full_like(inp[name], 0x55)  # every code 5
        inp[zpn] = np.full_like(inp[zpn], 5)
    out, acc = orc.forward(problem_of(shape), inp, nthreads=1, want_acc=True)
    if np.any(acc != 0) or np.any(out & 0x7FFF):
        fail("zero weights did not give a zero output")


def pin_zero_weight_route_skipped(orc):
    """A route whose softmax weight underflows to exactly 0 adds nothing, even when
    its expert produces NaN (the finalizer skips zero-scale routes)."""
    shape, inp = _small_inputs(T=1, H=64, I=32, E=3, k=2, bits=4, block=32, dt=FP16)
    inp = dict(inp)
    inp["logits"] = _logits_bits([[0.0, -60000.0, -60000.0]], FP16)
    s = inp["fc2_s"].copy()
    s[1] = 0x7E00  # NaN scales in expert 1, the second route
    inp["fc2_s"] = s
    out, acc = orc.forward(problem_of(shape), inp, nthreads=1, want_acc=True)
    if not np.isfinite(acc).all():
        fail("zero-weight route was not skipped")
    _, _, y0 = dense_expert(inp, shape, 0, bits_to_f64(inp["x"], FP16)[0])
    if not np.allclose(acc[0], y0, rtol=1e-12, atol=1e-12):
        fail("single surviving route with weight 1")


def pin_full_softmax_routing(orc):
    """normalize_routing_weights = 0: each selected expert's weight is its
    probability under the softmax over all E logits (scipy), the selection is
    unchanged, and with k = E both readings give the full softmax."""
    rng = np.random.default_rng(8)
    for dt in (BF16, FP16):
        T, E, k = 7, 9, 3
        lv = rng.standard_normal((T, E)) * 2.0
        lg = _logits_bits(lv, dt)
        lvq = bits_to_f64(lg, dt)
        p = oracle_mod.Problem(T, 64, 32, E, k, 4, 32, dt, full_softmax=1)
        idx, w = orc.route(p, lg)
        idx_n, w_n = orc.route(oracle_mod.Problem(T, 64, 32, E, k, 4, 32, dt), lg)
        if not np.array_equal(idx, idx_n):
            fail("full softmax changes the selection")
        for t in range(T):
            full = scipy.special.softmax(lvq[t])
            if not np.allclose(w[t], full[idx[t]], rtol=1e-12, atol=0):
                fail(f"full-softmax weights of token {t}")
        pk = oracle_mod.Problem(T, 64, 32, E, E, 4, 32, dt, full_softmax=1)
        _, wk = orc.route(pk, lg)
        _, wk_n = orc.route(oracle_mod.Problem(T, 64, 32, E, E, 4, 32, dt), lg)
        if not np.allclose(wk, wk_n, rtol=1e-12, atol=0):
            fail("k = E: full softmax and renormalised weights differ")


def pin_biases_dense_over_experts(orc):
    """FC1 / FC2 biases: every expert for every token with the biases added after
    each matmul (torch float64), under both routing-weight readings."""
    for bits, block, dt, full in ((4, 32, BF16, 0), (2, 32, FP16, 1), (3, 64, BF16, 1)):
        shape, inp = _small_inputs(T=5, H=128, I=64, E=5, k=2, bits=bits, block=block, dt=dt, bias_std=0.5)
        p = problem_of(shape)
        p.full_softmax = full
        _, acc = orc.forward(p, inp, nthreads=2, want_acc=True)
        x = bits_to_f64(inp["x"], dt)
        lv = bits_to_f64(inp["logits"], dt)
        for t in range(shape.T):
            sel = sorted(range(shape.E), key=lambda e: (-lv[t, e], e))[: shape.k]
            wsel = scipy.special.softmax(lv[t])[sel] if full else scipy.special.softmax(lv[t, sel])
            total = np.zeros(shape.H)
            for e, w in zip(sel, wsel):
                total += w * dense_expert(inp, shape, e, x[t])[2]
            if not np.allclose(acc[t], total, rtol=1e-11, atol=1e-12):
                fail(f"biased layer bits={bits} full_softmax={full} token {t}")


def pin_fc2_bias_with_zero_weights(orc):
    """All weights zero (zero point equal to every code): each route's expert output
    is its FC2 bias, whatever the FC1 bias, so the layer gives sum_j w_j b2[e_j]."""
    shape, inp = _small_inputs(T=4, H=64, I=32, E=4, k=2, bits=4, block=32, explicit_zp=True, bias_std=1.0)
    inp = dict(inp)
    for name, zpn in (("fc1_q", "fc1_zp"), ("fc2_q", "fc2_zp")):
        inp[name] = np.full_like(inp[name], 0x33)  # every code 3
        inp[zpn] = np.full_like(inp[zpn], 3)
    p = problem_of(shape)
    idx, w = orc.route(p, inp["logits"])
    _, acc = orc.forward(p, inp, nthreads=1, want_acc=True)
    b2 = bits_to_f64(inp["fc2_b"], shape.dtype)
    want = np.einsum("tj,tjh->th", w, b2[idx])
    if not np.allclose(acc, want, rtol=1e-14, atol=0):
        fail("zero weights with biases: output is not the weighted FC2 biases")


def pin_full_softmax_nan_row(orc):
    """With full-softmax weights a NaN logit anywhere in a token's row (never
    selected: NaN ranks lowest) makes that token's weights NaN, as a softmax over
    the row would; the renormalised weights of the selected logits stay finite."""
    lv = np.array([[1.0, 0.5, np.nan, -1.0, 2.0], [0.1, 0.2, 0.3, 0.4, 0.5]])
    lg = _logits_bits(lv, BF16)
    for full in (0, 1):
        idx, w = orc.route(oracle_mod.Problem(2, 64, 32, 5, 2, 4, 32, BF16, full_softmax=full), lg)
        if 2 in idx[0]:
            fail("a NaN logit was selected")
        if full and not (np.isnan(w[0]).all() and np.isfinite(w[1]).all()):
            fail("full softmax: a NaN in the row must give NaN weights for that token only")
        if not full and not np.isfinite(w).all():
            fail("renormalised weights of finite selected logits must be finite")


def pin_nan_propagates(orc):
    shape, inp = _small_inputs(T=2, H=64, I=32, E=4, k=2, dt=BF16)
    inp = dict(inp)
    x = inp["x"].copy()
    x[1, 5] = 0x7FC0
    inp["x"] = x
    out, _ = orc.forward(problem_of(shape), inp, nthreads=1)
    nan = ((out & 0x7F80) == 0x7F80) & ((out & 0x7F) != 0)
    if not nan[1].all() or nan[0].any():
        fail("NaN input is not kept as NaN in exactly its token's outputs")


def _router_problem(T, H, E, dt):
    return oracle_mod.Problem(T, H, 32, E, 1, 4, 32, dt)


def pin_router_integer_bruteforce(orc):
    """Small-integer x and router weights: every product and sum is exact, so the
    logits equal Python integer dot products (rounded once when beyond 2^8)."""
    rng = np.random.default_rng(31)
    for dt in (BF16, FP16):
        T, H, E = 5, 48, 7
        xi = rng.integers(-4, 5, size=(T, H))
        wi = rng.integers(-3, 4, size=(E, H))
        xb = synthetic.float_to_bits(xi.astype(np.float64), dt)
        wb = synthetic.float_to_bits(wi.astype(np.float64), dt)
        got = orc.router_logits(_router_problem(T, H, E, dt), xb, wb)
        want = [[sum(int(a) * int(b) for a, b in zip(xi[t], wi[e])) for e in range(E)] for t in range(T)]
        ref = synthetic.float_to_bits(np.array(want, dtype=np.float64), dt)
        if not np.array_equal(got, ref):
            fail("router logits differ from integer dot products")


def pin_router_one_hot_and_layout(orc):
    """x = e_i gives logits[t][e] = w_router[e][i] exactly (the weight is [E][H],
    one row per expert): a transposed operand or a wrong stride fails."""
    rng = np.random.default_rng(32)
    T, H, E = 6, 40, 9
    wb = synthetic.float_to_bits(rng.standard_normal((E, H)), BF16)
    x = np.zeros((T, H))
    cols = rng.choice(H, size=T, replace=False)
    x[np.arange(T), cols] = 1.0
    got = orc.router_logits(_router_problem(T, H, E, BF16), synthetic.float_to_bits(x, BF16), wb)
    if not np.array_equal(got, wb[:, cols].T):
        fail("one-hot x does not select the router weight column")


def pin_router_rounding_and_scaling(orc):
    """Random x and weights: the logits are torch float64 matmul results rounded
    once to the dtype (numpy float16 for FP16); doubling x doubles them exactly;
    permuting the experts permutes the columns bit for bit."""
    rng = np.random.default_rng(33)
    T, H, E = 7, 96, 11
    for dt in (BF16, FP16):
        xb = synthetic.float_to_bits(rng.standard_normal((T, H)), dt)
        wb = synthetic.float_to_bits(rng.standard_normal((E, H)) * 0.05, dt)
        p = _router_problem(T, H, E, dt)
        got = orc.router_logits(p, xb, wb)
        ref64 = (torch.from_numpy(bits_to_f64(xb, dt)) @ torch.from_numpy(bits_to_f64(wb, dt)).T).numpy()
        if dt == FP16:
            ref = ref64.astype(np.float16).view(np.uint16)
        else:
            ref = synthetic.float_to_bits(ref64, dt)
        if (got != ref).mean() > 0.0:
            # a float64 sum order different from the oracle's may round across a tie
            # only when the value sits exactly on a rounding boundary
            if (got != ref).mean() > 0.01:
                fail("router logits are not the float64 dot products rounded once")
        x2 = synthetic.float_to_bits(bits_to_f64(xb, dt) * 2.0, dt)
        got2 = orc.router_logits(p, x2, wb)
        if not np.array_equal(bits_to_f64(got2, dt), 2.0 * bits_to_f64(got, dt)):
            fail("router logits are not linear in x")
        perm = rng.permutation(E)
        if not np.array_equal(orc.router_logits(p, xb, wb[perm]), got[:, perm]):
            fail("permuting the experts does not permute the logits")


def pin_fp4_element_and_scale_tables(orc):
    """E2M1: the closed set {0, 0.5, 1, 1.5, 2, 3, 4, 6}, increasing in the code's
    low three bits, bit 3 the sign; E4M3 against torch's float8_e4m3fn and E8M0
    against float8_e8m0fnu, every byte (NaN where torch has NaN)."""
    e2, e8, e4 = orc.fp4_tables()
    if not np.array_equal(e2[:8], [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]):
        fail("E2M1 magnitudes")
    if not np.array_equal(e2[8:], -e2[:8]) or not np.signbit(e2[8]):
        fail("E2M1 sign bit")
    b = torch.arange(256, dtype=torch.uint8)
    r4 = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    r8 = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for got, ref, name in ((e4, r4, "E4M3"), (e8, r8, "E8M0")):
        if not np.array_equal(np.isnan(got), np.isnan(ref)) or not np.array_equal(got[~np.isnan(ref)],
                                                                               ref[~np.isnan(ref)]):
            fail(f"{name} scale values")


def _fp4_dense_expert(inp, shape, e, xrow):
    """y of expert e from torch float64 with the weights decoded through torch's
    float8 dtypes (scales) and the E2M1 set (elements)."""
    e2m1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])

    def mat(q, s8, rows, K, g):
        codes = lsb_first_codes(q, 4, rows * K).reshape(rows, K)
        sb = torch.from_numpy(np.ascontiguousarray(s8, dtype=np.uint8).reshape(rows, K // shape.block))
        fdt = torch.float8_e8m0fnu if shape.format == 1 else torch.float8_e4m3fn
        scale = np.repeat(sb.view(fdt).to(torch.float64).numpy(), shape.block, axis=1)
        return torch.from_numpy(e2m1[codes] * scale * g)

    H, I = shape.H, shape.inter
    g1 = float(inp["g1"][e]) if shape.format == 2 else 1.0
    g2 = float(inp["g2"][e]) if shape.format == 2 else 1.0
    W1 = mat(inp["fc1_q"][e], inp["fc1_s"][e], 2 * I, H, g1)
    W2 = mat(inp["fc2_q"][e], inp["fc2_s"][e], H, I, g2)
    gu = W1 @ torch.from_numpy(xrow)
    h = torch.nn.functional.silu(gu[0::2]) * gu[1::2]
    return (W2 @ h).numpy()


def pin_fp4_dense_over_experts(orc):
    """MXFP4 and NVFP4 layers: the oracle's forward against every expert computed
    densely in torch float64 from the format definitions and weighted by the
    routing (brute force over experts), before the one rounding."""
    for fmt in (1, 2):
        shape = synthetic.Shape(T=3, H=64, inter=32, E=4, k=2, bits=4, block=32 if fmt == 1 else 16,
                                dtype=BF16, format=fmt)
        inp = synthetic.make_numpy(shape, synthetic.Recipe(logit_std=1.0), 40 + fmt)
        p = oracle_mod.Problem(shape.T, shape.H, shape.inter, shape.E, shape.k, shape.bits, shape.block,
                               shape.dtype, 0, fmt, inp.get("g1"), inp.get("g2"))
        _, acc = orc.forward(p, inp, nthreads=1, want_acc=True)
        x = bits_to_f64(inp["x"], shape.dtype)
        lg = bits_to_f64(inp["logits"], shape.dtype)
        for t in range(shape.T):
            order = sorted(range(shape.E), key=lambda e: (-lg[t, e], e))[:shape.k]
            w = scipy.special.softmax(lg[t, order])
            ref = sum(w[j] * _fp4_dense_expert(inp, shape, order[j], x[t]) for j in range(shape.k))
            if not np.allclose(acc[t], ref, rtol=1e-9, atol=1e-12):
                fail(f"FP4 format {fmt}: forward differs from the dense torch reference")


ALL_PINS = [
    pin_golden_packing, pin_unpack_random, pin_bits_to_double, pin_golden_rounding,
    pin_rounding_fp16_exhaustive, pin_rounding_bf16, pin_dequant, pin_golden_routing,
    pin_route_bruteforce, pin_permute, pin_dense_ffn_E1_k1, pin_bruteforce_dense_over_experts,
    pin_one_hot, pin_token_permutation, pin_zero_weights, pin_zero_weight_route_skipped,
    pin_nan_propagates, pin_full_softmax_routing, pin_biases_dense_over_experts,
    pin_fc2_bias_with_zero_weights, pin_full_softmax_nan_row, pin_router_integer_bruteforce,
    pin_router_one_hot_and_layout, pin_router_rounding_and_scaling, pin_fp4_element_and_scale_tables,
    pin_fp4_dense_over_experts,
]
