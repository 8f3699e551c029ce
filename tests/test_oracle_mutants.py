"""Planted mistakes in the CPU oracle must each fail at least one pin.

Each case copies oracle/qmoe_oracle.c, applies one plausible mistake (a dropped
term, a wrong sign, index or operand, a swapped order), compiles the copy into
a temporary library and runs the pin set of tests/pins.py against it. The
planted mistakes live only in the temporary copy; the oracle itself is not
touched. CPU only.
"""
import os

import pytest

import oracle as oracle_mod
from tests import pins

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "qmoe_oracle.c")

MUTANTS = {
    "gate_up_swapped": ("silu(gu[2 * i]) * gu[2 * i + 1]", "silu(gu[2 * i + 1]) * gu[2 * i]"),
    "zero_point_sign": ("((double)code_at(qrow, bits, kk) - z) * s", "((double)code_at(qrow, bits, kk) + z) * s"),
    "combine_weight_dropped": ("acc[m] += w[j] * y[m];", "acc[m] += y[m];"),
    "tie_to_higher_index": ("  if (la != lb) return la > lb;\n  return a < b;", "  if (la != lb) return la > lb;\n  return a > b;"),
    "nibble_order": ("(kk % 2) ? (b >> 4) : (b & 0xF)", "(kk % 2) ? (b & 0xF) : (b >> 4)"),
    "scale_index": ("scales[row * nblk + b]", "scales[row + b]"),
    "silu_sign": ("z / (1.0 + exp(-z))", "z / (1.0 + exp(z))"),
    "fc1_expert_stride": ("(int64_t)expert * rows1 + n, wrow);", "(int64_t)expert * rows2 + n, wrow);"),
    "int3_field_order": ("(group >> (3 * (kk % 8))) & 0x7", "(group >> (3 * (7 - kk % 8))) & 0x7"),
    "int2_field_width": ("(b >> (2 * (kk % 4))) & 0x3", "(b >> (kk % 4)) & 0x3"),
    "ties_away_from_zero": ("rint(a / quantum)", "floor(a / quantum + 0.5)"),
    "zero_weight_not_skipped": ("if (w[j] == 0.0) continue;", ""),
    "last_route_dropped": ("for (int j = 0; j < p->k; ++j) {\n    if (w[j] == 0.0)", "for (int j = 0; j + 1 < p->k; ++j) {\n    if (w[j] == 0.0)"),
    "softmax_denominator": ("for (int j = 0; j < k; ++j) w[j] /= denom;", "for (int j = 0; j < k; ++j) w[j] /= denom + 1e-3;"),
    "permute_unstable": ("for (int64_t r = 0; r < R; ++r) {\n    const int64_t pos", "for (int64_t r = R - 1; r >= 0; --r) {\n    const int64_t pos"),
    "fp16_bias": ("const int bias = dtype == ORACLE_BF16 ? 127 : 15;", "const int bias = dtype == ORACLE_BF16 ? 127 : 16;"),
    "fp16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "fc2_reads_gate": ("for (int i = 0; i < I; ++i) acc += wrow[i] * h[i];", "for (int i = 0; i < I; ++i) acc += wrow[i] * gu[2 * i];"),
    "fc1_bias_dropped": ("    if (fc1_b) acc += oracle_bits_to_double(fc1_b[(int64_t)expert * rows1 + n], p->dtype);\n", ""),
    "fc1_bias_gate_up_swapped": ("fc1_b[(int64_t)expert * rows1 + n]", "fc1_b[(int64_t)expert * rows1 + (n ^ 1)]"),
    "fc2_bias_dropped": ("    if (fc2_b) acc += oracle_bits_to_double(fc2_b[(int64_t)expert * rows2 + m], p->dtype);\n", ""),
    "fc2_bias_wrong_expert": ("fc2_b[(int64_t)expert * rows2 + m]", "fc2_b[m]"),
    "full_softmax_ignored": ("  if (p->full_softmax) {", "  if (0) {"),
    "full_softmax_last_expert_dropped": ("for (int e = 0; e < E; ++e) denom += exp(", "for (int e = 0; e + 1 < E; ++e) denom += exp("),
    "router_weight_transposed": ("w_router[(int64_t)e * p->H + h]", "w_router[(int64_t)h * p->E + e]"),
    "router_last_term_dropped": ("      for (int h = 0; h < p->H; ++h)\n        acc += oracle_bits_to_double(x[t * p->H + h]",
                                 "      for (int h = 0; h + 1 < p->H; ++h)\n        acc += oracle_bits_to_double(x[t * p->H + h]"),
    "router_x_row_ignored": ("oracle_bits_to_double(x[t * p->H + h], p->dtype) *", "oracle_bits_to_double(x[h], p->dtype) *"),
    "e2m1_exponent_bias": ("ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    "e2m1_subnormal": ("e == 0 ? 0.5 * m :", "e == 0 ? 1.0 * m :"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e8m0_bias": ("ldexp(1.0, (int)bits - 127)", "ldexp(1.0, (int)bits - 128)"),
    "nvfp4_global_scale_dropped": ("(double)g[expert] : 1.0;", "1.0 : 1.0;"),
    "fp4_scale_block_index": ("s8[row * nblk + kk / p->block]", "s8[row * nblk + kk / 32]"),
    "x_not_read_per_token": ("xr[kk] = oracle_bits_to_double(J->x[t * H + kk], p->dtype);", "xr[kk] = oracle_bits_to_double(J->x[kk], p->dtype);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site of {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    lib = oracle_mod.compile_source(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle_mod.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            caught.append(f"{pin.__name__}: {e}")
            break
    assert caught, f"no pin catches the planted mistake {name}"
