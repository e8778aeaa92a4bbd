"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of oracle.c (on the CPU), builds it,
routes the oracle module to it, and runs the pins of test_oracle.py: at least
one pin must fail.  The untouched source must pass them all.
"""
import os
import subprocess

import pytest

import oracle

from . import test_oracle as pins
from . import test_oracle_fp4 as fp4pins
from . import test_oracle_fp8 as fp8pins
from . import test_oracle_moe as moepins
from . import test_oracle_mx as mxpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "eps_outside_root": ("double inv_rms = 1.0 / sqrt(mean_sq + eps);", "double inv_rms = 1.0 / sqrt(mean_sq) + eps;"),
    "eps_dropped": ("double inv_rms = 1.0 / sqrt(mean_sq + eps);", "double inv_rms = 1.0 / sqrt(mean_sq);"),
    "mean_off_by_one": ("double mean_sq = sum_sq / (double)H;", "double mean_sq = sum_sq / (double)(H + 1);"),
    "gemma_without_one": ("return norm_kind == ORACLE_NORM_GEMMA ? 1.0 + g : g;", "return g;"),
    "gemma_always": ("return norm_kind == ORACLE_NORM_GEMMA ? 1.0 + g : g;", "return 1.0 + g;"),
    "residual_dropped": ("r[h] = bf16_bits_to_double(r0[t * H + h]) + y;", "r[h] = y;"),
    "residual_subtracted": ("r[h] = bf16_bits_to_double(r0[t * H + h]) + y;",
                            "r[h] = bf16_bits_to_double(r0[t * H + h]) - y;"),
    "weight_transposed": ("y += bf16_bits_to_double(xt[k]) * bf16_bits_to_double(wh[k]);",
                          "y += bf16_bits_to_double(xt[k]) * bf16_bits_to_double(W[(k % H) * K + (h % K)]);"),
    "weight_index_shift": ("y += bf16_bits_to_double(xt[k]) * bf16_bits_to_double(wh[k]);",
                           "y += bf16_bits_to_double(xt[k]) * bf16_bits_to_double(wh[(k + 1) % K]);"),
    "single_precision_dot": ("            double y = 0.0;", "            float y = 0.0f;"),
    "sum_of_abs": ("sum_sq += r[h] * r[h];", "sum_sq += fabs(r[h]);"),
    "norm_weight_ignored": ("o[h] = r[h] * inv_rms * norm_weight(gamma, h, norm_kind);", "o[h] = r[h] * inv_rms;"),
    "add_path_drops_y": ("r[h] = bf16_bits_to_double(r0[t * H + h]) + bf16_bits_to_double(y[t * H + h]);",
                         "r[h] = bf16_bits_to_double(r0[t * H + h]);"),
    "round_truncates": ("double qi = nearbyint(q);", "double qi = trunc(q);"),
    "round_ties_away": ("double qi = nearbyint(q);", "double qi = round(q);"),
    "e4m3_bias_8": ("v = ldexp(8.0 + (double)f, e - 10);", "v = ldexp(8.0 + (double)f, e - 11);"),
    "e4m3_subnormal_unit": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "e4m3_no_nan": ("    if (e == 15 && f == 7)\n        return NAN;\n", ""),
    "e4m3_sign_dropped": ("return sign ? -v : v;", "return v;"),
    "fp8_w_scale_by_token": ("double sw = (double)w_scale[w_per_row ? h : 0];",
                             "double sw = (double)w_scale[w_per_row ? (t % H) : 0];"),
    "fp8_x_scale_ignored": ("r[h] = bf16_bits_to_double(r0[t * H + h]) + sx * sw * dot;",
                            "r[h] = bf16_bits_to_double(r0[t * H + h]) + sw * dot;"),
    "fp8_x_scale_first_row": ("double sx = (double)x_scale[x_per_row ? t : 0];", "double sx = (double)x_scale[0];"),
    "e2m1_bias_2": ("double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 1);",
                    "double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 2);"),
    "e2m1_subnormal_one": ("double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 1);",
                           "double v = e == 0 ? 1.0 * f : ldexp(1.0 + 0.5 * f, e - 1);"),
    "nvfp4_nibbles_swapped": ("uint8_t code = (k & 1) ? (uint8_t)(wh[k / 2] >> 4) : (uint8_t)(wh[k / 2] & 0xF);",
                              "uint8_t code = (k & 1) ? (uint8_t)(wh[k / 2] & 0xF) : (uint8_t)(wh[k / 2] >> 4);"),
    "nvfp4_block_32": ("oracle_e4m3_to_double(sh[k / 16])", "oracle_e4m3_to_double(sh[k / 32])"),
    "nvfp4_tensor_scale_ignored": ("double w = (double)gs * oracle_e4m3_to_double(sh[k / 16])",
                                   "double w = oracle_e4m3_to_double(sh[k / 16])"),
    "e8m0_bias_128": ("return ldexp(1.0, (int)E - 127);", "return ldexp(1.0, (int)E - 128);"),
    "e8m0_nan_dropped": ("    if (E == 255)\n        return NAN;\n", ""),
    "mxfp4_block_16": ("oracle_e8m0_to_double(scales[k / 32])", "oracle_e8m0_to_double(scales[k / 16])"),
    "moe_ties_to_larger_index": ("if (best < 0 || (double)lt[e] > (double)lt[best])",
                                 "if (best < 0 || (double)lt[e] >= (double)lt[best])"),
    "moe_softmax_over_all_experts": ("for (long j = 0; j < k; ++j)\n            denom += exp((double)lt[it[j]] - top);",
                                     "for (long j = 0; j < E; ++j)\n            denom += exp((double)lt[j] - top);"),
    "moe_permute_slot_major": ("        for (long t = 0; t < T; ++t)\n            for (long j = 0; j < k; ++j)\n                if (ids[t * k + j] == e) {",
                               "        for (long j = 0; j < k; ++j)\n            for (long t = 0; t < T; ++t)\n                if (ids[t * k + j] == e) {"),
    "moe_gate_dropped": ("                r[h] += gate * dot;", "                r[h] += dot;"),
    "moe_wrong_expert": ("while (!(row >= offsets[e] && row < offsets[e + 1]))", "while (!(row >= offsets[e] && row <= offsets[e + 1]))"),
    "mxfp4_nibbles_swapped": ("(k % 2 == 0) ? (uint8_t)(byte & 0x0F) : (uint8_t)(byte >> 4);",
                              "(k % 2 == 0) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0x0F);"),
}


def _pin_calls():
    calls = [(f"hand[{c['name']}]", (lambda c=c: pins.test_hand_worked_cases(c))) for c in pins._load_cases()]
    for name in dir(pins):
        if name.startswith("test_") and name != "test_hand_worked_cases":
            calls.append((name, getattr(pins, name)))
    # FP8 pins (parametrized ones called with each of their parameters)
    for code, value in [(0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0xB8, -1.0)]:
        calls.append((f"fp8.format_facts[{code:#x}]", lambda c=code, v=value: fp8pins.test_format_facts(c, v)))
    for kind in (0, 1):
        calls.append((f"fp8.unit_scales[{kind}]", lambda k=kind: fp8pins.test_unit_scales_equal_bf16_region(k)))
    for name in dir(fp8pins):
        if name.startswith("test_") and name not in ("test_format_facts", "test_unit_scales_equal_bf16_region"):
            calls.append(("fp8." + name, getattr(fp8pins, name)))
    # NVFP4 pins
    for kind in (0, 1):
        calls.append((f"fp4.unit_scales[{kind}]", lambda k=kind: fp4pins.test_unit_scales_equal_bf16_region(k)))
    for name in dir(fp4pins):
        if name.startswith("test_") and name != "test_unit_scales_equal_bf16_region":
            calls.append(("fp4." + name, getattr(fp4pins, name)))
    # MoE pins
    for name in dir(moepins):
        if name.startswith("test_"):
            calls.append(("moe." + name, getattr(moepins, name)))
    # MXFP4 pins
    for kind in (0, 1):
        calls.append((f"mx.unit_scales[{kind}]", lambda k=kind: mxpins.test_unit_scales_equal_bf16_region(k)))
    for name in dir(mxpins):
        if name.startswith("test_") and name != "test_unit_scales_equal_bf16_region":
            calls.append(("mx." + name, getattr(mxpins, name)))
    return calls


def _failing_pins():
    failed = []
    for name, fn in _pin_calls():
        try:
            fn()
        except (AssertionError, ValueError, pytest.fail.Exception):
            failed.append(name)
    return failed


def _build(tmp_path, text, tag):
    src = tmp_path / f"oracle_{tag}.c"
    src.write_text(text)
    so = tmp_path / f"liboracle_{tag}.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", "-fno-fast-math",
                    "-ffp-contract=off", str(src), "-o", str(so), "-lm"], check=True)
    return str(so)


def test_unmodified_source_passes_every_pin(tmp_path):
    so = _build(tmp_path, open(SRC).read(), "clean")
    with oracle.using_library(so):
        assert _failing_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not unique"
    so = _build(tmp_path, text.replace(old, new), name)
    with oracle.using_library(so):
        failed = _failing_pins()
    assert failed, f"no pin caught the planted mistake {name}"
