"""Plant plausible mistakes in a copy of the oracle and check the pins catch them.

Each mutant edits one line of a temporary copy of oracle/oracle.c (never the
real file), compiles it with gcc on the CPU and reruns a selection of the pins
from test_oracle_pins.py against it. The test passes only if at least one pin
fails on the mutant, i.e. the pins are sensitive to that class of mistake.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    # a dropped term: the last block of every row is skipped
    "drop_last_block": (
        "double acc = 0.0, err = 0.0;\n        for (int64_t b = 0; b < nb; ++b) {\n            uint16_t dw, dx;",
        "double acc = 0.0, err = 0.0;\n        for (int64_t b = 0; b < nb - 1; ++b) {\n            uint16_t dw, dx;"),
    # a wrong sign of the Q4_0 offset
    "q4_offset_sign": (
        "q[j] = (int32_t)(blk[2 + j] & 0x0f) - 8;",
        "q[j] = (int32_t)(blk[2 + j] & 0x0f) + 8;"),
    # swapped nibble order (high nibble first)
    "q4_nibble_order": (
        "q[j] = (int32_t)(blk[2 + j] & 0x0f) - 8;\n            q[j + 16] = (int32_t)(blk[2 + j] >> 4) - 8;",
        "q[j] = (int32_t)(blk[2 + j] >> 4) - 8;\n            q[j + 16] = (int32_t)(blk[2 + j] & 0x0f) - 8;"),
    # a wrong index: activation block taken from the row index
    "wrong_x_index": (
        "int64_t s = block_dot(fmt, w + (r * nb + b) * bb, xq + b * 34, &dw, &dx);\n            double t",
        "int64_t s = block_dot(fmt, w + (r * nb + b) * bb, xq + (r % nb) * 34, &dw, &dx);\n            double t"),
    # a wrong operand: the weight scale used twice
    "scale_operand": (
        "oracle_half_to_double(dw) * oracle_half_to_double(dx) * (double)s;",
        "oracle_half_to_double(dw) * oracle_half_to_double(dw) * (double)s;"),
    # ties to even instead of ties away from zero in the quantizer
    "quant_round_even": ("float r = roundf(v);", "float r = rintf(v);"),
    # the quantizer scale computed with 128 instead of 127
    "quant_scale_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    # fp16 rounding by truncation
    "half_truncate": ("double m = rint(v * ldexp(1.0, 10 - expo));",
                      "double m = floor(v * ldexp(1.0, 10 - expo));"),
    # sigmoid with the wrong sign of the gate
    "sigmoid_sign": ("1.0 / (1.0 + exp(-*gate))", "1.0 / (1.0 + exp(*gate))"),
    # silu with the wrong sign inside the exponential
    "silu_sign": ("h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];", "h[i] = g[i] / (1.0 + exp(g[i])) * u[i];"),
    # argmax keeping the last index on ties
    "argmax_last_tie": ("if (y[i] > y[best])", "if (y[i] >= y[best])"),
    # the fp32-activation product reading the first block's activation for every block
    "xf32_x_index": ("(double)v[i] * (double)x[b * 32 + i]", "(double)v[i] * (double)x[i]"),
    # the fp32-activation product without the block scale
    "xf32_scale_dropped": ("acc += d * t;", "acc += t;"),
    # dp4a reading unsigned bytes
    "dp4a_unsigned": ("int8_t ab = (int8_t)(uint8_t)", "uint8_t ab = (uint8_t)"),
}

PINS = [
    pins.test_dp4a_smoke_value_from_pages,
    pins.test_dp4a_signed_bytes_and_accumulate,
    pins.test_float_to_half_rne_matches_ieee_binary16,
    pins.test_quantize_hand_worked_blocks,
    pins.test_quantize_zero_and_ties_away_from_zero,
    pins.test_hand_worked_block_sums_and_outputs,
    pins.test_hand_worked_two_block_row,
    pins.test_decode_block_q4_0_offset_and_order,
    lambda m: pins.test_oracle_equals_exact_rational_dmmv(m, 8, 4, 64),
    lambda m: pins.test_oracle_equals_exact_rational_dmmv(m, 2, 3, 160),
    pins.test_argmax_first_index_of_the_maximum,
    pins.test_accumulate_epilogue_hand_values,
    pins.test_swiglu_hand_values,
    pins.test_xf32_hand_worked_blocks,
    lambda m: pins.test_xf32_oracle_equals_exact_rational(m, 2, 3, 160),
]


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    d = tmp_path / "mut"
    d.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(src.replace(old, new))
    so = d / "liboracle_mut.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(d / "oracle.c"), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, old, new)
    caught = []
    with oracle.using_library(so):
        for pin in PINS:
            try:
                pin(oracle)
            except AssertionError:
                caught.append(getattr(pin, "__name__", "pin"))
    assert caught, f"no pin caught the planted mistake {name}"


def test_unmutated_copy_passes_all_selected_pins(tmp_path):
    so = _build_mutant(tmp_path, "float d = amax / 127.0f;", "float d = amax / 127.0f;")
    with oracle.using_library(so):
        for pin in PINS:
            pin(oracle)
