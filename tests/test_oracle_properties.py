"""Property-based pins of the CPU oracle (hypothesis): arbitrary block bytes, not
only the seeded distributions of the workloads.

* Block sums: for any Q8_0 / Q4_0 weight blocks and any Q8_0 activation blocks,
  the oracle's int32 block sums equal the integer dot product of the decoded
  codes, decoded here with numpy views (another decoder, another loop).
* DMMV: every term d_w * d_x * s_b is exact in fp64 (11 + 11 + 20 significant
  bits), so the oracle's fp64 row sum differs from the exact rational value by at
  most its summation rounding, nb * 2^-53 times the row's error scale, and the
  error scale is the sum of the terms' magnitudes to the same precision.
* Quantizer: for finite fp32 blocks, |q| <= 127, the largest magnitude maps to
  +-127, signs are kept, every code is within half a step (plus the fp32 product's
  rounding) of x / d, and the stored scale is numpy's IEEE binary16 rounding of
  the fp32 amax / 127.
Each property also catches, by itself, planted mistakes from the mutant harness
(test_properties_catch_planted_mistake). Not collected where hypothesis is missing
(tests/conftest.py).
"""
from fractions import Fraction

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402

Q4_0, Q8_0 = 2, 8

# finite binary16 bit patterns (exponent field 0..30), either sign
half_bits = st.builds(lambda s, e, m: (s << 15) | (e << 10) | m,
                      st.integers(0, 1), st.integers(0, 30), st.integers(0, 1023))


def _block(d_bits, payload):
    return np.concatenate([np.array([d_bits & 0xFF, d_bits >> 8], dtype=np.uint8),
                           np.array(payload, dtype=np.uint8)])


def blocks(fmt, n):
    nq = 32 if fmt == Q8_0 else 16
    one = st.builds(_block, half_bits, st.lists(st.integers(0, 255), min_size=nq, max_size=nq))
    return st.lists(one, min_size=n, max_size=n).map(np.concatenate)


@st.composite
def dmmv_case(draw):
    fmt = draw(st.sampled_from([Q8_0, Q4_0]))
    rows = draw(st.integers(1, 3))
    nb = draw(st.integers(1, 5))
    w = draw(blocks(fmt, rows * nb))
    xq = draw(blocks(Q8_0, nb))
    return fmt, rows, nb * 32, w, xq


def _codes(fmt, w, rows, nb):
    """Decoded weight codes [rows][nb][32] and fp16 scales [rows][nb] (numpy views)."""
    bb = 34 if fmt == Q8_0 else 18
    wb = w.reshape(rows, nb, bb)
    d = wb[:, :, :2].copy().view(np.float16)[..., 0].astype(np.float64)
    if fmt == Q8_0:
        v = wb[:, :, 2:].view(np.int8).astype(np.int64)
    else:
        qs = wb[:, :, 2:].astype(np.int64)
        v = np.concatenate([(qs & 15) - 8, (qs >> 4) - 8], axis=-1)
    return v, d


def check_block_sums(oracle_mod, case):
    fmt, rows, cols, w, xq = case
    nb = cols // 32
    wv, _ = _codes(fmt, w, rows, nb)
    xv, _ = _codes(Q8_0, xq, 1, nb)
    want = np.einsum("rbi,bi->rb", wv, xv[0])
    got = oracle_mod.block_sums(fmt, w, rows, cols, xq)
    assert np.array_equal(got.astype(np.int64), want)


def check_dmmv(oracle_mod, case):
    fmt, rows, cols, w, xq = case
    nb = cols // 32
    wv, wd = _codes(fmt, w, rows, nb)
    xv, xd = _codes(Q8_0, xq, 1, nb)
    y, e = oracle_mod.dmmv(fmt, w, rows, cols, xq)
    for r in range(rows):
        terms = [Fraction(float(wd[r, b])) * Fraction(float(xd[0, b])) * int(np.dot(wv[r, b], xv[0, b]))
                 for b in range(nb)]
        exact = sum(terms, Fraction(0))
        scale = sum((abs(t) for t in terms), Fraction(0))
        tol = Fraction(nb, 2 ** 53) * scale
        assert abs(Fraction(float(y[r])) - exact) <= tol
        assert abs(Fraction(float(e[r])) - scale) <= tol


_LIM = float(np.float32(2.0 ** 100))
finite_block = st.lists(st.floats(min_value=-_LIM, max_value=_LIM, allow_nan=False, width=32)
                        .filter(lambda v: v == 0.0 or abs(v) >= 2.0 ** -100), min_size=32, max_size=32)


def check_quantizer(oracle_mod, blocks_):
    x = np.array(blocks_, dtype=np.float32)
    out = oracle_mod.quantize_q8_0(x.reshape(-1)).reshape(len(blocks_), 34)
    for k in range(len(blocks_)):
        xb = x[k].astype(np.float64)
        q = out[k, 2:].view(np.int8).astype(np.int64)
        stored = out[k, :2].copy().view(np.float16)[0]
        amax = np.float32(np.max(np.abs(x[k])))
        d = np.float32(amax / np.float32(127.0))            # IEEE fp32 division
        with np.errstate(over="ignore"):                    # above 65504 the binary16 value is inf
            d16 = np.float16(d)
        assert stored == d16
        assert np.all(np.abs(q) <= 127)
        if amax == 0:
            assert np.all(q == 0)
            continue
        assert np.abs(q[np.argmax(np.abs(xb))]) == 127
        assert np.all((q == 0) | (np.sign(q) == np.sign(xb)))
        ratio = xb / float(d)
        # half a step, plus the fp32 reciprocal and product roundings (relative 2^-22 of the ratio)
        assert np.all(np.abs(q - ratio) <= 0.5 + np.abs(ratio) * 2.0 ** -21 + 1e-12)


quantizer_case = st.lists(finite_block, min_size=1, max_size=3)


@settings(max_examples=150, deadline=None, derandomize=True)
@given(dmmv_case())
def test_block_sums_equal_integer_dot_of_decoded_codes(oracle_mod, case):
    check_block_sums(oracle_mod, case)


@settings(max_examples=150, deadline=None, derandomize=True)
@given(dmmv_case())
def test_dmmv_within_fp64_summation_bound_of_exact_value(oracle_mod, case):
    check_dmmv(oracle_mod, case)


@settings(max_examples=200, deadline=None, derandomize=True)
@given(quantizer_case)
def test_quantizer_invariants_on_arbitrary_blocks(oracle_mod, blocks_):
    check_quantizer(oracle_mod, blocks_)


# planted mistakes (from the mutant harness) that these properties must catch by
# themselves: a dropped block, the Q4_0 offset sign and nibble order, a wrong
# activation index, a wrong scale operand and the quantizer's /128
PROPERTY_MUTANTS = ["drop_last_block", "q4_offset_sign", "q4_nibble_order", "wrong_x_index", "scale_operand",
                    "quant_scale_128"]


def _falsified(check, strategy, n=100) -> bool:
    """Whether a search of n generated cases (no shrinking) finds one that fails."""
    @settings(max_examples=n, deadline=None, derandomize=True, database=None, phases=[hyp.Phase.generate])
    @given(strategy)
    def run(case):
        check(oracle, case)
    try:
        run()
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name", PROPERTY_MUTANTS)
def test_properties_catch_planted_mistake(tmp_path, name):
    from tests.test_oracle_mutants import MUTANTS, _build_mutant
    so = _build_mutant(tmp_path, *MUTANTS[name])
    with oracle.using_library(so):
        caught = [c.__name__ for c, strat in ((check_block_sums, dmmv_case()), (check_dmmv, dmmv_case()),
                                              (check_quantizer, quantizer_case)) if _falsified(c, strat)]
    assert caught, f"no property caught the planted mistake {name}"
