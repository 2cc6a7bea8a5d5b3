"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

None of these compares the oracle with itself: each case is a value printed on
the pages (the dp4a smoke), a block worked out by hand from the block
definitions, exact rational arithmetic on tiny matrices (a different loop over a
different decoder), a library routine the oracle's helper must agree with
(numpy's IEEE binary16 conversion), or an invariant of the definition. Each
plausible mistake in the oracle (a dropped term, a wrong sign or offset, a
swapped nibble order, a transposed operand, a wrong rounding rule) fails at
least one of them; test_oracle_mutants.py plants such mistakes and checks it.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from gguf_block_quant_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
Q4_0, Q8_0 = 2, 8


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------- block building
def _vals(spec, n):
    """Expand a value spec from the golden files into n integers."""
    if spec.startswith("all:"):
        return [int(spec[4:], 0)] * n
    if spec.startswith("ramp:"):
        off = int(spec[5:])
        return [i + off for i in range(n)]
    if spec.startswith("onehot:"):
        k = int(spec[7:])
        return [1 if i == k else 0 for i in range(n)]
    if spec.startswith("first:"):
        first, rest = spec.split(",")
        return [int(first[6:], 0)] + [int(rest[5:], 0)] * (n - 1)
    raise ValueError(spec)


def block_q8(d_bits, q):
    b = np.zeros(34, dtype=np.uint8)
    d = int(d_bits, 0) if isinstance(d_bits, str) else int(d_bits)
    b[0], b[1] = d & 0xFF, d >> 8
    b[2:] = np.array(q, dtype=np.int64).astype(np.int8).view(np.uint8)
    return b


def block_q4(d_bits, qs_bytes):
    b = np.zeros(18, dtype=np.uint8)
    d = int(d_bits, 0)
    b[0], b[1] = d & 0xFF, d >> 8
    b[2:] = np.array(qs_bytes, dtype=np.uint8)
    return b


# ------------------------------------------------------------------- pages
def test_dp4a_smoke_value_from_pages(oracle_mod):
    g = load("dp4a_smoke.json")
    a = oracle_mod.pack_int8x4(g["a"])
    b = oracle_mod.pack_int8x4(g["b"])
    assert oracle_mod.dp4a(a, b, g["c"]) == g["expect"] == 70


def test_dp4a_signed_bytes_and_accumulate(oracle_mod):
    # (-1)*(-1) + 127*(-128) + (-128)*(-128) + 0*5 = 1 - 16256 + 16384 = 129, plus c
    a = oracle_mod.pack_int8x4([-1, 127, -128, 0])
    b = oracle_mod.pack_int8x4([-1, -128, -128, 5])
    assert oracle_mod.dp4a(a, b, 1000) == 1129


# -------------------------------------------------------------------- fp16
def test_half_to_double_matches_ieee_binary16_for_every_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_float_to_half_rne_matches_ieee_binary16(oracle_mod):
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32),
        (g.uniform(1e-3, 1e-2, 2000)).astype(np.float32),
        (g.standard_normal(2000) * 1e-6).astype(np.float32),     # subnormal halves
        (g.standard_normal(1000) * 3e4).astype(np.float32),      # near overflow
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24,
                  2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -14, 6.1e-5, 1.0 / 127.0],
                 dtype=np.float32),
    ])
    # exact midpoints between neighbouring halves exercise ties-to-even
    h = np.arange(0x0001, 0x7bff, 97, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.float_to_half_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- quantizer
def test_quantize_hand_worked_blocks(oracle_mod):
    for case in load("quantize_hand.json")["cases"]:
        x = np.zeros(32, dtype=np.float32)
        x[: len(case["x"])] = case["x"]
        blk = oracle_mod.quantize_q8_0(x)
        d_bits = int(blk[0]) | (int(blk[1]) << 8)
        assert d_bits == int(case["d_bits"], 0), case["name"]
        q = blk[2:].view(np.int8).astype(int)
        want = np.zeros(32, dtype=int)
        want[: len(case["q"])] = case["q"]
        assert np.array_equal(q, want), case["name"]


def test_quantize_invariants_on_random_blocks(oracle_mod):
    x = synth.activations(32 * 512, seed=11)
    xq = oracle_mod.quantize_q8_0(x).reshape(-1, 34)
    xb = x.reshape(-1, 32).astype(np.float64)
    q = xq[:, 2:].view(np.int8).astype(np.int64)
    d16 = xq[:, :2].copy().view(np.float16).reshape(-1).astype(np.float64)
    assert np.all(np.abs(q) <= 127)
    # the element of largest magnitude maps to +-127
    arg = np.argmax(np.abs(xb), axis=1)
    assert np.all(np.abs(q[np.arange(len(q)), arg]) == 127)
    # reconstruction error with the fp32 scale: |x - d*q| <= d/2 (+ fp32 rounding)
    d32 = (np.max(np.abs(xb), axis=1) / 127.0)
    err = np.abs(xb - d32[:, None] * q)
    assert np.all(err <= d32[:, None] * (0.5 + 1e-5))
    # the stored scale is the fp16 rounding of the fp32 scale
    assert np.all(np.abs(d16 - d32) <= np.abs(d32) * 2.0 ** -11)


@pytest.mark.parametrize("k", [-3, -1, 1, 4])
def test_quantize_commutes_with_power_of_two_scaling(oracle_mod, k):
    x = synth.activations(32 * 64, seed=12)
    a = oracle_mod.quantize_q8_0(x).reshape(-1, 34)
    b = oracle_mod.quantize_q8_0((x * np.float32(2.0 ** k)).astype(np.float32)).reshape(-1, 34)
    assert np.array_equal(a[:, 2:], b[:, 2:])          # identical int8 codes
    da = a[:, :2].copy().view(np.uint16).reshape(-1).astype(np.int64)
    db = b[:, :2].copy().view(np.uint16).reshape(-1).astype(np.int64)
    assert np.array_equal(db - da, np.full_like(da, k << 10))  # exponent field moves by k


def test_quantize_zero_and_ties_away_from_zero(oracle_mod):
    z = oracle_mod.quantize_q8_0(np.zeros(64, dtype=np.float32))
    assert not z.any()
    x = np.zeros(32, dtype=np.float32)
    x[0] = 127.0
    x[1:9] = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5]
    q = oracle_mod.quantize_q8_0(x)[2:].view(np.int8)
    assert list(q[1:9]) == [1, 2, 3, 4, -1, -2, -3, -4]


# ----------------------------------------------------------------- blocks
def _hand_case_blocks(case):
    if case["fmt"] == "q8_0":
        w = block_q8(case["w_d"], _vals(case["w_q"], 32))
        fmt = Q8_0
    else:
        w = block_q4(case["w_d"], _vals(case["w_qs_bytes"], 16))
        fmt = Q4_0
    x = block_q8(case["x_d"], _vals(case["x_q"], 32))
    return fmt, w, x


def test_hand_worked_block_sums_and_outputs(oracle_mod):
    for case in load("hand_blocks.json")["cases"]:
        fmt, w, x = _hand_case_blocks(case)
        s = oracle_mod.block_sums(fmt, w, 1, 32, x)
        assert s[0, 0] == case["s"], case["name"]
        y, e = oracle_mod.dmmv(fmt, w, 1, 32, x)
        assert y[0] == case["y"], case["name"]
        assert e[0] == abs(case["y"]), case["name"]


def test_hand_worked_two_block_row(oracle_mod):
    g = load("hand_blocks.json")["two_block_row"]
    w = np.concatenate([block_q8(b["d"], _vals(b["q"], 32)) for b in g["w"]])
    x = np.concatenate([block_q8(b["d"], _vals(b["q"], 32)) for b in g["x"]])
    assert list(oracle_mod.block_sums(Q8_0, w, 1, 64, x)[0]) == g["s"]
    y, e = oracle_mod.dmmv(Q8_0, w, 1, 64, x)
    assert y[0] == g["y"] and e[0] == g["e"]


def test_decode_block_q4_0_offset_and_order(oracle_mod):
    qs = np.arange(16, dtype=np.uint8) | (np.arange(15, -1, -1, dtype=np.uint8) << 4)
    d, q = oracle_mod.decode_block(Q4_0, block_q4("0x3c00", qs))
    assert d == 0x3C00
    assert list(q[:16]) == [j - 8 for j in range(16)]
    assert list(q[16:]) == [15 - j - 8 for j in range(16)]


# --------------------------------------------------- exact rational brute force
def _exact_dmmv(fmt, w, rows, cols, xq):
    """Exact y via Fractions, decoding blocks with numpy views (a different
    decoder and a different loop from the oracle's)."""
    nb = cols // 32
    xb = xq.reshape(nb, 34)
    xd = xb[:, :2].copy().view(np.float16).reshape(-1)
    xv = xb[:, 2:].view(np.int8).astype(int)
    if fmt == Q8_0:
        wb = w.reshape(rows, nb, 34)
        wd = wb[:, :, :2].copy().view(np.float16)[..., 0]
        wv = wb[:, :, 2:].view(np.int8).astype(int)
    else:
        wb = w.reshape(rows, nb, 18)
        wd = wb[:, :, :2].copy().view(np.float16)[..., 0]
        qs = wb[:, :, 2:].astype(int)
        wv = np.concatenate([(qs & 15) - 8, (qs >> 4) - 8], axis=-1)
    out = []
    for r in range(rows):
        acc = Fraction(0)
        for b in range(nb):
            s = sum(int(wv[r, b, i]) * int(xv[b, i]) for i in range(32))
            acc += Fraction(float(wd[r, b])) * Fraction(float(xd[b])) * s
        out.append(acc)
    return out


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
@pytest.mark.parametrize("rows,cols", [(1, 32), (4, 64), (3, 160)])
def test_oracle_equals_exact_rational_dmmv(oracle_mod, fmt, rows, cols):
    w = synth.weight_blocks(fmt, rows, cols, seed=21 + rows)
    xq = synth.activation_blocks(cols // 32, seed=22 + cols)
    y, e = oracle_mod.dmmv(fmt, w, rows, cols, xq)
    exact = _exact_dmmv(fmt, w, rows, cols, xq)
    for r in range(rows):
        assert abs(Fraction(y[r]) - exact[r]) <= abs(exact[r]) * Fraction(1, 10 ** 15) + Fraction(1, 10 ** 300)
        assert e[r] >= abs(y[r]) * (1 - 1e-15)


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_oracle_equals_dequantized_float_dot(oracle_mod, fmt):
    rows, cols = 4, 64
    w = synth.weight_blocks(fmt, rows, cols, seed=31)
    x = synth.activations(cols, seed=32)
    xq = oracle_mod.quantize_q8_0(x)
    wf = oracle_mod.dequantize(fmt, w).reshape(rows, cols)
    xf = oracle_mod.dequantize(Q8_0, xq)
    ref = np.array([sum(float(wf[r, i]) * float(xf[i]) for i in range(cols)) for r in range(rows)])
    y, _ = oracle_mod.dmmv(fmt, w, rows, cols, xq)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-300)


# -------------------------------------------------------------- invariants
@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
@pytest.mark.parametrize("k", [-2, 3])
def test_dmmv_scales_exactly_with_power_of_two_input(oracle_mod, fmt, k):
    rows, cols = 16, 256
    w = synth.weight_blocks(fmt, rows, cols, seed=41)
    x = synth.activations(cols, seed=42)
    y1, _ = oracle_mod.dmmv(fmt, w, rows, cols, oracle_mod.quantize_q8_0(x))
    xs = (x * np.float32(2.0 ** k)).astype(np.float32)
    y2, _ = oracle_mod.dmmv(fmt, w, rows, cols, oracle_mod.quantize_q8_0(xs))
    assert np.array_equal(y2, y1 * 2.0 ** k)


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_dmmv_row_permutation_equivariance(oracle_mod, fmt):
    rows, cols = 37, 128
    bb = 34 if fmt == Q8_0 else 18
    w = synth.weight_blocks(fmt, rows, cols, seed=51)
    xq = synth.activation_blocks(cols // 32, seed=52)
    perm = np.random.default_rng(5).permutation(rows)
    wp = w.reshape(rows, -1)[perm].reshape(-1)
    y, _ = oracle_mod.dmmv(fmt, w, rows, cols, xq)
    yp, _ = oracle_mod.dmmv(fmt, wp, rows, cols, xq)
    assert np.array_equal(yp, y[perm])
    assert w.size == rows * cols // 32 * bb


def test_q4_0_offset_identity(oracle_mod):
    """sum (q-8) x = sum q x - 8 sum x, with q re-encoded as a Q8_0 block."""
    rows, cols = 8, 128
    nb = cols // 32
    w4 = synth.weight_blocks(Q4_0, rows, cols, seed=61)
    xq = synth.activation_blocks(nb, seed=62)
    qs = w4.reshape(rows * nb, 18)[:, 2:]
    q = np.concatenate([qs & 15, qs >> 4], axis=1).astype(np.int8)   # 0..15, no offset
    w8 = np.zeros((rows * nb, 34), dtype=np.uint8)
    w8[:, :2] = w4.reshape(rows * nb, 18)[:, :2]
    w8[:, 2:] = q.view(np.uint8)
    ones = np.zeros((1 * nb, 34), dtype=np.uint8)
    ones[:, 0:2] = np.frombuffer(np.float16(1.0).tobytes(), dtype=np.uint8)
    ones[:, 2:] = 1
    s4 = oracle_mod.block_sums(Q4_0, w4, rows, cols, xq)
    s8 = oracle_mod.block_sums(Q8_0, w8.reshape(-1), rows, cols, xq)
    sx = oracle_mod.block_sums(Q8_0, ones.reshape(-1), 1, cols, xq)[0]
    assert np.array_equal(s4, s8 - 8 * sx[None, :])


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_zero_scales_give_zero_rows(oracle_mod, fmt):
    rows, cols = 5, 96
    bb = 34 if fmt == Q8_0 else 18
    w = synth.weight_blocks(fmt, rows, cols, seed=71).reshape(-1, bb).copy()
    w[:, :2] = 0
    xq = synth.activation_blocks(cols // 32, seed=72)
    y, e = oracle_mod.dmmv(fmt, w.reshape(-1), rows, cols, xq)
    assert not y.any() and not e.any()


def test_block_sums_reproduce_dmmv(oracle_mod):
    rows, cols = 6, 192
    w = synth.weight_blocks(Q8_0, rows, cols, seed=81)
    xq = synth.activation_blocks(cols // 32, seed=82)
    s = oracle_mod.block_sums(Q8_0, w, rows, cols, xq)
    dw = w.reshape(rows, -1, 34)[:, :, :2].copy().view(np.float16)[..., 0].astype(np.float64)
    dx = xq.reshape(-1, 34)[:, :2].copy().view(np.float16).reshape(-1).astype(np.float64)
    y, _ = oracle_mod.dmmv(Q8_0, w, rows, cols, xq)
    ref = [sum(dw[r, b] * dx[b] * s[r, b] for b in range(cols // 32)) for r in range(rows)]
    np.testing.assert_allclose(y, ref, rtol=1e-15)


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_batched_equals_separate_calls(oracle_mod, fmt):
    rows, cols, batch = 9, 128, 4
    w = synth.weight_blocks(fmt, rows, cols, seed=91)
    xq = synth.activation_blocks(batch * cols // 32, seed=92)
    yb, eb = oracle_mod.dmmv_batched(fmt, w, rows, cols, xq, batch)
    for v in range(batch):
        y, e = oracle_mod.dmmv(fmt, w, rows, cols, xq.reshape(batch, -1)[v])
        assert np.array_equal(yb[v], y) and np.array_equal(eb[v], e)


def test_expert_gather_equals_separate_calls_and_flags_bad_index(oracle_mod):
    rows, cols, n_exp = 6, 64, 5
    per = rows * cols // 32 * 18
    stack = synth.weight_blocks(Q4_0, n_exp * rows, cols, seed=101)
    xq = synth.activation_blocks(3 * cols // 32, seed=102)
    idx = np.array([4, 0, 2], dtype=np.int32)
    y, e, st = oracle_mod.expert_gather(Q4_0, stack, per, rows, cols, idx, n_exp,
                                        xq, cols // 32 * 34)
    assert st == 0
    for k, ex in enumerate(idx):
        yk, _ = oracle_mod.dmmv(Q4_0, stack[ex * per:(ex + 1) * per], rows, cols,
                                xq.reshape(3, -1)[k])
        assert np.array_equal(y[k], yk)
    # shared activation (stride 0) and an out-of-range index
    y2, _, st2 = oracle_mod.expert_gather(Q4_0, stack, per, rows, cols,
                                          np.array([1, 5, -1], dtype=np.int32), n_exp,
                                          xq, 0)
    assert st2 == 1
    assert np.all(np.isnan(y2[1])) and np.all(np.isnan(y2[2]))
    y1, _ = oracle_mod.dmmv(Q4_0, stack[per:2 * per], rows, cols, xq.reshape(3, -1)[0])
    assert np.array_equal(y2[0], y1)


# ------------------------------------------------------------------ repack
def test_repack_hand_example_and_round_trip(oracle_mod):
    src = np.arange(18, dtype=np.uint8)           # one Q4_0 block: d bytes 0,1 then qs 2..17
    dst = oracle_mod.repack(Q4_0, src, 1, 32)
    assert list(dst) == list(range(2, 18)) + [0, 1]
    for fmt, rows, cols in [(Q8_0, 7, 96), (Q4_0, 5, 256)]:
        w = synth.weight_blocks(fmt, rows, cols, seed=111)
        r = oracle_mod.repack(fmt, w, rows, cols)
        assert np.array_equal(np.sort(r), np.sort(w))
        assert np.array_equal(oracle_mod.unpack(fmt, r, rows, cols), w)


# --------------------------------------------------------------- tolerance
def test_within_tolerance_criterion(oracle_mod):
    ok, worst = oracle_mod.within_tolerance([1.0 + 1e-5], [1.0], [1.0])
    assert ok and worst < 1.0
    ok, _ = oracle_mod.within_tolerance([1.0 + 2e-5], [1.0], [1.0])
    assert not ok


# ------------------------------------------------------------------ argmax
def test_argmax_first_index_of_the_maximum(oracle_mod):
    assert oracle_mod.argmax([1.0, 3.0, 2.0]) == (1, 3.0)
    assert oracle_mod.argmax([5.0, 5.0, 1.0])[0] == 0            # ties: the smallest index
    assert oracle_mod.argmax([-2.0, -1.0, -1.0, -3.0])[0] == 1
    assert oracle_mod.argmax([7.0])[0] == 0
    assert oracle_mod.argmax(np.zeros(0))[0] == -1
    g = np.random.default_rng(4)
    v = g.standard_normal(10007)
    assert oracle_mod.argmax(v)[0] == int(np.argmax(v))


# --------------------------------------------------------------- epilogues
def test_accumulate_epilogue_hand_values(oracle_mod):
    """Hand-worked: the Q8_0 block of hand_blocks' 'qw=1, qx=127' case gives
    W.x = 31.75; with gate 0, sigmoid(0) = 1/2 exactly."""
    case = [c for c in load("hand_blocks.json")["cases"] if c["name"] == "q8_0 qw=1 qx=127"][0]
    fmt, w, x = _hand_case_blocks(case)
    y, e = oracle_mod.dmmv_acc(fmt, w, 1, 32, x, [1.0])
    assert y[0] == 1.0 + 31.75 and e[0] == 31.75
    y, e = oracle_mod.dmmv_acc(fmt, w, 1, 32, x, [-2.0], gate=0.0)
    assert y[0] == -2.0 + 0.5 * 31.75 and e[0] == 0.5 * 31.75
    # a large gate saturates the sigmoid to 1, a very negative one to 0
    y, _ = oracle_mod.dmmv_acc(fmt, w, 1, 32, x, [0.0], gate=60.0)
    assert abs(y[0] - 31.75) < 1e-20 * 31.75 + 1e-12
    y, _ = oracle_mod.dmmv_acc(fmt, w, 1, 32, x, [3.0], gate=-800.0)
    assert y[0] == 3.0


def test_accumulate_equals_dmmv_plus_y(oracle_mod):
    rows, cols = 7, 96
    w = synth.weight_blocks(Q4_0, rows, cols, seed=201)
    xq = synth.activation_blocks(cols // 32, seed=202)
    y0 = np.linspace(-1, 1, rows)
    y, e = oracle_mod.dmmv_acc(Q4_0, w, rows, cols, xq, y0)
    d, de = oracle_mod.dmmv(Q4_0, w, rows, cols, xq)
    assert np.array_equal(y, y0 + d) and np.array_equal(e, de)


def test_swiglu_hand_values(oracle_mod):
    h = oracle_mod.swiglu([0.0, 1.0, -1.0, 40.0, -40.0, 2.0], [3.0, 2.0, 2.0, 0.5, 7.0, -1.0])
    e = np.e
    want = [0.0, 2.0 / (1 + 1 / e), -2.0 / (1 + e), 20.0, -40.0 * 7.0 / (1 + e ** 40), -2.0 / (1 + e ** -2)]
    np.testing.assert_allclose(h, want, rtol=1e-14, atol=1e-300)
    assert h[1] == 2.0 / (1.0 + np.exp(-1.0))            # 1.4621171572600098
    assert abs(h[1] - 1.4621171572600098) < 1e-15


# ------------------------------------------------- fp32-activation product
def _exact_dmmv_xf32(fmt, w, rows, cols, x):
    """Exact W.x for fp32 x via Fractions, decoding blocks with numpy views."""
    nb = cols // 32
    if fmt == Q8_0:
        wb = w.reshape(rows, nb, 34)
        wv = wb[:, :, 2:].view(np.int8).astype(int)
    else:
        wb = w.reshape(rows, nb, 18)
        qs = wb[:, :, 2:].astype(int)
        wv = np.concatenate([(qs & 15) - 8, (qs >> 4) - 8], axis=-1)
    wd = wb[:, :, :2].copy().view(np.float16)[..., 0]
    xf = [Fraction(float(v)) for v in np.asarray(x, dtype=np.float32)]
    out, scale = [], []
    for r in range(rows):
        acc, err = Fraction(0), Fraction(0)
        for b in range(nb):
            d = Fraction(float(wd[r, b]))
            terms = [d * int(wv[r, b, i]) * xf[32 * b + i] for i in range(32)]
            acc += sum(terms)
            err += sum(abs(t) for t in terms)
        out.append(acc)
        scale.append(err)
    return out, scale


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 160)])
def test_xf32_oracle_equals_exact_rational(oracle_mod, fmt, rows, cols):
    w = synth.weight_blocks(fmt, rows, cols, seed=61 + rows)
    x = synth.activations(cols, seed=62 + cols)
    y, e = oracle_mod.dmmv_xf32(fmt, w, rows, cols, x)
    exact, scale = _exact_dmmv_xf32(fmt, w, rows, cols, x)
    for r in range(rows):
        assert abs(Fraction(y[r]) - exact[r]) <= scale[r] * Fraction(1, 10 ** 14)
        assert abs(Fraction(e[r]) - scale[r]) <= scale[r] * Fraction(1, 10 ** 14)


def test_xf32_hand_worked_blocks(oracle_mod):
    # Q8_0, d = 1.0, every q = 1, x = 0.5 everywhere: 32 * 0.5 = 16
    w8 = block_q8("0x3c00", [1] * 32)
    y, e = oracle_mod.dmmv_xf32(Q8_0, w8, 1, 32, np.full(32, 0.5, dtype=np.float32))
    assert y[0] == 16.0 and e[0] == 16.0
    # Q4_0, d = 0.5, every qs byte 0xF0: elements 0..15 are 0 - 8, 16..31 are 15 - 8
    w4 = block_q4("0x3800", [0xF0] * 16)
    y, e = oracle_mod.dmmv_xf32(Q4_0, w4, 1, 32, np.ones(32, dtype=np.float32))
    assert y[0] == 0.5 * (16 * -8 + 16 * 7) and e[0] == 0.5 * (16 * 8 + 16 * 7)
    x = np.zeros(32, dtype=np.float32)
    x[20] = 3.0                                  # high nibble of qs byte 4: value 7
    y, _ = oracle_mod.dmmv_xf32(Q4_0, w4, 1, 32, x)
    assert y[0] == 0.5 * 7 * 3.0
    # two blocks of a row: the second block's activation is x[32..63]
    w2 = np.concatenate([block_q8("0x3c00", [1] * 32), block_q8("0x4000", [-2] * 32)])
    x2 = np.concatenate([np.full(32, 0.25, dtype=np.float32), np.full(32, 1.0, dtype=np.float32)])
    y, _ = oracle_mod.dmmv_xf32(Q8_0, w2, 1, 64, x2)
    assert y[0] == 32 * 0.25 + 2.0 * (-2) * 32


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_xf32_equals_quantized_product_when_x_is_representable(oracle_mod, fmt):
    """An x that Q8_0 represents exactly (x = 2^-7 * q, every block holding a
    +-127) quantizes to itself, so both products are the same sums in the same
    order: bit for bit equal."""
    rows, cols = 9, 256
    w = synth.weight_blocks(fmt, rows, cols, seed=71)
    rng = np.random.default_rng(72)
    q = rng.integers(-127, 128, size=cols)
    q[::32] = 127
    x = (q * 2.0 ** -7).astype(np.float32)
    xq = oracle_mod.quantize_q8_0(x)
    assert np.array_equal(oracle_mod.dequantize(Q8_0, xq), x.astype(np.float64))
    y1, e1 = oracle_mod.dmmv(fmt, w, rows, cols, xq)
    y2, e2 = oracle_mod.dmmv_xf32(fmt, w, rows, cols, x)
    assert np.array_equal(y1, y2)
