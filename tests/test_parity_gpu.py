"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar (fixed by the method's statement): per-block int32 dot products are bit for
bit the oracle's; every fp32 output row satisfies
    |y - y_ref| <= 1e-5 * sum_b |d_w d_x s_b| + 1e-6
where y_ref and the error scale come from the oracle (fp64); the quantizer's
bytes are bit for bit the oracle's. Every output buffer is pre-filled with a NaN
sentinel so rows the kernel never wrote show up.

Inputs come from gguf_block_quant_gb300.synth (seeded draws, no arithmetic of
the method); expected values only from oracle/.
"""
import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu

Q4_0, Q8_0 = Z.Q4_0, Z.Q8_0
REL, ABS = 1e-5, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    Z.lib()
    Z.device_status(clear=True)
    yield
    assert Z.device_status() == 0, "a kernel reported a device fault"


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def nan_out(*shape) -> torch.Tensor:
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def check_y(y: torch.Tensor, y_ref, e_ref):
    yh = y.double().cpu().numpy().reshape(np.shape(y_ref))
    assert not np.isnan(yh).any(), "some rows were never written (NaN sentinel)"
    ok, worst = oracle.within_tolerance(yh, y_ref, e_ref, REL, ABS)
    assert ok, f"tolerance exceeded: worst |dy|/bound = {worst:.3g}"
    return worst


def run_dmmv(fmt, w_np, rows, cols, xq_np, layout=Z.GGUF, w_dev=None):
    w = w_dev if w_dev is not None else dev(w_np)
    if layout == Z.REPACKED and w_dev is None:
        w = Z.repack(fmt, w, rows, cols)
    y = nan_out(rows)
    Z.dmmv(fmt, w, rows, cols, dev(xq_np), y=y, layout=layout)
    torch.cuda.synchronize()
    return y


# ----------------------------------------------------------------- dp4a smoke
def test_dp4a_selftest_pages_value_and_random():
    pack = oracle.pack_int8x4
    a = [pack([1, 2, 3, 4])]
    b = [pack([5, 6, 7, 8])]
    c = [0]
    g = np.random.default_rng(3)
    for _ in range(500):
        a.append(int(g.integers(0, 1 << 32)))
        b.append(int(g.integers(0, 1 << 32)))
        c.append(int(g.integers(-(1 << 20), 1 << 20)))
    to_i32 = lambda v: np.array(v, dtype=np.uint32).view(np.int32)
    out = Z.selftest_dp4a(dev(to_i32(a)), dev(to_i32(b)), dev(np.array(c, dtype=np.int32)))
    out = out.cpu().numpy()
    assert out[0] == 70
    ref = [oracle.dp4a(int(x), int(y), int(z)) for x, y, z in zip(a, b, c)]
    assert list(out) == ref


# ----------------------------------------------------------------- quantizer
@pytest.mark.parametrize("k", [32, 2048, 4096, 32 * 1001, 4096 * 8])
def test_quantize_bit_exact(k):
    x = synth.activations(k, seed=k)
    xq = Z.quantize_act_q8_0(dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_q8_0(x))


def test_quantize_bit_exact_special_blocks():
    blocks = []
    for case in [[127.0, 2.5, -2.5, 0.5, -0.5, 1.5, 63.5, -127.0], [-254.0, 3.0, -3.0, 1.0, 100.0],
                 [], [1.0, -1.0], [1e-30, -3e-31], [60000.0, -1.0], [5e-8, 1e-8]]:
        b = np.zeros(32, dtype=np.float32)
        b[:len(case)] = case
        blocks.append(b)
    g = np.random.default_rng(9)
    for s in (1e-6, 1e-2, 1.0, 1e3):
        blocks.append((g.standard_normal(32) * s).astype(np.float32))
    x = np.concatenate(blocks)
    xq = Z.quantize_act_q8_0(dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_q8_0(x))


# -------------------------------------------------- dense DMMV vs the oracle
SHAPES = [
    # (fmt, rows, cols): pipelined-kernel shapes (cols % 256 == 0) with ragged
    # row counts spanning several tiles, and plain-kernel shapes
    (Q8_0, 64, 2048), (Q8_0, 1000, 512), (Q8_0, 777, 1024), (Q8_0, 1531, 4096), (Q8_0, 301, 8192),
    (Q4_0, 4096, 4096), (Q4_0, 2999, 2048), (Q4_0, 513, 512), (Q4_0, 257, 8192),
    (Q8_0, 1, 32), (Q8_0, 37, 96), (Q4_0, 53, 160), (Q4_0, 5, 224), (Q8_0, 19, 14336), (Q4_0, 33, 16384),
]


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", SHAPES)
def test_dmmv_matches_oracle(fmt, rows, cols, layout):
    w = synth.weight_blocks(fmt, rows, cols, seed=rows + cols)
    x = synth.activations(cols, seed=rows)
    xq_ref = oracle.quantize_q8_0(x)
    xq = Z.quantize_act_q8_0(dev(x))
    y = nan_out(rows)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    Z.dmmv(fmt, wd, rows, cols, xq, y=y, layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    y_ref, e_ref = oracle.dmmv(fmt, w, rows, cols, xq_ref)
    check_y(y, y_ref, e_ref)


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 300, 2048), (Q4_0, 300, 4096), (Q8_0, 70, 512),
                                           (Q4_0, 41, 96), (Q8_0, 9, 14336)])
def test_block_sums_bit_exact(fmt, rows, cols, layout):
    w = synth.weight_blocks(fmt, rows, cols, seed=5 * rows)
    xq = synth.activation_blocks(cols // 32, seed=6 * rows)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    s = Z.debug_block_sums(fmt, wd, rows, cols, dev(xq), layout=layout)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), oracle.block_sums(fmt, w, rows, cols, xq))


@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 500, 4096), (Q4_0, 700, 2048), (Q8_0, 90, 512),
                                           (Q4_0, 3, 8192), (Q8_0, 10, 96)])
def test_exact_integer_outputs_equal_oracle_bitwise(fmt, rows, cols):
    """Unit scales and small codes keep every fp32 partial sum an exact integer,
    so the kernel's y must equal the oracle's exactly: this pins the hot kernel's
    integer block sums end to end."""
    w = synth.weight_blocks_small(fmt, rows, cols, seed=rows, qmax=7)
    xq = synth.activation_blocks(cols // 32, seed=cols, qmax=15, fixed_scale=1.0)
    for layout in (Z.GGUF, Z.REPACKED):
        y = run_dmmv(fmt, w, rows, cols, xq, layout=layout)
        y_ref, _ = oracle.dmmv(fmt, w, rows, cols, xq)
        assert np.array_equal(y.double().cpu().numpy(), y_ref)


@pytest.mark.parametrize("fmt,cols", [(Q8_0, 2048), (Q4_0, 4096), (Q8_0, 160)])
def test_row_permutation_equivariance_bitwise(fmt, cols):
    rows = 611
    w = synth.weight_blocks(fmt, rows, cols, seed=77)
    xq = synth.activation_blocks(cols // 32, seed=78)
    perm = np.random.default_rng(1).permutation(rows)
    wp = w.reshape(rows, -1)[perm].reshape(-1)
    y = run_dmmv(fmt, w, rows, cols, xq).cpu().numpy()
    yp = run_dmmv(fmt, wp, rows, cols, xq).cpu().numpy()
    assert np.array_equal(yp, y[perm])


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
def test_power_of_two_input_scaling_exact(fmt):
    rows, cols, k = 999, 2048, 3
    w = synth.weight_blocks(fmt, rows, cols, seed=88)
    x = synth.activations(cols, seed=89)
    xs = (x * np.float32(2.0 ** k)).astype(np.float32)
    wd = dev(w)
    y1 = nan_out(rows)
    y2 = nan_out(rows)
    Z.dmmv(fmt, wd, rows, cols, Z.quantize_act_q8_0(dev(x)), y=y1)
    Z.dmmv(fmt, wd, rows, cols, Z.quantize_act_q8_0(dev(xs)), y=y2)
    torch.cuda.synchronize()
    assert torch.equal(y2, y1 * 2.0 ** k)


def test_layouts_agree_bitwise():
    for fmt, rows, cols in [(Q8_0, 333, 4096), (Q4_0, 333, 2048), (Q4_0, 40, 96)]:
        w = synth.weight_blocks(fmt, rows, cols, seed=3)
        xq = synth.activation_blocks(cols // 32, seed=4)
        a = run_dmmv(fmt, w, rows, cols, xq, layout=Z.GGUF)
        b = run_dmmv(fmt, w, rows, cols, xq, layout=Z.REPACKED)
        assert torch.equal(a, b)


def test_zero_rows_is_a_no_op():
    y = nan_out(4)
    Z.q8_0(torch.empty(16, dtype=torch.uint8, device="cuda"), 0, 64,
           torch.empty(80, dtype=torch.uint8, device="cuda"), y=y)
    torch.cuda.synchronize()
    assert torch.isnan(y).all()


# ----------------------------------------------------------------- repack
@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 123, 4096), (Q4_0, 1000, 2048), (Q4_0, 7, 96)])
def test_repack_bit_exact(fmt, rows, cols):
    w = synth.weight_blocks(fmt, rows, cols, seed=rows)
    r = Z.repack(fmt, dev(w), rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(r.cpu().numpy(), oracle.repack(fmt, w, rows, cols))


# ----------------------------------------------------------------- batched
@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 1434, 4096), (Q4_0, 901, 2048), (Q8_0, 99, 160),
                                           (Q4_0, 300, 8192), (Q8_0, 257, 3072), (Q8_0, 77, 512),
                                           (Q4_0, 411, 2304)])
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 7, 8])
def test_batched_matches_oracle_and_single_calls(fmt, rows, cols, batch, layout):
    w = synth.weight_blocks(fmt, rows, cols, seed=batch)
    x = synth.activations(cols, seed=10 + batch, batch=batch)
    xq = Z.quantize_act_q8_0(dev(x))
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    y = nan_out(batch, rows)
    Z.dmmv_batched(fmt, wd, rows, cols, xq, batch, y=y, layout=layout)
    torch.cuda.synchronize()
    xq_ref = oracle.quantize_q8_0(x)
    y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, xq_ref, batch)
    check_y(y, y_ref, e_ref)
    # deterministic: the same call again gives the same bits
    y2 = nan_out(batch, rows)
    Z.dmmv_batched(fmt, wd, rows, cols, xq, batch, y=y2, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    if batch == 1 or _vector_split_shape(cols, batch):
        # batch 1, and every batch the vector-split kernel takes, is the
        # single-vector computation per vector, bit for bit
        nbx = cols // 32 * 34
        for v in range(batch):
            ys = nan_out(rows)
            Z.dmmv(fmt, wd, rows, cols, xq[v * nbx:(v + 1) * nbx].clone(), y=ys, layout=layout)
            torch.cuda.synchronize()
            assert torch.equal(ys, y[v]), f"vector {v} differs from its single-vector call"


@pytest.mark.parametrize("fmt", [Q8_0, Q4_0])
@pytest.mark.parametrize("cols", [256, 512])
@pytest.mark.parametrize("batch", [2, 8])
def test_batched_extreme_codes_exact(fmt, cols, batch):
    """Only the formats' extreme codes (Q8_0 -128 / 127, Q4_0 0 / 15 against
    activation codes -128 / 127), unit scales, at most 16 blocks a row: every
    output is an exact integer below 2^24, so the batched kernel's block sums
    must give the oracle's values bit for bit."""
    rows = 77
    w = synth.extreme_code_blocks(fmt, rows * cols // 32, seed=cols + batch, stream=synth.S_WEIGHT)
    xq = synth.extreme_code_blocks(Q8_0, batch * cols // 32, seed=cols * batch)
    y = nan_out(batch, rows)
    Z.dmmv_batched(fmt, dev(w), rows, cols, dev(xq), batch, y=y)
    torch.cuda.synchronize()
    y_ref, _ = oracle.dmmv_batched(fmt, w, rows, cols, xq, batch)
    assert np.array_equal(y.double().cpu().numpy(), y_ref)


def _vector_split_shape(cols, batch):
    """Widths and batches the vector-split batched kernel takes: pipelined widths
    (multiples of 256 up to 8192), two vectors per warp up to 4096 columns, one
    vector per warp (batch <= 4) beyond."""
    if batch < 2 or cols % 256 or cols > 8192:
        return False
    return cols <= 4096 or batch <= 4


@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 333, 4096), (Q4_0, 517, 2048), (Q8_0, 130, 1024),
                                           (Q4_0, 41, 8192), (Q8_0, 65, 3072), (Q4_0, 23, 96)])
@pytest.mark.parametrize("batch", [2, 3, 5, 8])
def test_batched_exact_integer_outputs_equal_oracle_bitwise(fmt, rows, cols, batch):
    """Unit scales and small codes: every fp32 partial sum is an exact integer,
    so each batched output equals the oracle's exactly (pins the batched
    kernel's integer block sums)."""
    w = synth.weight_blocks_small(fmt, rows, cols, seed=rows + batch, qmax=7)
    xq = synth.activation_blocks(batch * cols // 32, seed=cols + batch, qmax=15, fixed_scale=1.0)
    for layout in (Z.GGUF, Z.REPACKED):
        wd = dev(w)
        if layout == Z.REPACKED:
            wd = Z.repack(fmt, wd, rows, cols)
        y = nan_out(batch, rows)
        Z.dmmv_batched(fmt, wd, rows, cols, dev(xq), batch, y=y, layout=layout)
        torch.cuda.synchronize()
        y_ref, _ = oracle.dmmv_batched(fmt, w, rows, cols, xq, batch)
        assert np.array_equal(y.double().cpu().numpy(), y_ref)


# ------------------------------------------------------------ expert gather
def _moe_stack(fmt, rows, cols, n_slots, seed):
    return synth.weight_blocks(fmt, n_slots * rows, cols, seed=seed)


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
def test_expert_gather_small_stack(layout):
    rows, cols, n_exp = 96, 512, 12
    per = rows * cols // 32 * 18
    stack = _moe_stack(Q4_0, rows, cols, n_exp, seed=5)
    idx = np.array([11, 0, 7, 7, 3], dtype=np.int32)
    x = synth.activations(cols, seed=6, batch=len(idx))
    xq_ref = oracle.quantize_q8_0(x)
    sd = dev(stack)
    if layout == Z.REPACKED:
        sd = torch.cat([Z.repack(Q4_0, sd[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
    y = nan_out(len(idx), rows)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.expert_gather(Q4_0, sd, per, rows, cols, dev(idx), n_exp, dev(xq_ref), cols // 32 * 34, y=y,
                    status=st, layout=layout)
    torch.cuda.synchronize()
    y_ref, e_ref, st_ref = oracle.expert_gather(Q4_0, stack, per, rows, cols, idx, n_exp, xq_ref,
                                                cols // 32 * 34)
    assert st.item() == 0 == st_ref
    check_y(y, y_ref, e_ref)
    for k, e in enumerate(idx):
        ys = run_dmmv(Q4_0, None, rows, cols, xq_ref.reshape(len(idx), -1)[k], layout=layout,
                      w_dev=sd[e * per:(e + 1) * per])
        assert torch.equal(ys, y[k])


@pytest.mark.parametrize("cols", [512, 96])
def test_expert_gather_bad_index_gives_nan_and_status(cols):
    rows, n_exp = 40, 4
    per = rows * cols // 32 * 34
    stack = _moe_stack(Q8_0, rows, cols, n_exp, seed=8)
    xq = synth.activation_blocks(cols // 32, seed=9)
    idx = np.array([2, 4, -1, 0], dtype=np.int32)
    y = torch.zeros(len(idx), rows, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.expert_gather(Q8_0, dev(stack), per, rows, cols, dev(idx), n_exp, dev(xq), 0, y=y, status=st)
    torch.cuda.synchronize()
    y_ref, e_ref, st_ref = oracle.expert_gather(Q8_0, stack, per, rows, cols, idx, n_exp, xq, 0)
    assert st.item() == 1 == st_ref
    yh = y.cpu().numpy()
    assert np.isnan(yh[1]).all() and np.isnan(yh[2]).all()
    good = [0, 3]
    ok, _ = oracle.within_tolerance(yh[good], y_ref[good], e_ref[good])
    assert ok


# ------------------------------------------------------- end-to-end host step
@pytest.mark.parametrize("fmt,rows,cols,batch", [(Q4_0, 4096, 4096, 1), (Q8_0, 1000, 4096, 4),
                                                 (Q8_0, 33, 96, 2)])
def test_host_step_matches_oracle(fmt, rows, cols, batch):
    w = synth.weight_blocks(fmt, rows, cols, seed=21)
    x = synth.activations(cols, seed=22, batch=batch)
    xh = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    yh = torch.full((batch, rows), float("nan"), dtype=torch.float32).pin_memory()
    ws = torch.empty(Z.host_step_workspace_bytes(rows, cols, batch), dtype=torch.uint8, device="cuda")
    Z.host_step(fmt, dev(w), rows, cols, xh, yh, ws, batch=batch)
    torch.cuda.synchronize()
    xq_ref = oracle.quantize_q8_0(x)
    y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, xq_ref, batch)
    check_y(yh, y_ref, e_ref)


@pytest.mark.parametrize("fmt,rows,cols,batch", [(Q4_0, 4096, 4096, 1), (Q8_0, 1000, 4096, 4),
                                                 (Q8_0, 33, 96, 2), (Q4_0, 777, 2048, 8)])
def test_host_step_mapped_and_copied_buffers_agree_bitwise(fmt, rows, cols, batch):
    """Page-locked host buffers are read and written by the kernels in place;
    pageable ones are copied through the workspace; an interior slice of a larger
    page-locked buffer is in place too. All give the same bits."""
    w = dev(synth.weight_blocks(fmt, rows, cols, seed=31))
    x = np.ascontiguousarray(synth.activations(cols, seed=32, batch=batch)).reshape(batch, cols)
    ws = torch.empty(Z.host_step_workspace_bytes(rows, cols, batch), dtype=torch.uint8, device="cuda")
    outs = []
    for pinned, interior in ((True, False), (False, False), (True, True), (False, True)):
        if interior:
            big_x = torch.zeros(batch * cols + 64, dtype=torch.float32)
            big_y = torch.full((batch * rows + 96,), float("nan"), dtype=torch.float32)
            if pinned:
                big_x, big_y = big_x.pin_memory(), big_y.pin_memory()
            xh = big_x[16:16 + batch * cols].view(batch, cols)
            yh = big_y[32:32 + batch * rows].view(batch, rows)
            xh.copy_(torch.from_numpy(x))
        else:
            xh = torch.from_numpy(x.copy())
            yh = torch.full((batch, rows), float("nan"), dtype=torch.float32)
            if pinned:
                xh, yh = xh.pin_memory(), yh.pin_memory()
        Z.host_step(fmt, w, rows, cols, xh, yh, ws, batch=batch)
        torch.cuda.synchronize()
        if interior:
            # the bytes around the slice are untouched
            assert torch.isnan(big_y[:32]).all() and torch.isnan(big_y[32 + batch * rows:]).all()
        outs.append(yh.clone())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    y_ref, e_ref = oracle.dmmv_batched(fmt, synth.weight_blocks(fmt, rows, cols, seed=31), rows, cols,
                                       oracle.quantize_q8_0(x if batch > 1 else x[0]), batch)
    check_y(outs[0], y_ref, e_ref)


# ------------------------------------------------------- fused fp32 activation
@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols,batch", [(Q4_0, 4096, 4096, 1), (Q8_0, 1531, 2048, 1),
                                                 (Q8_0, 700, 512, 3), (Q4_0, 99, 8192, 8),
                                                 (Q8_0, 37, 96, 1), (Q4_0, 77, 160, 5), (Q8_0, 5, 14336, 2),
                                                 (Q8_0, 1434, 4096, 8), (Q4_0, 901, 2048, 4), (Q8_0, 333, 4096, 2),
                                                 (Q4_0, 300, 8192, 3), (Q8_0, 517, 2048, 7), (Q4_0, 1000, 4096, 5)])
def test_fused_f32_equals_quantize_then_dmmv_bitwise(fmt, rows, cols, batch, layout):
    w = synth.weight_blocks(fmt, rows, cols, seed=cols + batch)
    x = synth.activations(cols, seed=rows, batch=batch)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    xd = dev(x)
    yf = nan_out(batch, rows)
    Z.dmmv_f32(fmt, wd, rows, cols, xd, batch=batch, y=yf, layout=layout)
    xq = Z.quantize_act_q8_0(xd)
    nbx = cols // 32 * 34
    yu = nan_out(batch, rows)
    for v in range(batch):
        # each vector through the two-kernel path (a 16-byte aligned copy of its blocks)
        Z.dmmv(fmt, wd, rows, cols, xq[v * nbx:(v + 1) * nbx].clone(), y=yu[v], layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(yf, yu), "fused and two-kernel results differ"
    y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, oracle.quantize_q8_0(x), batch)
    check_y(yf, y_ref, e_ref)


def test_fused_f32_chain_with_reused_buffers():
    """A decode chain whose layers reuse ping-pong activation/output buffers:
    each layer's input is the previous layer's output (dependent launches)."""
    rows = cols = 2048
    fmt = Q4_0
    ws = [synth.weight_blocks(fmt, rows, cols, seed=300 + i) for i in range(6)]
    x = synth.activations(cols, seed=301)
    bufs = [dev(x), nan_out(rows)]
    wds = [dev(w) for w in ws]
    for i, wd in enumerate(wds):
        Z.dmmv_f32(fmt, wd, rows, cols, bufs[i % 2], y=bufs[(i + 1) % 2])
    torch.cuda.synchronize()
    got = bufs[len(wds) % 2].cpu().numpy()
    # the same chain through the oracle (each layer's fp32 output rounded to fp32 as the kernel stores it)
    cur = x
    for i, w in enumerate(ws):
        y_ref, e_ref = oracle.dmmv(fmt, w, rows, cols, oracle.quantize_q8_0(cur))
        if i == len(ws) - 1:
            ok, worst = oracle.within_tolerance(got, y_ref, e_ref)
            assert ok, worst
        else:
            # the next layer consumes the kernel's own output (fp32); take it from a second run
            yk = nan_out(rows)
            Z.dmmv_f32(fmt, wds[i], rows, cols, dev(cur), y=yk)
            torch.cuda.synchronize()
            yk = yk.cpu().numpy()
            ok, worst = oracle.within_tolerance(yk, y_ref, e_ref)
            assert ok, worst
            cur = yk


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q4_0, 512, 2048), (Q8_0, 300, 512), (Q4_0, 40, 96)])
def test_expert_gather2_equals_two_gathers_bitwise(fmt, rows, cols, layout):
    n_exp = 6
    bb = 18 if fmt == Q4_0 else 34
    per = rows * cols // 32 * bb
    sa = synth.weight_blocks(fmt, n_exp * rows, cols, seed=41)
    sb = synth.weight_blocks(fmt, n_exp * rows, cols, seed=42, stream=synth.S_WEIGHT2)
    idx = np.array([5, 1, 3, 3, 0, 7], dtype=np.int32)   # 7 is out of range
    xq = synth.activation_blocks(cols // 32, seed=43)
    da, db = dev(sa), dev(sb)
    if layout == Z.REPACKED:
        da = torch.cat([Z.repack(fmt, da[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
        db = torch.cat([Z.repack(fmt, db[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
    ia = dev(idx)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ya, yb = Z.expert_gather2(fmt, da, db, per, rows, cols, ia, n_exp, dev(xq), 0, status=st2, layout=layout)
    ref_a = nan_out(len(idx), rows)
    ref_b = nan_out(len(idx), rows)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.expert_gather(fmt, da, per, rows, cols, ia, n_exp, dev(xq), 0, y=ref_a, status=st, layout=layout)
    Z.expert_gather(fmt, db, per, rows, cols, ia, n_exp, dev(xq), 0, y=ref_b, status=st, layout=layout)
    torch.cuda.synchronize()
    assert st2.item() == 1 and st.item() == 1
    assert torch.equal(ya[:5], ref_a[:5]) and torch.equal(yb[:5], ref_b[:5])
    assert torch.isnan(ya[5]).all() and torch.isnan(yb[5]).all()
    y_ref, e_ref, _ = oracle.expert_gather(fmt, sb, per, rows, cols, idx, n_exp, xq, 0)
    check_y(yb[:5], y_ref[:5], e_ref[:5])


# ------------------------------------------------------------ argmax epilogue
def _argmax_case(fmt, rows, cols, layout, seed):
    w = synth.weight_blocks(fmt, rows, cols, seed=seed)
    xq = synth.activation_blocks(cols // 32, seed=seed + 1)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    return w, xq, wd


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q4_0, 248320 // 8, 2048), (Q8_0, 5000, 4096), (Q4_0, 1, 256),
                                           (Q8_0, 77, 512), (Q4_0, 3001, 8192)])
def test_argmax_matches_own_logits_and_oracle(fmt, rows, cols, layout):
    w, xq, wd = _argmax_case(fmt, rows, cols, layout, seed=rows)
    xqd = dev(xq)
    y = nan_out(rows)
    Z.dmmv(fmt, wd, rows, cols, xqd, y=y, layout=layout)
    mx = torch.full((1,), float("nan"), device="cuda")
    idx = Z.dmmv_argmax(fmt, wd, rows, cols, xqd, max_out=mx, layout=layout)
    torch.cuda.synchronize()
    yh = y.cpu().numpy()
    i = int(idx.item())
    # the same fp32 logits: the first index of their maximum, and that value
    assert i == int(np.argmax(yh)) and mx.item() == yh[i]
    # against the oracle: the pick is a valid argmax within the tolerance
    y_ref, e_ref = oracle.dmmv(fmt, w, rows, cols, xq)
    j, _ = oracle.argmax(y_ref)
    tol = REL * (e_ref[i] + e_ref[j]) + 2 * ABS
    assert y_ref[i] >= y_ref[j] - tol


def test_argmax_ties_pick_the_first_row():
    fmt, rows, cols = Q4_0, 4000, 2048
    w, xq, wd = _argmax_case(fmt, rows, cols, Z.GGUF, seed=9)
    xqd = dev(xq)
    y = Z.dmmv(fmt, wd, rows, cols, xqd)
    torch.cuda.synchronize()
    r = int(torch.argmax(y).item())
    rb = cols // 32 * 18
    w2 = w.reshape(rows, rb).copy()
    for p in (3, 1777, 3999):             # identical copies of the maximal row, before and after it
        w2[p] = w2[r]
    first = min(3, r)
    idx = Z.dmmv_argmax(fmt, dev(w2.reshape(-1)), rows, cols, xqd)
    torch.cuda.synchronize()
    assert int(idx.item()) == first


def test_argmax_workspace_is_reusable_back_to_back():
    fmt, rows, cols = Q8_0, 2048, 4096
    outs = []
    ws = torch.empty(Z.ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    for seed in (1, 2, 3):
        w, xq, wd = _argmax_case(fmt, rows, cols, Z.GGUF, seed=seed)
        outs.append((Z.dmmv_argmax(fmt, wd, rows, cols, dev(xq), workspace=ws), wd, dev(xq)))
    torch.cuda.synchronize()
    for idx, wd, xqd in outs:
        y = Z.dmmv(fmt, wd, rows, cols, xqd)
        torch.cuda.synchronize()
        assert int(idx.item()) == int(torch.argmax(y).item())


# ------------------------------------------------------- accumulate epilogue
@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 2048, 512), (Q4_0, 1000, 4096), (Q8_0, 57, 96)])
@pytest.mark.parametrize("gate", [None, 0.0, -1.3, 2.7])
def test_accumulate_epilogue_matches_oracle(fmt, rows, cols, layout, gate):
    w = synth.weight_blocks(fmt, rows, cols, seed=rows + 3)
    xq = synth.activation_blocks(cols // 32, seed=cols + 3)
    y0 = synth.activations(rows, seed=5, scale=0.05)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    y = dev(y0.copy())
    g = None if gate is None else torch.tensor([gate], dtype=torch.float32, device="cuda")
    Z.dmmv_acc(fmt, wd, rows, cols, dev(xq), y, gate=g, layout=layout)
    torch.cuda.synchronize()
    y_ref, e_ref = oracle.dmmv_acc(fmt, w, rows, cols, xq, y0.astype(np.float64), gate=gate)
    d_ref, _ = oracle.dmmv(fmt, w, rows, cols, xq)
    yh = y.double().cpu().numpy()
    # DMMV bound scaled by the gate, the fp32 sigmoid (a few ulp) times |W.x|, the final rounding
    bound = REL * e_ref + ABS + 4 * 2.0 ** -24 * np.abs(d_ref) + 2.0 ** -24 * np.abs(y_ref)
    assert np.all(np.abs(yh - y_ref) <= bound), float(np.max(np.abs(yh - y_ref) / bound))


def test_accumulate_without_gate_into_zero_equals_store_bitwise():
    for fmt, rows, cols in [(Q4_0, 4096, 4096), (Q8_0, 77, 160)]:
        w = synth.weight_blocks(fmt, rows, cols, seed=17)
        xq = dev(synth.activation_blocks(cols // 32, seed=18))
        wd = dev(w)
        y = torch.zeros(rows, device="cuda")
        Z.dmmv_acc(fmt, wd, rows, cols, xq, y)
        ys = Z.dmmv(fmt, wd, rows, cols, xq)
        torch.cuda.synchronize()
        assert torch.equal(y, ys)


# ---------------------------------------------------------- SwiGLU epilogue
def _stacks(fmt, rows, cols, n_exp, layout, seed):
    bb = 18 if fmt == Q4_0 else 34
    per = rows * cols // 32 * bb
    sg = synth.weight_blocks(fmt, n_exp * rows, cols, seed=seed)
    su = synth.weight_blocks(fmt, n_exp * rows, cols, seed=seed + 1, stream=synth.S_WEIGHT2)
    dg, du = dev(sg), dev(su)
    if layout == Z.REPACKED:
        dg = torch.cat([Z.repack(fmt, dg[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
        du = torch.cat([Z.repack(fmt, du[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
    return per, sg, su, dg, du


def _swiglu_bound(g_ref, u_ref, e_g, e_u, h_ref):
    """|h - h_ref| bound from the DMMV tolerances of g and u (|silu'| <= 1.1)
    plus the fp32 epilogue (exp, divide, multiply: a few ulp of h)."""
    tg, tu = REL * e_g + ABS, REL * e_u + ABS
    silu = g_ref / (1.0 + np.exp(-g_ref))
    return 1.1 * tg * np.abs(u_ref) + np.abs(silu) * tu + 1.1 * tg * tu + 16 * 2.0 ** -24 * np.abs(h_ref) + 1e-12


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q4_0, 512, 2048), (Q8_0, 300, 512), (Q4_0, 37, 256),
                                           (Q8_0, 1000, 4096)])
def test_swiglu_epilogue_matches_gather2_and_oracle(fmt, rows, cols, layout):
    n_exp = 6
    per, sg, su, dg, du = _stacks(fmt, rows, cols, n_exp, layout, seed=51)
    idx = np.array([5, 1, 3, 3, 0, 7, 2], dtype=np.int32)   # 7 is out of range
    xs = np.concatenate([synth.activation_blocks(cols // 32, seed=60 + k) for k in range(len(idx))])
    xstride = cols // 32 * 34
    ia, xd = dev(idx), dev(xs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = nan_out(len(idx), rows)
    Z.expert_swiglu(fmt, dg, du, rows, cols, xd, idx=ia, expert_stride=per, n_experts=n_exp,
                    xq_stride=xstride, h=h, status=st, layout=layout)
    ga, ua = Z.expert_gather2(fmt, dg, du, per, rows, cols, ia, n_exp, xd, xstride, layout=layout)
    torch.cuda.synchronize()
    assert st.item() == 1
    good = [k for k in range(len(idx)) if idx[k] < n_exp]
    assert torch.isnan(h[5]).all()
    hh = h[good].double().cpu().numpy()
    # against the kernel's own fp32 gate and up values: the epilogue alone
    g32 = ga[good].double().cpu().numpy()
    u32 = ua[good].double().cpu().numpy()
    h64 = g32 / (1.0 + np.exp(-g32)) * u32
    assert np.all(np.abs(hh - h64) <= 16 * 2.0 ** -24 * np.abs(h64) + 1e-30)
    # against the oracle: gate and up in fp64, then swiglu
    g_ref, e_g, _ = oracle.expert_gather(fmt, sg, per, rows, cols, idx, n_exp, xs, xstride)
    u_ref, e_u, _ = oracle.expert_gather(fmt, su, per, rows, cols, idx, n_exp, xs, xstride)
    g_ref, e_g, u_ref, e_u = g_ref[good], e_g[good], u_ref[good], e_u[good]
    h_ref = oracle.swiglu(g_ref.ravel(), u_ref.ravel()).reshape(g_ref.shape)
    bound = _swiglu_bound(g_ref, u_ref, e_g, e_u, h_ref)
    assert np.all(np.abs(hh - h_ref) <= bound), float(np.max(np.abs(hh - h_ref) / bound))


@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 2048, 2048), (Q4_0, 4096, 4096)])
def test_swiglu_dense_pair_without_index(fmt, rows, cols):
    _, sg, su, dg, du = _stacks(fmt, rows, cols, 1, Z.GGUF, seed=70)
    xq = synth.activation_blocks(cols // 32, seed=72)
    xd = dev(xq)
    h = nan_out(1, rows)
    Z.expert_swiglu(fmt, dg, du, rows, cols, xd, h=h)
    g = Z.dmmv(fmt, dg, rows, cols, xd)
    u = Z.dmmv(fmt, du, rows, cols, xd)
    torch.cuda.synchronize()
    hh = h[0].double().cpu().numpy()
    g32, u32 = g.double().cpu().numpy(), u.double().cpu().numpy()
    h64 = g32 / (1.0 + np.exp(-g32)) * u32
    assert np.all(np.abs(hh - h64) <= 16 * 2.0 ** -24 * np.abs(h64) + 1e-30)
    g_ref, e_g = oracle.dmmv(fmt, sg, rows, cols, xq)
    u_ref, e_u = oracle.dmmv(fmt, su, rows, cols, xq)
    h_ref = oracle.swiglu(g_ref, u_ref)
    assert np.all(np.abs(hh - h_ref) <= _swiglu_bound(g_ref, u_ref, e_g, e_u, h_ref))


# ------------------------------------------------ fp32 (unquantized) activation
@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols,batch", [
    (Q4_0, 1000, 2048, 1), (Q8_0, 777, 4096, 1), (Q4_0, 300, 8192, 2), (Q8_0, 129, 8192, 1),
    (Q8_0, 200, 768, 3), (Q4_0, 64, 512, 1), (Q8_0, 33, 256, 8),      # 8 and 16 lanes per row
    (Q4_0, 45, 96, 2), (Q8_0, 20, 160, 1), (Q4_0, 7, 8224, 1),        # plain kernel widths
])
def test_xf32_matches_oracle(fmt, rows, cols, batch, layout):
    w = synth.weight_blocks(fmt, rows, cols, seed=rows + 11)
    x = synth.activations(cols, seed=cols + 12, batch=batch)
    wd = dev(w)
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    xd = dev(x)
    y = nan_out(batch, rows)
    Z.dmmv_xf32(fmt, wd, rows, cols, xd, batch=batch, y=y, layout=layout)
    y2 = nan_out(batch, rows)
    Z.dmmv_xf32(fmt, wd, rows, cols, xd, batch=batch, y=y2, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "two calls differ"
    xs = np.asarray(x, dtype=np.float32).reshape(batch, cols)
    for v in range(batch):
        y_ref, e_ref = oracle.dmmv_xf32(fmt, w, rows, cols, xs[v])
        check_y(y[v], y_ref, e_ref)


def test_xf32_ragged_tiles_and_zero_rows():
    fmt, cols = Q4_0, 2048
    for rows in (1, 17, 4097):
        w = synth.weight_blocks(fmt, rows, cols, seed=rows)
        x = synth.activations(cols, seed=5)
        y = nan_out(rows)
        Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), y=y)
        torch.cuda.synchronize()
        y_ref, e_ref = oracle.dmmv_xf32(fmt, w, rows, cols, x)
        check_y(y, y_ref, e_ref)
    # rows == 0 launches nothing and succeeds
    Z.dmmv_xf32(fmt, dev(synth.weight_blocks(fmt, 1, cols, seed=1)), 0, cols, dev(x), y=nan_out(1))


def _xf32_tall_rows(extra=0):
    """Rows enough for the fp32-activation tensor-core kernel (it takes matrices
    of at least 4 groups of 128 rows per SM), plus a ragged tail."""
    return 4 * 128 * torch.cuda.get_device_properties(0).multi_processor_count + extra


@pytest.mark.parametrize("fmt,cols,extra", [(Q4_0, 2048, 37), (Q8_0, 512, 0), (Q4_0, 8192, 129), (Q8_0, 768, 5)])
def test_xf32_tall_matches_oracle(fmt, cols, extra):
    """The tensor-core path of the fp32-activation DMMV (tall GGUF matrices):
    every row within the tolerance of the oracle, a partial last row group
    included, and two calls give the same bits."""
    rows = _xf32_tall_rows(extra)
    w = synth.weight_blocks(fmt, rows, cols, seed=cols + extra)
    x = synth.activations(cols, seed=cols + 1)
    y = nan_out(rows)
    Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), y=y)
    y2 = nan_out(rows)
    Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), y=y2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "two calls differ"
    y_ref, e_ref = oracle.dmmv_xf32(fmt, w, rows, cols, x)
    check_y(y, y_ref, e_ref)


def test_xf32_tall_batched_slots():
    fmt, cols, batch = Q4_0, 512, 3
    rows = _xf32_tall_rows(64)
    w = synth.weight_blocks(fmt, rows, cols, seed=9)
    x = synth.activations(cols, seed=10, batch=batch)
    y = nan_out(batch, rows)
    Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), batch=batch, y=y)
    torch.cuda.synchronize()
    for v in range(batch):
        y_ref, e_ref = oracle.dmmv_xf32(fmt, w, rows, cols, np.asarray(x, dtype=np.float32)[v])
        check_y(y[v], y_ref, e_ref)


@pytest.mark.parametrize("fmt,cols", [(Q4_0, 2048), (Q8_0, 1024)])
def test_xf32_wide_dynamic_range(fmt, cols):
    """The tensor-core kernel splits each activation block, scaled by a power of
    two, into three fp16 parts: blocks whose magnitudes span 1e-30 .. 1e30, a
    1e12 range inside one block, all-zero blocks, signed zeros and blocks near
    the fp32 normal limit still meet the tolerance."""
    rows = _xf32_tall_rows()
    w = synth.weight_blocks(fmt, rows, cols, seed=cols + 3)
    g = np.random.Generator(np.random.PCG64(77))
    nb = cols // 32
    x = g.standard_normal(cols).astype(np.float64)
    block_scale = 10.0 ** g.uniform(-30, 30, size=nb)
    x *= np.repeat(block_scale, 32)
    x[5 * 32:6 * 32] = 0.0                                   # an all-zero block
    x[6 * 32:7 * 32] = -0.0
    x[7 * 32:8 * 32] *= 10.0 ** g.uniform(-12, 0, size=32)   # 1e12 range inside a block
    x[8 * 32:9 * 32] = g.standard_normal(32) * 1e-36         # near the fp32 normal limit
    x[9 * 32] = 3.0e30                                       # one huge element, the rest tiny
    x[9 * 32 + 1:10 * 32] = 1e-20
    x = x.astype(np.float32)
    y = nan_out(rows)
    Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), y=y)
    torch.cuda.synchronize()
    y_ref, e_ref = oracle.dmmv_xf32(fmt, w, rows, cols, x)
    check_y(y, y_ref, e_ref)


def test_xf32_exact_on_representable_activations():
    """Unit weight scales and activations that are small integers times 2^-4:
    every product and partial sum is an exact fp32 value, so the tensor-core
    kernel's result equals the oracle's exactly."""
    for fmt in (Q4_0, Q8_0):
        rows, cols = _xf32_tall_rows(3), 512
        w = synth.weight_blocks_small(fmt, rows, cols, seed=fmt, qmax=7)
        g = np.random.Generator(np.random.PCG64(fmt + 1))
        x = (g.integers(-15, 16, size=cols) / 16.0).astype(np.float32)
        y = nan_out(rows)
        Z.dmmv_xf32(fmt, dev(w), rows, cols, dev(x), y=y)
        torch.cuda.synchronize()
        y_ref, _ = oracle.dmmv_xf32(fmt, w, rows, cols, x)
        assert np.array_equal(y.double().cpu().numpy(), y_ref), fmt


# ------------------------------------------------- one-launch expert FFN
def _ffn_case(fmt_gu, fmt_dn, hidden, ffn, n_exp, idx, seed):
    bgu = 18 if fmt_gu == Q4_0 else 34
    bdn = 18 if fmt_dn == Q4_0 else 34
    gu_per = ffn * hidden // 32 * bgu
    dn_per = hidden * ffn // 32 * bdn
    g = synth.weight_blocks(fmt_gu, n_exp * ffn, hidden, seed=seed)
    u = synth.weight_blocks(fmt_gu, n_exp * ffn, hidden, seed=seed, stream=synth.S_WEIGHT2)
    d = synth.weight_blocks(fmt_dn, n_exp * hidden, ffn, seed=seed, stream=synth.S_WEIGHT3)
    x = synth.activations(hidden, seed=seed + 1)
    return dict(g=g, u=u, d=d, x=x, gu_per=gu_per, dn_per=dn_per, idx=np.asarray(idx, dtype=np.int32))


@pytest.mark.parametrize("fmt_gu,fmt_dn,hidden,ffn", [(Q4_0, Q8_0, 2048, 512), (Q8_0, Q8_0, 4096, 1024),
                                                      (Q4_0, Q4_0, 1024, 256), (Q8_0, Q4_0, 2560, 2048)])
def test_expert_ffn_equals_swiglu_then_down_gather(fmt_gu, fmt_dn, hidden, ffn):
    n_exp = 6
    c = _ffn_case(fmt_gu, fmt_dn, hidden, ffn, n_exp, [5, 0, 3, 3, 2, 1, 4], seed=hidden + ffn)
    gd, ud, dd, ia = dev(c["g"]), dev(c["u"]), dev(c["d"]), dev(c["idx"])
    xq = Z.quantize_act_q8_0(dev(c["x"]))
    n = len(c["idx"])
    ws = Z.expert_ffn_workspace(n, ffn)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):  # the counters are reset by every call: repeated calls agree
        y, h = Z.expert_ffn(fmt_gu, gd, ud, c["gu_per"], fmt_dn, dd, c["dn_per"], hidden, ffn, ia, n_exp, xq,
                            y=nan_out(n, hidden), workspace=ws, status=st)
        torch.cuda.synchronize()
        outs.append((y.clone(), h.clone()))
    assert st.item() == 0
    for y, h in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(h, outs[0][1])
    y, h = outs[0]
    # the same results through the separate entry points, bit for bit
    h2 = Z.expert_swiglu(fmt_gu, gd, ud, ffn, hidden, xq, idx=ia, expert_stride=c["gu_per"], n_experts=n_exp)
    hq = Z.quantize_act_q8_0(h2.reshape(-1))
    y2 = Z.expert_gather(fmt_dn, dd, c["dn_per"], hidden, ffn, ia, n_exp, hq, ffn // 32 * 34)
    torch.cuda.synchronize()
    assert torch.equal(h, h2)
    assert torch.equal(y, y2)
    # against the oracle: the down DMMV of the kernel's own h, quantized by the oracle
    hh = h.cpu().numpy()
    hq_ref = oracle.quantize_q8_0(hh.reshape(-1))
    assert np.array_equal(hq.cpu().numpy(), hq_ref)
    y_ref, e_ref, s = oracle.expert_gather(fmt_dn, c["d"], c["dn_per"], hidden, ffn, c["idx"], n_exp, hq_ref,
                                           ffn // 32 * 34)
    assert s == 0
    check_y(y, y_ref, e_ref)


@pytest.mark.parametrize("n", [1, 40])
def test_expert_ffn_selection_sizes(n):
    """One selected expert (the whole grid on one expert's rows) and 40 (few CTAs
    per expert, the gate/up share of the grid rounded down to a handful): h and y
    equal the separate entry points bit for bit."""
    fmt_gu, fmt_dn, hidden, ffn, n_exp = Q4_0, Q8_0, 1024, 256, 8
    idx = [(7 * k + 3) % n_exp for k in range(n)]
    c = _ffn_case(fmt_gu, fmt_dn, hidden, ffn, n_exp, idx, seed=n + 11)
    gd, ud, dd, ia = dev(c["g"]), dev(c["u"]), dev(c["d"]), dev(c["idx"])
    xq = Z.quantize_act_q8_0(dev(c["x"]))
    y, h = Z.expert_ffn(fmt_gu, gd, ud, c["gu_per"], fmt_dn, dd, c["dn_per"], hidden, ffn, ia, n_exp, xq,
                        y=nan_out(n, hidden))
    h2 = Z.expert_swiglu(fmt_gu, gd, ud, ffn, hidden, xq, idx=ia, expert_stride=c["gu_per"], n_experts=n_exp)
    y2 = Z.expert_gather(fmt_dn, dd, c["dn_per"], hidden, ffn, ia, n_exp, Z.quantize_act_q8_0(h2.reshape(-1)),
                         ffn // 32 * 34)
    torch.cuda.synchronize()
    assert torch.equal(h, h2) and torch.equal(y, y2)
    assert not torch.isnan(y).any()


def test_expert_ffn_bad_index_then_reuse_workspace():
    fmt_gu, fmt_dn, hidden, ffn, n_exp = Q4_0, Q8_0, 2048, 512, 4
    c = _ffn_case(fmt_gu, fmt_dn, hidden, ffn, n_exp, [1, 9, 0], seed=77)   # 9 is out of range
    gd, ud, dd = dev(c["g"]), dev(c["u"]), dev(c["d"])
    xq = Z.quantize_act_q8_0(dev(c["x"]))
    ws = Z.expert_ffn_workspace(3, ffn)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, h = Z.expert_ffn(fmt_gu, gd, ud, c["gu_per"], fmt_dn, dd, c["dn_per"], hidden, ffn, dev(c["idx"]), n_exp,
                        xq, y=nan_out(3, hidden), workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 1
    assert torch.isnan(y[1]).all() and torch.isnan(h[1]).all()
    assert not torch.isnan(y[0]).any() and not torch.isnan(y[2]).any()
    # the workspace's counters are back to zero: a second call with good indices is right
    good = dev(np.array([1, 3, 0], dtype=np.int32))
    y2, _ = Z.expert_ffn(fmt_gu, gd, ud, c["gu_per"], fmt_dn, dd, c["dn_per"], hidden, ffn, good, n_exp, xq,
                         y=nan_out(3, hidden), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y2[0], y[0]) and torch.equal(y2[2], y[2]) and not torch.isnan(y2[1]).any()


def test_expert_ffn_too_many_experts_for_one_resident_grid_is_a_shape_error():
    """Every CTA of the one-launch FFN must be resident at once (a waiting down CTA
    must never hold a slot a gate/up CTA needs), so a selection larger than half
    the CTAs that fit returns ERR_SHAPE before any launch, and the device is
    left without a fault."""
    hidden, ffn = 256, 256
    w_gu = dev(synth.weight_blocks(Q4_0, ffn, hidden, seed=3))
    w_dn = dev(synth.weight_blocks(Q8_0, hidden, ffn, seed=4))
    xq = Z.quantize_act_q8_0(dev(synth.activations(hidden, seed=5)))
    n = 4000
    idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    with pytest.raises(Z.ZdmmvError) as err:
        Z.expert_ffn(Q4_0, w_gu, w_gu, 0, Q8_0, w_dn, 0, hidden, ffn, idx, 1, xq)
    assert err.value.code == 2  # ZDMMV_ERR_SHAPE
    assert Z.device_status() == 0
