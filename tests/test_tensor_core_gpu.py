"""The fp16 tensor-core batched kernel (zdmmv_bmma.cuh).

Forced with ZDMMV_BATCH_KERNEL=mma (read once per process, so those checks run in
a child process): results against the oracle on ragged and chunked shapes for
1..8 vectors, exact integer outputs bit for bit on the formats' extreme codes,
and that the tensor-core kernel is the one that ran (its results are not bitwise
the single-vector calls', as the vector split's are). In the default process:
the kernel is chosen for 5..8 vectors on matrices with a 32-row group for every
SM, and the vector split (bitwise the single-vector calls) below that; the fused
entry point (fp32 activations) then gives the bits of the quantizer followed by
the batched call."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z
Q4, Q8 = Z.Q4_0, Z.Q8_0
checked = 0
# ragged last 32-row group, one row past a group, uneven chunks of 32 blocks
# (1280 columns: 32 + 8 blocks; 2304: 32 + 32 + 8), exactly one group, whole chunks
for fmt, rows, cols in [(Q8, 1000, 2304), (Q4, 33, 1280), (Q8, 32, 4096), (Q4, 4101, 4096), (Q8, 47, 1536),
                        (Q4, 250, 1280), (Q8, 1434, 4096)]:
    for batch in (1, 3, 5, 8):
        w = synth.weight_blocks(fmt, rows, cols, seed=rows + cols)
        x = synth.activations(cols, seed=batch + cols, batch=batch)
        xq = Z.quantize_act_q8_0(torch.from_numpy(x).cuda())
        y = Z.dmmv_batched(fmt, torch.from_numpy(w).cuda(), rows, cols, xq, batch)
        torch.cuda.synchronize()
        y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, oracle.quantize_q8_0(x), batch)
        ok, worst = oracle.within_tolerance(y.double().cpu().numpy().reshape(batch, rows), y_ref, e_ref)
        assert ok, (fmt, rows, cols, batch, worst)
        checked += 1
# the formats' extreme codes (Q8_0 -128 / 127, Q4_0 0 / 15) in 16 blocks of each row,
# zero codes elsewhere, against activation codes -128 / 127, unit scales: every
# output is an exact integer below 2^24, so the kernel's block sums (its fp16
# codes with their offsets and the accumulator start that removes them) must give
# the oracle's values bit for bit
for fmt in (Q8, Q4):
    bb, zero = (34, 0x00) if fmt == Q8 else (18, 0x88)
    for cols in (1280, 2304):
        for batch in (2, 8):
            rows, nb = 77, cols // 32
            w = synth.extreme_code_blocks(fmt, rows * nb, seed=cols + batch, stream=synth.S_WEIGHT)
            w = w.reshape(rows, nb, bb)
            g = np.random.default_rng(cols * 10 + batch)
            for r in range(rows):
                keep = g.permutation(nb)[:16]
                off = np.setdiff1d(np.arange(nb), keep)
                w[r, off, 2:] = zero
            w = np.ascontiguousarray(w).reshape(-1)
            xq = synth.extreme_code_blocks(Q8, batch * nb, seed=cols * batch)
            y = Z.dmmv_batched(fmt, torch.from_numpy(w).cuda(), rows, cols, torch.from_numpy(xq).cuda(), batch)
            torch.cuda.synchronize()
            y_ref, _ = oracle.dmmv_batched(fmt, w, rows, cols, xq, batch)
            assert np.array_equal(y.double().cpu().numpy().reshape(batch, rows), y_ref), (fmt, cols, batch)
            checked += 1
# the fused entry point takes the same kernel with the quantization in its
# prologue: the bits of the quantizer followed by the batched call
for fmt, rows, cols, batch in [(Q8, 300, 2304, 2), (Q4, 65, 4096, 3), (Q8, 1434, 1280, 8)]:
    w = torch.from_numpy(synth.weight_blocks(fmt, rows, cols, seed=rows)).cuda()
    x = torch.from_numpy(synth.activations(cols, seed=cols + batch, batch=batch)).cuda()
    yf = Z.dmmv_f32(fmt, w, rows, cols, x, batch=batch)
    yb = Z.dmmv_batched(fmt, w, rows, cols, Z.quantize_act_q8_0(x.reshape(-1)), batch)
    torch.cuda.synchronize()
    assert torch.equal(yf.reshape(batch, rows), yb.reshape(batch, rows)), (fmt, rows, cols, batch)
    checked += 1
# the launch is the tensor-core kernel: the vector split gives every vector's
# single-vector result bit for bit; the tensor-core kernel sums the blocks of a
# row in another order, so some output bits differ
w = torch.from_numpy(synth.weight_blocks(Q8, 512, 4096, seed=1)).cuda()
xq = Z.quantize_act_q8_0(torch.from_numpy(synth.activations(4096, seed=2, batch=4)).cuda())
yb = Z.dmmv_batched(Q8, w, 512, 4096, xq, 4)
ys = torch.stack([Z.dmmv(Q8, w, 512, 4096, xq[v * 4352:(v + 1) * 4352].clone()) for v in range(4)])
torch.cuda.synchronize()
assert not torch.equal(yb.reshape(4, 512), ys)
assert Z.device_status() == 0
print("ok", checked)
"""


def test_tensor_core_batched_kernel():
    env = dict(os.environ, ZDMMV_BATCH_KERNEL="mma")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "ok 39"


def _rows_for_every_sm(extra):
    """Rows giving every SM one 32-row group of the tensor-core kernel, plus extra."""
    return 32 * torch.cuda.get_device_properties(0).multi_processor_count + extra


def _batched_and_singles(fmt, rows, cols, batch, seed):
    w = synth.weight_blocks(fmt, rows, cols, seed=seed)
    x = synth.activations(cols, seed=seed + 1, batch=batch)
    wd = torch.from_numpy(w).cuda()
    xq = Z.quantize_act_q8_0(torch.from_numpy(x).cuda())
    y = torch.full((batch, rows), float("nan"), device="cuda")
    Z.dmmv_batched(fmt, wd, rows, cols, xq, batch, y=y)
    y2 = torch.full((batch, rows), float("nan"), device="cuda")
    Z.dmmv_batched(fmt, wd, rows, cols, xq, batch, y=y2)
    nbx = cols // 32 * 34
    ys = torch.stack([Z.dmmv(fmt, wd, rows, cols, xq[v * nbx:(v + 1) * nbx].clone()) for v in range(batch)])
    torch.cuda.synchronize()
    y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, oracle.quantize_q8_0(x), batch)
    ok, worst = oracle.within_tolerance(y.double().cpu().numpy(), y_ref, e_ref)
    assert ok, worst
    assert torch.equal(y, y2), "the same call gave other bits"
    return y, ys


@pytest.mark.parametrize("fmt,extra,cols,batch", [(synth.Q8_0, 37, 4096, 5), (synth.Q8_0, 0, 4096, 8),
                                                  (synth.Q4_0, 129, 2304, 6), (synth.Q4_0, 5, 1280, 7)])
def test_default_batches_of_five_or_more_take_the_tensor_cores(fmt, extra, cols, batch):
    y, ys = _batched_and_singles(fmt, _rows_for_every_sm(extra), cols, batch, seed=extra + cols)
    assert not torch.equal(y, ys), "expected the tensor-core kernel's reduction order"


@pytest.mark.parametrize("fmt,extra,cols,batch", [(synth.Q8_0, 37, 4096, 4), (synth.Q4_0, -40, 2304, 8)])
def test_default_smaller_batches_and_matrices_keep_the_vector_split(fmt, extra, cols, batch):
    """4 vectors, or fewer rows than a 32-row group per SM: the vector split,
    bitwise the single-vector calls."""
    y, ys = _batched_and_singles(fmt, _rows_for_every_sm(extra), cols, batch, seed=extra + cols + 1)
    assert torch.equal(y, ys)


@pytest.mark.parametrize("fmt,extra,cols,batch", [(synth.Q8_0, 37, 4096, 5), (synth.Q8_0, 0, 4096, 8),
                                                  (synth.Q4_0, 129, 2304, 6), (synth.Q4_0, 5, 1280, 7),
                                                  (synth.Q8_0, 37, 4096, 4)])
def test_fused_entry_equals_quantize_then_batched(fmt, extra, cols, batch):
    """zdmmv_dmmv_f32 with 4..8 vectors: bit for bit the quantizer followed by the
    batched call (the tensor-core kernel from 5 vectors on these shapes, the
    vector split at 4), and within the oracle's tolerance."""
    rows = _rows_for_every_sm(extra)
    w = synth.weight_blocks(fmt, rows, cols, seed=extra + 3)
    x = synth.activations(cols, seed=extra + 4, batch=batch)
    wd = torch.from_numpy(w).cuda()
    xd = torch.from_numpy(x).cuda()
    yf = torch.full((batch, rows), float("nan"), device="cuda")
    Z.dmmv_f32(fmt, wd, rows, cols, xd, batch=batch, y=yf)
    yb = torch.full((batch, rows), float("nan"), device="cuda")
    Z.dmmv_batched(fmt, wd, rows, cols, Z.quantize_act_q8_0(xd.reshape(-1)), batch, y=yb)
    torch.cuda.synchronize()
    assert torch.equal(yf, yb)
    y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, oracle.quantize_q8_0(x), batch)
    ok, worst = oracle.within_tolerance(yf.double().cpu().numpy(), y_ref, e_ref)
    assert ok, worst
