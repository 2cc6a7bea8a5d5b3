"""The integer tensor-core batched kernel (ZDMMV_BATCH_KERNEL=mma; the variable
is read once per process, so the checks run in a child process): results
against the oracle on ragged, chunked and narrow shapes, the formats' extreme
codes bit for bit, and that the tensor-core kernel is the one that ran (its
results are not bitwise the single-vector calls', as the default kernel's are)."""
import os
import subprocess
import sys

import pytest

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
# ragged last slab (rows % 16), uneven chunks (2304 columns: 40 + 32 blocks), fewer
# block pairs than warps (256 columns), one and two chunks, 16 rows exactly
for fmt, rows, cols in [(Q8, 1000, 2304), (Q4, 33, 256), (Q8, 17, 256), (Q4, 4101, 4096), (Q8, 16, 4096),
                        (Q4, 250, 1280), (Q8, 1434, 4096)]:
    for batch in (2, 5, 8):
        w = synth.weight_blocks(fmt, rows, cols, seed=rows + cols)
        x = synth.activations(cols, seed=batch + cols, batch=batch)
        xq = Z.quantize_act_q8_0(torch.from_numpy(x).cuda())
        y = Z.dmmv_batched(fmt, torch.from_numpy(w).cuda(), rows, cols, xq, batch)
        torch.cuda.synchronize()
        y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, oracle.quantize_q8_0(x), batch)
        ok, worst = oracle.within_tolerance(y.double().cpu().numpy(), y_ref, e_ref)
        assert ok, (fmt, rows, cols, batch, worst)
        checked += 1
# extreme codes, unit scales, at most 16 blocks a row: exact integers, bit for bit
for fmt in (Q8, Q4):
    for cols in (256, 512):
        for batch in (2, 8):
            rows = 77
            w = synth.extreme_code_blocks(fmt, rows * cols // 32, seed=cols + batch, stream=synth.S_WEIGHT)
            xq = synth.extreme_code_blocks(Q8, batch * cols // 32, seed=cols * batch)
            y = Z.dmmv_batched(fmt, torch.from_numpy(w).cuda(), rows, cols, torch.from_numpy(xq).cuda(), batch)
            torch.cuda.synchronize()
            y_ref, _ = oracle.dmmv_batched(fmt, w, rows, cols, xq, batch)
            assert np.array_equal(y.double().cpu().numpy(), y_ref), (fmt, cols, batch)
            checked += 1
# the launch is the tensor-core kernel: the vector split (the default) gives every
# vector's single-vector result bit for bit; the tensor-core kernel sums the blocks
# of a row in another order, so some output bits differ
w = torch.from_numpy(synth.weight_blocks(Q8, 512, 4096, seed=1)).cuda()
xq = Z.quantize_act_q8_0(torch.from_numpy(synth.activations(4096, seed=2, batch=8)).cuda())
yb = Z.dmmv_batched(Q8, w, 512, 4096, xq, 8)
ys = torch.stack([Z.dmmv(Q8, w, 512, 4096, xq[v * 4352:(v + 1) * 4352].clone()) for v in range(8)])
torch.cuda.synchronize()
assert not torch.equal(yb, ys)
print("ok", checked)
"""


def test_tensor_core_batched_kernel():
    env = dict(os.environ, ZDMMV_BATCH_KERNEL="mma")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "ok 29"
