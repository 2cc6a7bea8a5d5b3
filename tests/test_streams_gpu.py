"""Launch configuration on the GPU: calls run on the stream they are given (a
side stream, ordered by events against the default one), and the same results
come out with programmatic dependent launch switched off (ZDMMV_PDL=0, read once
per process, so that case runs in a child process)."""
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


def test_calls_run_on_the_given_stream():
    Z.lib()
    fmt, rows, cols, layers = Z.Q4_0, 2048, 4096, 6
    ws = [synth.weight_blocks(fmt, rows, cols, seed=900 + i) for i in range(layers)]
    xs = [synth.activations(cols, seed=950 + i) for i in range(layers)]
    side = torch.cuda.Stream()
    wd = [torch.from_numpy(w).cuda() for w in ws]
    xd = [torch.from_numpy(x).cuda() for x in xs]
    ready = torch.cuda.Event()
    ready.record()
    ys = []
    with torch.cuda.stream(side):
        side.wait_event(ready)
        for w, x in zip(wd, xd):
            ys.append(Z.dmmv_f32(fmt, w, rows, cols, x, stream=side))   # a chain on the side stream
    done = torch.cuda.Event()
    done.record(side)
    torch.cuda.current_stream().wait_event(done)
    torch.cuda.synchronize()
    for w, x, y in zip(ws, xs, ys):
        y_ref, e_ref = oracle.dmmv(fmt, w, rows, cols, oracle.quantize_q8_0(x))
        ok, worst = oracle.within_tolerance(y.double().cpu().numpy(), y_ref, e_ref)
        assert ok, worst


_CHILD = r"""
import sys, json, numpy as np, torch
sys.path.insert(0, {root!r})
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z
out = []
for fmt, rows, cols, seed in [(Z.Q4_0, 4096, 4096, 1), (Z.Q8_0, 3000, 2048, 2)]:
    w = torch.from_numpy(synth.weight_blocks(fmt, rows, cols, seed=seed)).cuda()
    x = torch.from_numpy(synth.activations(cols, seed=seed + 1, batch=2)).cuda()
    y1 = Z.dmmv_f32(fmt, w, rows, cols, x[0])
    yb = Z.dmmv_batched(fmt, w, rows, cols, Z.quantize_act_q8_0(x), 2)
    torch.cuda.synchronize()
    out.append(np.concatenate([y1.cpu().numpy(), yb.cpu().numpy().ravel()]).view(np.uint32).tolist())
print(json.dumps(out))
"""


def _run_child(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout.strip().splitlines()[-1]


def test_results_do_not_depend_on_programmatic_dependent_launch():
    assert _run_child({"ZDMMV_PDL": "0"}) == _run_child({"ZDMMV_PDL": "1"})


_CHILD_VSPLIT = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z
# the last shape is the tensor-core kernel's by default (a 32-row group per SM)
for fmt, rows, cols, batch in [(Z.Q8_0, 1434, 4096, 8), (Z.Q4_0, 901, 2048, 3), (Z.Q8_0, 4900, 4096, 8)]:
    w = torch.from_numpy(synth.weight_blocks(fmt, rows, cols, seed=batch)).cuda()
    xq = Z.quantize_act_q8_0(torch.from_numpy(synth.activations(cols, seed=batch + 3, batch=batch)).cuda())
    yb = Z.dmmv_batched(fmt, w, rows, cols, xq, batch)
    nbx = cols // 32 * 34
    for v in range(batch):
        ys = Z.dmmv(fmt, w, rows, cols, xq[v * nbx:(v + 1) * nbx].clone())
        torch.cuda.synchronize()
        assert torch.equal(ys, yb[v]), (fmt, cols, batch, v)
print("ok")
"""


def test_vector_split_kernel_equals_single_vector_calls_bitwise():
    """ZDMMV_BATCH_KERNEL=vsplit (read once per process, hence a child process)
    keeps every batch on the vector split, also those the tensor-core kernel
    takes by default: each vector's output equals its single-vector call bit for
    bit."""
    env = dict(os.environ, ZDMMV_BATCH_KERNEL="vsplit")
    r = subprocess.run([sys.executable, "-c", _CHILD_VSPLIT.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "ok"
