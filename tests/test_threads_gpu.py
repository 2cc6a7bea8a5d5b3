"""Calls from several host threads at once, each on its own stream, from the
first call of a fresh process (the per-device set-up runs concurrently): every
result equals the same call made afterwards from one thread, bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, threading, numpy as np, torch
sys.path.insert(0, {root!r})
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z
Q4, Q8 = Z.Q4_0, Z.Q8_0
torch.cuda.init()
cases = []
for i, (fmt, rows, cols, batch) in enumerate([(Q4, 4096, 4096, 1), (Q8, 3000, 2048, 4), (Q4, 1024, 8192, 2),
                                              (Q8, 777, 4096, 8)]):
    w = torch.from_numpy(synth.weight_blocks(fmt, rows, cols, seed=40 + i)).cuda()
    x = torch.from_numpy(np.ascontiguousarray(synth.activations(cols, seed=50 + i, batch=batch))).cuda()
    cases.append((fmt, rows, cols, batch, w, x.reshape(-1)))
torch.cuda.synchronize()

def run(case, stream):
    fmt, rows, cols, batch, w, x = case
    with torch.cuda.stream(stream):
        xq = Z.quantize_act_q8_0(x, stream=stream)
        if batch == 1:
            a = Z.dmmv_f32(fmt, w, rows, cols, x, stream=stream)
            b = Z.dmmv(fmt, w, rows, cols, xq, stream=stream)
            idx = Z.dmmv_argmax(fmt, w, rows, cols, xq, stream=stream)[0]
            out = [a, b, idx]
        else:
            out = [Z.dmmv_batched(fmt, w, rows, cols, xq, batch, stream=stream),
                   Z.dmmv_f32(fmt, w, rows, cols, x, batch=batch, stream=stream)]
    stream.synchronize()
    return [o.clone() for o in out]

streams = [torch.cuda.Stream() for _ in cases]
results = [None] * len(cases)
errors = []
def worker(k):
    try:
        outs = []
        for _ in range(5):
            outs.append(run(cases[k], streams[k]))
        results[k] = outs
    except Exception as e:  # reported by the parent
        errors.append(repr(e))
threads = [threading.Thread(target=worker, args=(k,)) for k in range(len(cases))]
for t in threads: t.start()
for t in threads: t.join()
assert not errors, errors
s = torch.cuda.Stream()
for k, case in enumerate(cases):
    ref = run(case, s)
    for outs in results[k]:
        for a, b in zip(outs, ref):
            assert torch.equal(a, b), k
assert Z.device_status() == 0
print("ok")
"""


def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "ok"
