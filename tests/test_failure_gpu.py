"""Failure detection on the GPU without faulting it: a bounded wait on a
barrier that nothing completes must give up, report the fault through the
device status word, and leave the context usable for the next launch."""
import time

import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    Z.lib()
    assert Z.device_status(clear=True) == 0
    t0 = time.perf_counter()
    r = Z.selftest_wait_timeout()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert r.item() == 1, "the wait should have given up"
    assert 0.5 < elapsed < 30.0
    bits = Z.device_status(clear=True)
    assert bits & Z.FAULT_WAIT_TIMEOUT
    assert Z.device_status() == 0
    # the context is still usable: a normal DMMV afterwards is correct
    rows, cols = 256, 2048
    w = synth.weight_blocks(Z.Q4_0, rows, cols, seed=5)
    x = synth.activations(cols, seed=6)
    y = Z.dmmv_f32(Z.Q4_0, torch.from_numpy(w).cuda(), rows, cols, torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    y_ref, e_ref = oracle.dmmv(Z.Q4_0, w, rows, cols, oracle.quantize_q8_0(x))
    ok, worst = oracle.within_tolerance(y.double().cpu().numpy(), y_ref, e_ref)
    assert ok, worst
    assert Z.device_status() == 0
