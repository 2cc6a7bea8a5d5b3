"""The allocation-free argmax entry point, for callers that cannot allocate
device memory (an engine that plans all device memory at load time, a plugin
whose host owns every allocation, a decode loop that must not call cudaMalloc).

It is called through the C ABI (ctypes, raw device pointers) and must return
the same pick as zdmmv_dmmv_argmax with a caller workspace, on two calls in a
row that share the library's fixed scratch array. This file is collected last
so that a run stopping at the first failure has run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu


def test_no_alloc_argmax_matches_the_workspace_entry_point():
    L = Z.lib()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(Z.Q4_0, 248320 // 4, 2048, 31), (Z.Q8_0, 3000, 4096, 32)]   # two calls in a row
    for fmt, rows, cols, seed in cases:
        w = torch.from_numpy(synth.weight_blocks(fmt, rows, cols, seed=seed)).cuda()
        xq = torch.from_numpy(synth.activation_blocks(cols // 32, seed=seed + 1)).cuda()
        idx = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        mx = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        rc = L.zdmmv_dmmv_argmax_noalloc(fmt, w.data_ptr(), Z.GGUF, rows, cols, xq.data_ptr(),
                                         idx.data_ptr(), mx.data_ptr(), ctypes.c_void_p(stream))
        assert rc == 0, Z.STATUS.get(rc)
        ref_mx = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        ref = Z.dmmv_argmax(fmt, w, rows, cols, xq, max_out=ref_mx)
        torch.cuda.synchronize()
        assert int(idx.item()) == int(ref.item())
        # the same logit, within the tolerance used for every DMMV output
        y_ref, e_ref = oracle.dmmv(fmt, w.cpu().numpy().reshape(rows, -1)[int(ref.item())], 1, cols,
                                   xq.cpu().numpy())
        ok, worst = oracle.within_tolerance([mx.item()], [ref_mx.item()], e_ref)
        assert ok, worst
    assert Z.device_status() == 0
