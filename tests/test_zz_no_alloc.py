"""The allocation-free argmax entry point, for callers that cannot allocate
device memory (an engine that plans all device memory at load time, a plugin
whose host owns every allocation, a decode loop that must not call cudaMalloc).

It is called through the C ABI (ctypes, raw device pointers). Its pick and
maximum must equal those of zdmmv_dmmv_argmax with a caller workspace bit for
bit (both run the same kernels, only the partials live elsewhere), the pick must
be a valid argmax of the CPU oracle's logits within the DMMV tolerance, and the
maximum must be the kernel's own fp32 logit of that row, on calls in a row that
share the library's fixed scratch array: both layouts, a matrix with fewer rows
than the launch has CTAs, and no max output. Free device memory must not change
across a call. This file is collected last so that a run stopping at the first
failure has run every other test; it also passes on its own in a fresh process.
"""
import ctypes
import gc

import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6

# (fmt, layout, rows, cols, seed, with max_out); consecutive calls share the scratch
CASES = [
    (Z.Q4_0, Z.GGUF, 248320 // 4, 2048, 31, True),
    (Z.Q8_0, Z.GGUF, 3000, 4096, 32, True),
    (Z.Q4_0, Z.REPACKED, 5000, 2048, 33, True),
    (Z.Q8_0, Z.GGUF, 100, 4096, 34, True),      # fewer rows than CTAs in a full launch
    (Z.Q8_0, Z.REPACKED, 7, 512, 35, True),
    (Z.Q4_0, Z.GGUF, 20000, 2048, 36, False),   # no max output
]


def _noalloc(L, fmt, wd, layout, rows, cols, xqd, idx, mx):
    stream = torch.cuda.current_stream().cuda_stream
    return L.zdmmv_dmmv_argmax_noalloc(fmt, wd.data_ptr(), layout, rows, cols, xqd.data_ptr(), idx.data_ptr(),
                                       mx.data_ptr() if mx is not None else None, ctypes.c_void_p(stream))


def _inputs(fmt, layout, rows, cols, seed):
    w = synth.weight_blocks(fmt, rows, cols, seed=seed)
    xq = synth.activation_blocks(cols // 32, seed=seed + 1)
    wd = torch.from_numpy(w).cuda()
    if layout == Z.REPACKED:
        wd = Z.repack(fmt, wd, rows, cols)
    return w, xq, wd, torch.from_numpy(xq).cuda()


def test_no_alloc_argmax_matches_the_workspace_entry_point_and_the_oracle():
    L = Z.lib()
    for fmt, layout, rows, cols, seed, with_max in CASES:
        w, xq, wd, xqd = _inputs(fmt, layout, rows, cols, seed)
        idx = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        mx = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda") if with_max else None
        rc = _noalloc(L, fmt, wd, layout, rows, cols, xqd, idx, mx)
        assert rc == 0, Z.STATUS.get(rc)
        ref_mx = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        ref = Z.dmmv_argmax(fmt, wd, rows, cols, xqd, max_out=ref_mx, layout=layout)
        y = Z.dmmv(fmt, wd, rows, cols, xqd, layout=layout)
        torch.cuda.synchronize()
        i = int(idx.item())
        # the workspace entry point's pick and maximum, bit for bit
        assert i == int(ref.item())
        if with_max:
            assert mx.view(torch.int32).item() == ref_mx.view(torch.int32).item()
            # the maximum is the kernel's own fp32 logit of the picked row, and the first maximum
            yh = y.cpu().numpy()
            assert mx.item() == yh[i] and i == int(np.argmax(yh))
        # a valid argmax of the oracle's logits within the DMMV tolerance
        y_ref, e_ref = oracle.dmmv(fmt, w, rows, cols, xq)
        j, _ = oracle.argmax(y_ref)
        assert 0 <= i < rows
        assert y_ref[i] >= y_ref[j] - (REL * (e_ref[i] + e_ref[j]) + 2 * ABS)
    assert Z.device_status() == 0


def test_no_alloc_argmax_allocates_nothing():
    L = Z.lib()
    fmt, layout, rows, cols = Z.Q4_0, Z.GGUF, 248320 // 8, 2048
    _, _, wd, xqd = _inputs(fmt, layout, rows, cols, 40)
    idx = torch.empty(1, dtype=torch.int32, device="cuda")
    mx = torch.empty(1, dtype=torch.float32, device="cuda")
    assert _noalloc(L, fmt, wd, layout, rows, cols, xqd, idx, mx) == 0   # the first call sets the device up
    torch.cuda.synchronize()
    first = int(idx.item())
    # tensors of earlier tests are freed by the garbage collector at arbitrary
    # points: collect them now and keep the collector off while measuring
    gc.collect()
    gc.disable()
    try:
        torch_before = torch.cuda.memory_allocated()
        free_before, _ = torch.cuda.mem_get_info()
        for _ in range(2):
            assert _noalloc(L, fmt, wd, layout, rows, cols, xqd, idx, mx) == 0
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        torch_after = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert torch_after == torch_before
    assert free_after == free_before
    assert int(idx.item()) == first
