"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every function include/zdmmv.h declares, and rejects bad arguments on the host
before any launch. No kernel runs here (no GPU on this machine)."""
import ctypes

import pytest

from gguf_block_quant_gb300 import zdmmv


@pytest.fixture(scope="module")
def L():
    return zdmmv.lib()


def test_every_declared_function_is_exported(L):
    names = zdmmv.header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(zdmmv._SIGS), "binding and header disagree"


def _header_params():
    """{function: [C type of each parameter]} parsed from include/zdmmv.h."""
    import os
    import re
    from gguf_block_quant_gb300 import _build
    text = open(os.path.join(_build.INCLUDE, "zdmmv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(zdmmv_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        ps = [" ".join(p.split()) for p in params.split(",")] if params.strip() not in ("", "void") else []
        out[name] = ["ptr" if "*" in p else p.rsplit(" ", 1)[0] for p in ps]
    return out


def test_binding_signatures_match_the_header():
    """Every ctypes signature in the binding has the header's parameter count and,
    parameter by parameter, the matching ctypes type (pointers and streams as
    void*, int64_t, size_t, and int for int and the enums)."""
    want = {"ptr": ctypes.c_void_p, "zdmmv_stream_t": ctypes.c_void_p, "int64_t": ctypes.c_int64,
            "size_t": ctypes.c_size_t, "int": ctypes.c_int, "zdmmv_fmt": ctypes.c_int,
            "zdmmv_layout": ctypes.c_int, "zdmmv_status": ctypes.c_int}
    hdr = _header_params()
    assert set(hdr) == set(zdmmv._SIGS)
    for name, (args, _res) in zdmmv._SIGS.items():
        assert len(args) == len(hdr[name]), (name, len(args), len(hdr[name]))
        for i, (a, c) in enumerate(zip(args, hdr[name])):
            typed_ptr = c == "ptr" and isinstance(a, type) and issubclass(a, ctypes._Pointer)
            assert a is want[c] or typed_ptr, (name, i, c, a)


def test_status_strings_and_sizes(L):
    assert L.zdmmv_status_str(0) == b"ok"
    assert L.zdmmv_status_str(2) == b"bad shape"
    assert b"sm_103a" in L.zdmmv_version()
    assert L.zdmmv_block_bytes(zdmmv.Q8_0) == 34
    assert L.zdmmv_block_bytes(zdmmv.Q4_0) == 18
    assert L.zdmmv_block_bytes(3) == 0
    assert L.zdmmv_repacked_bytes(zdmmv.Q4_0, 4096, 4096) == 4096 * 128 * 18
    assert L.zdmmv_repacked_bytes(zdmmv.Q8_0, 3, 33) == 0
    # x (batch*cols fp32) + Q8_0 blocks + y (batch*rows fp32), each rounded to 256 B
    assert L.zdmmv_host_step_workspace_bytes(100, 64, 2) == 512 + 256 + 1024
    assert L.zdmmv_host_step_workspace_bytes(100, 64, 9) == 0


# Host-side argument checks return before any CUDA call, so they run without a GPU.
FAKE = 1 << 20          # a 16-byte aligned non-null "device" address, never dereferenced
ODD = FAKE + 2


def test_dmmv_argument_checks(L):
    for fn in (L.zdmmv_q8_0, L.zdmmv_q4_0):
        assert fn(None, 0, 4, 64, FAKE, FAKE, None) == 1            # null weights
        assert fn(FAKE, 0, 4, 48, FAKE, FAKE, None) == 2            # cols % 32
        assert fn(FAKE, 0, 4, 0, FAKE, FAKE, None) == 2             # cols == 0
        assert fn(FAKE, 0, -1, 64, FAKE, FAKE, None) == 2           # rows < 0
        assert fn(FAKE, 7, 4, 64, FAKE, FAKE, None) == 4            # layout
        assert fn(ODD, 0, 4, 64, FAKE, FAKE, None) == 3             # misaligned w
        assert fn(FAKE, 0, 4, 64, ODD, FAKE, None) == 3             # misaligned xq
        assert fn(FAKE, 0, 4, 64, FAKE, FAKE + 1, None) == 3        # misaligned y
    assert L.zdmmv_q8_0_batched(FAKE, 0, 4, 64, FAKE, 0, FAKE, None) == 2
    assert L.zdmmv_q8_0_batched(FAKE, 0, 4, 64, FAKE, 9, FAKE, None) == 2
    assert L.zdmmv_q4_0_batched(FAKE, 0, 4, 64, FAKE, 9, FAKE, None) == 2


def test_empty_inputs_are_no_ops(L):
    # rows == 0 / k == 0 / n == 0 return OK without touching the device
    assert L.zdmmv_q8_0(None, 0, 0, 64, None, None, None) == 0
    assert L.zdmmv_quantize_act_q8_0(None, 0, None, None) == 0
    assert L.zdmmv_expert_gather(2, FAKE, 1 << 16, 0, 4, 64, FAKE, 0, 8, FAKE, 0, FAKE, None, None) == 0
    assert L.zdmmv_repack(8, None, 0, 64, None, 0, None) == 0
    assert L.zdmmv_selftest_dp4a(None, None, None, None, 0, None) == 0


def test_other_argument_checks(L):
    assert L.zdmmv_quantize_act_q8_0(FAKE, 33, FAKE, None) == 2
    assert L.zdmmv_quantize_act_q8_0(None, 64, FAKE, None) == 1
    assert L.zdmmv_quantize_act_q8_0(FAKE + 2, 64, FAKE, None) == 3
    # the ready gather (indices already read by an earlier expert call) checks the same arguments
    for g in (L.zdmmv_expert_gather, L.zdmmv_expert_gather_ready):
        assert g(3, FAKE, 1 << 16, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 5      # format
        assert g(2, FAKE, 1 << 16, 0, 4, 64, None, 2, 8, FAKE, 0, FAKE, None, None) == 1      # idx null
        assert g(2, FAKE, 8, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 2            # stride < matrix
        assert g(2, FAKE, 1 << 16, 0, 4, 64, FAKE, 2, 8, FAKE, 40, FAKE, None, None) == 2     # xq stride < vector
        assert g(2, FAKE, (1 << 16) + 8, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 3  # stride % 16
        assert g(2, FAKE, 1 << 16, 0, 4, 64, FAKE, -1, 8, FAKE, 0, FAKE, None, None) == 2     # n < 0
        assert g(2, FAKE, 1 << 16, 0, 4, 64, FAKE + 2, 2, 8, FAKE, 0, FAKE, None, None) == 3  # idx misaligned
        assert g(2, FAKE, 1 << 16, 0, 4, 64, FAKE, 0, 8, FAKE, 0, FAKE, None, None) == 0      # n == 0
    gf = L.zdmmv_expert_gather_f32
    assert gf(2, FAKE, 1 << 16, 0, 4, 256, FAKE, 0, 8, FAKE, 0, FAKE, None, 0, None) == 0      # n == 0
    assert gf(3, FAKE, 1 << 16, 0, 4, 256, FAKE, 2, 8, FAKE, 0, FAKE, None, 0, None) == 5      # format
    assert gf(2, FAKE, 1 << 16, 0, 4, 96, FAKE, 2, 8, FAKE, 0, FAKE, None, 0, None) == 2       # off the pipelined widths
    assert gf(2, FAKE, 1 << 16, 0, 4, 256, None, 2, 8, FAKE, 0, FAKE, None, 1, None) == 1      # idx null
    assert gf(2, FAKE, 1 << 16, 0, 4, 256, FAKE, 2, 8, FAKE + 4, 0, FAKE, None, 0, None) == 3  # x not 16-byte aligned
    assert gf(2, FAKE, 1 << 16, 0, 4, 256, FAKE, 2, 8, FAKE, 258, FAKE, None, 0, None) == 3    # x stride % 4
    assert gf(2, FAKE, 1 << 16, 0, 4, 256, FAKE, 2, 8, FAKE, 128, FAKE, None, 0, None) == 2    # x stride < cols
    assert gf(2, FAKE, 8, 0, 4, 256, FAKE, 2, 8, FAKE, 0, FAKE, None, 0, None) == 2            # stride < matrix
    assert gf(2, FAKE, 1 << 16, 2, 4, 256, FAKE, 2, 8, FAKE, 0, FAKE, None, 0, None) == 4      # layout
    assert L.zdmmv_repack(8, FAKE, 4, 64, FAKE + 4096, 10, None) == 6                     # dst too small
    assert L.zdmmv_repack(8, FAKE, 4, 64, FAKE + 16, 4096, None) == 2                     # overlap
    assert L.zdmmv_repack(3, FAKE, 4, 64, FAKE + 4096, 4096, None) == 5
    assert L.zdmmv_host_step(8, FAKE, 0, 4, 64, FAKE, 1, FAKE, FAKE, 10, None) == 6
    assert L.zdmmv_host_step(8, FAKE, 0, 4, 64, FAKE, 0, FAKE, FAKE, 1 << 20, None) == 2
    assert L.zdmmv_device_status(None, 0) == 1
    assert L.zdmmv_selftest_wait_timeout(None, None) == 1
    c = L.zdmmv_dmmv_acc
    assert c(8, FAKE, 0, 0, 64, None, None, None, None) == 0        # no rows
    assert c(8, FAKE, 0, 4, 64, FAKE, None, None, None) == 1        # y null
    assert c(8, FAKE, 0, 4, 48, FAKE, None, FAKE, None) == 2
    assert c(8, FAKE, 0, 4, 64, FAKE, FAKE + 2, FAKE, None) == 3    # misaligned gate
    a = L.zdmmv_dmmv_argmax
    assert a(2, FAKE, 0, 100, 160, FAKE, FAKE, None, FAKE, 16384, None) == 2     # off the pipelined widths
    assert a(2, FAKE, 0, 0, 2048, FAKE, FAKE, None, FAKE, 16384, None) == 2      # no rows
    assert a(2, FAKE, 0, 100, 2048, FAKE, None, None, FAKE, 16384, None) == 1
    assert a(2, FAKE, 0, 100, 2048, FAKE, FAKE, None, FAKE, 1024, None) == 6     # workspace too small
    assert a(2, FAKE, 0, 100, 2048, FAKE, FAKE, None, FAKE + 4, 16384, None) == 3
    f = L.zdmmv_dmmv_f32
    assert f(8, FAKE, 0, 0, 64, None, 1, None, None) == 0                                # rows == 0
    assert f(8, None, 0, 4, 64, FAKE, 1, FAKE, None) == 1
    assert f(3, FAKE, 0, 4, 64, FAKE, 1, FAKE, None) == 5
    assert f(8, FAKE, 2, 4, 64, FAKE, 1, FAKE, None) == 4
    assert f(8, FAKE, 0, 4, 64, FAKE, 9, FAKE, None) == 2
    assert f(8, FAKE, 0, 4, 64, FAKE + 4, 1, FAKE, None) == 3
    assert f(8, FAKE + 8, 0, 4, 64, FAKE, 1, FAKE, None) == 3
    assert L.zdmmv_debug_block_sums(8, FAKE, 0, 4, 40, FAKE, FAKE, None) == 2
    g2 = L.zdmmv_expert_gather2
    assert g2(2, FAKE, None, 1 << 16, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, FAKE, None, None) == 1
    assert g2(2, FAKE, FAKE, 1 << 16, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, None, None, None) == 1
    assert g2(2, FAKE, FAKE + 8, 1 << 16, 0, 4, 64, FAKE, 2, 8, FAKE, 0, FAKE, FAKE, None, None) == 3
    assert g2(2, FAKE, FAKE, 1 << 16, 0, 4, 64, FAKE, 0, 8, FAKE, 0, FAKE, FAKE, None, None) == 0
    xf = L.zdmmv_dmmv_xf32
    assert xf(8, FAKE, 0, 0, 64, None, 1, None, None) == 0                              # rows == 0
    assert xf(8, None, 0, 4, 64, FAKE, 1, FAKE, None) == 1
    assert xf(3, FAKE, 0, 4, 64, FAKE, 1, FAKE, None) == 5
    assert xf(8, FAKE, 2, 4, 64, FAKE, 1, FAKE, None) == 4
    assert xf(8, FAKE, 0, 4, 48, FAKE, 1, FAKE, None) == 2                              # cols % 32
    assert xf(8, FAKE, 0, 4, 64, FAKE, 0, FAKE, None) == 2                              # batch 0
    assert xf(8, FAKE, 0, 4, 64, FAKE + 4, 1, FAKE, None) == 3                          # x not 16-byte aligned
    ff = L.zdmmv_expert_ffn
    wsb = L.zdmmv_expert_ffn_workspace_bytes(9, 512)
    assert wsb >= 9 * 512 * 4 + 2 * 9 * 4
    args = lambda **k: [k.get("fgu", 2), FAKE, FAKE, 1 << 21, k.get("fdn", 8), FAKE, 1 << 21,
                        k.get("hidden", 2048), k.get("ffn", 512), FAKE, k.get("n", 9), 129, FAKE, FAKE,
                        k.get("ws", FAKE), k.get("wsb", wsb), None, None]
    assert ff(*args(fgu=3)) == 5
    assert ff(*args(hidden=2048 + 32)) == 2          # off the pipelined widths
    assert ff(*args(ffn=4096)) == 2                  # down rows wider than the kernel takes
    assert ff(*args(n=0)) == 0
    assert ff(*args(ws=None)) == 1
    assert ff(*args(ws=FAKE + 16)) == 3              # workspace not 256-byte aligned
    assert ff(*args(wsb=wsb - 1)) == 6
    small = [2, FAKE, FAKE, 1 << 16, 8, FAKE, 1 << 21, 2048, 512, FAKE, 9, 129, FAKE, FAKE, FAKE, wsb, None, None]
    assert ff(*small) == 2                           # experts of the gate/up stack overlap
    sw = L.zdmmv_expert_swiglu
    assert sw(2, FAKE, FAKE, 1 << 16, 0, 4, 160, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 2  # off the pipelined widths
    assert sw(2, FAKE, FAKE, 0, 0, 4, 2048, None, 2, 0, FAKE, 0, FAKE, None, None) == 2       # no index, n > 1
    assert sw(2, FAKE, None, 1 << 16, 0, 4, 2048, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 1
    assert sw(2, FAKE, FAKE + 8, 1 << 16, 0, 4, 2048, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 3
    assert sw(2, FAKE, FAKE, 1 << 16, 0, 4, 2048, FAKE, 2, 8, FAKE, 100, FAKE, None, None) == 2  # xq stride short
    assert sw(2, FAKE, FAKE, 1008, 0, 4, 2048, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 2     # experts overlap
    assert sw(2, FAKE, FAKE, 1 << 16, 0, 4, 2048, FAKE, 0, 8, FAKE, 0, FAKE, None, None) == 0  # n == 0
    assert sw(3, FAKE, FAKE, 1 << 16, 0, 4, 2048, FAKE, 2, 8, FAKE, 0, FAKE, None, None) == 5
