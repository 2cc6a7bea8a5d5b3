"""ctypes binding of the plain-C CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this module.
The CUDA library never imports, links or calls it, and it imports nothing from
the CUDA library.

Every function here is a thin marshalling layer over the C function of the same
name; the arithmetic lives in ``oracle.c`` (see the header there for the
definitions it follows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

Q4_0 = 2
Q8_0 = 8
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34}
QUANT_BYTES = {Q4_0: 16, Q8_0: 32}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C99, no fast-math, no FMA contraction)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(L):
    """Declare the argument and result types of every exported function."""
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64 = ctypes.c_int64
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_half_to_double.restype = ctypes.c_double
    L.oracle_float_to_half_rne.argtypes = [ctypes.c_float]
    L.oracle_float_to_half_rne.restype = ctypes.c_uint16
    L.oracle_dp4a.argtypes = [ctypes.c_int32] * 3
    L.oracle_dp4a.restype = ctypes.c_int32
    L.oracle_block_bytes.argtypes = [ctypes.c_int]
    L.oracle_block_bytes.restype = ctypes.c_int
    L.oracle_quantize_q8_0.argtypes = [ctypes.POINTER(ctypes.c_float), i64, u8p]
    L.oracle_quantize_q8_0.restype = None
    L.oracle_decode_block.argtypes = [ctypes.c_int, u8p, ctypes.POINTER(ctypes.c_uint16), i32p]
    L.oracle_dequantize.argtypes = [ctypes.c_int, u8p, i64, f64p]
    L.oracle_block_sums.argtypes = [ctypes.c_int, u8p, i64, i64, u8p, i32p]
    L.oracle_dmmv.argtypes = [ctypes.c_int, u8p, i64, i64, u8p, f64p, f64p]
    L.oracle_dmmv_xf32.argtypes = [ctypes.c_int, u8p, i64, i64, ctypes.POINTER(ctypes.c_float), f64p, f64p]
    L.oracle_dmmv_batched.argtypes = [ctypes.c_int, u8p, i64, i64, u8p, ctypes.c_int,
                                      f64p, f64p]
    L.oracle_expert_gather.argtypes = [ctypes.c_int, u8p, i64, i64, i64, i32p, ctypes.c_int,
                                       ctypes.c_int, u8p, i64, f64p, f64p, i32p]
    L.oracle_dmmv_acc.argtypes = [ctypes.c_int, u8p, i64, i64, u8p, f64p, f64p, f64p]
    L.oracle_swiglu.argtypes = [f64p, f64p, i64, f64p]
    L.oracle_swiglu.restype = None
    L.oracle_argmax.argtypes = [f64p, i64, f64p]
    L.oracle_argmax.restype = ctypes.c_int64
    L.oracle_repack.argtypes = [ctypes.c_int, u8p, i64, i64, u8p]
    L.oracle_unpack.argtypes = [ctypes.c_int, u8p, i64, i64, u8p]
    return L


class using_library:
    """Context manager that routes this module's calls to another build of the
    oracle. Used only by the tests that plant a mistake in a copy of oracle.c and
    check that the pins catch it."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        lib()
        with _lock:
            self.saved = _lib
            _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _p(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(int(bits) & 0xFFFF)


def float_to_half_rne(f: float) -> int:
    return int(lib().oracle_float_to_half_rne(float(f)))


def dp4a(a: int, b: int, c: int = 0) -> int:
    def s32(v):
        v &= 0xFFFFFFFF
        return v - (1 << 32) if v >= (1 << 31) else v
    return int(lib().oracle_dp4a(s32(a), s32(b), s32(c)))


def pack_int8x4(vals) -> int:
    """Pack four signed int8 values into one 32-bit word, byte 0 = vals[0]."""
    w = 0
    for i, v in enumerate(vals):
        w |= (int(v) & 0xFF) << (8 * i)
    return w


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    if x.size % 32:
        raise ValueError("quantize_q8_0: length must be a multiple of 32")
    out = np.zeros(x.size // 32 * 34, dtype=np.uint8)
    if x.size:
        lib().oracle_quantize_q8_0(_p(x, ctypes.c_float), x.size, _p(out, ctypes.c_uint8))
    return out


def decode_block(fmt: int, blk) -> tuple[int, np.ndarray]:
    blk = _u8(blk)
    d = ctypes.c_uint16()
    q = np.zeros(32, dtype=np.int32)
    _check(lib().oracle_decode_block(fmt, _p(blk, ctypes.c_uint8), ctypes.byref(d),
                                     _p(q, ctypes.c_int32)), "decode_block")
    return int(d.value), q


def dequantize(fmt: int, blocks) -> np.ndarray:
    blocks = _u8(blocks)
    nblk = blocks.size // BLOCK_BYTES[fmt]
    out = np.zeros(nblk * 32, dtype=np.float64)
    _check(lib().oracle_dequantize(fmt, _p(blocks, ctypes.c_uint8), nblk,
                                   _p(out, ctypes.c_double)), "dequantize")
    return out


def block_sums(fmt: int, w, rows: int, cols: int, xq) -> np.ndarray:
    w, xq = _u8(w), _u8(xq)
    out = np.zeros((rows, cols // 32), dtype=np.int32)
    _check(lib().oracle_block_sums(fmt, _p(w, ctypes.c_uint8), rows, cols,
                                   _p(xq, ctypes.c_uint8), _p(out, ctypes.c_int32)),
           "block_sums")
    return out


def dmmv(fmt: int, w, rows: int, cols: int, xq) -> tuple[np.ndarray, np.ndarray]:
    """Returns (y_ref, err_scale), both float64 [rows]."""
    w, xq = _u8(w), _u8(xq)
    y = np.zeros(rows, dtype=np.float64)
    e = np.zeros(rows, dtype=np.float64)
    _check(lib().oracle_dmmv(fmt, _p(w, ctypes.c_uint8), rows, cols,
                             _p(xq, ctypes.c_uint8), _p(y, ctypes.c_double),
                             _p(e, ctypes.c_double)), "dmmv")
    return y, e


def dmmv_xf32(fmt: int, w, rows: int, cols: int, x) -> tuple[np.ndarray, np.ndarray]:
    """W.x with x taken as fp32 values (no quantization): (y_ref, err_scale), float64 [rows]."""
    w = _u8(w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.size != cols:
        raise ValueError("dmmv_xf32: x must hold cols values")
    y = np.zeros(rows, dtype=np.float64)
    e = np.zeros(rows, dtype=np.float64)
    _check(lib().oracle_dmmv_xf32(fmt, _p(w, ctypes.c_uint8), rows, cols, _p(x, ctypes.c_float),
                                  _p(y, ctypes.c_double), _p(e, ctypes.c_double)), "dmmv_xf32")
    return y, e


def dmmv_batched(fmt: int, w, rows: int, cols: int, xq, batch: int):
    w, xq = _u8(w), _u8(xq)
    y = np.zeros((batch, rows), dtype=np.float64)
    e = np.zeros((batch, rows), dtype=np.float64)
    _check(lib().oracle_dmmv_batched(fmt, _p(w, ctypes.c_uint8), rows, cols,
                                     _p(xq, ctypes.c_uint8), batch,
                                     _p(y, ctypes.c_double), _p(e, ctypes.c_double)),
           "dmmv_batched")
    return y, e


def expert_gather(fmt: int, w_stack, expert_stride: int, rows: int, cols: int, idx,
                  n_experts: int, xq, xq_stride: int):
    """Returns (y [n][rows], err_scale [n][rows], status)."""
    w_stack, xq = _u8(w_stack), _u8(xq)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    n = idx.size
    y = np.zeros((n, rows), dtype=np.float64)
    e = np.zeros((n, rows), dtype=np.float64)
    st = ctypes.c_int32(0)
    _check(lib().oracle_expert_gather(fmt, _p(w_stack, ctypes.c_uint8), expert_stride,
                                      rows, cols, _p(idx, ctypes.c_int32), n, n_experts,
                                      _p(xq, ctypes.c_uint8), xq_stride,
                                      _p(y, ctypes.c_double), _p(e, ctypes.c_double),
                                      ctypes.byref(st)), "expert_gather")
    return y, e, int(st.value)


def dmmv_acc(fmt: int, w, rows: int, cols: int, xq, y0, gate=None):
    """Returns (y0 + s * W.x, s * err_scale), s = sigmoid(gate) or 1."""
    w, xq = _u8(w), _u8(xq)
    y = np.array(y0, dtype=np.float64).reshape(-1).copy()
    e = np.zeros(rows, dtype=np.float64)
    g = None if gate is None else ctypes.byref(ctypes.c_double(float(gate)))
    _check(lib().oracle_dmmv_acc(fmt, _p(w, ctypes.c_uint8), rows, cols, _p(xq, ctypes.c_uint8), g,
                                 _p(y, ctypes.c_double), _p(e, ctypes.c_double)), "dmmv_acc")
    return y, e


def swiglu(g, u) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64).reshape(-1)
    u = np.ascontiguousarray(u, dtype=np.float64).reshape(-1)
    h = np.zeros_like(g)
    lib().oracle_swiglu(_p(g, ctypes.c_double), _p(u, ctypes.c_double), g.size, _p(h, ctypes.c_double))
    return h


def argmax(y) -> tuple[int, float]:
    """(first index of the maximum, the maximum)."""
    y = np.ascontiguousarray(y, dtype=np.float64).reshape(-1)
    m = ctypes.c_double(0.0)
    i = lib().oracle_argmax(_p(y, ctypes.c_double), y.size, ctypes.byref(m))
    return int(i), float(m.value)


def repack(fmt: int, src, rows: int, cols: int) -> np.ndarray:
    src = _u8(src)
    dst = np.zeros(rows * (cols // 32) * BLOCK_BYTES[fmt], dtype=np.uint8)
    _check(lib().oracle_repack(fmt, _p(src, ctypes.c_uint8), rows, cols,
                               _p(dst, ctypes.c_uint8)), "repack")
    return dst


def unpack(fmt: int, src, rows: int, cols: int) -> np.ndarray:
    src = _u8(src)
    dst = np.zeros(rows * (cols // 32) * BLOCK_BYTES[fmt], dtype=np.uint8)
    _check(lib().oracle_unpack(fmt, _p(src, ctypes.c_uint8), rows, cols,
                               _p(dst, ctypes.c_uint8)), "unpack")
    return dst


def within_tolerance(y, y_ref, err_scale, rel: float = 1e-5, abs_: float = 1e-6):
    """The pass criterion |y - y_ref| <= rel * sum_b |d_w d_x s_b| + abs, per row.
    Returns (ok, worst_ratio) where worst_ratio = max |y-y_ref| / bound."""
    y = np.asarray(y, dtype=np.float64)
    bound = rel * np.asarray(err_scale, dtype=np.float64) + abs_
    diff = np.abs(y - np.asarray(y_ref, dtype=np.float64))
    ratio = diff / bound
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(diff <= bound)), worst
