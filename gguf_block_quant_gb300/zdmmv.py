"""Thin Python binding of libzdmmv.so (the C ABI declared in include/zdmmv.h).

Argument marshalling only: every function passes device pointers
(``tensor.data_ptr()``), sizes and the current CUDA stream to the C entry point
of the same name and raises ``ZdmmvError`` on a non-OK status. All arithmetic
runs in the CUDA kernels; there is no CPU fallback, and loading fails loudly if
the library cannot be built or found.

torch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import re
import threading

import torch

from . import _build

Q4_0 = 2
Q8_0 = 8
GGUF = 0
REPACKED = 1
QK = 32
MAX_BATCH = 8
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34}
FAULT_WAIT_TIMEOUT = 1
FAULT_SMEM_ALIGN = 2
ARGMAX_WORKSPACE_BYTES = 16384

STATUS = {0: "ok", 1: "null pointer", 2: "bad shape", 3: "misaligned pointer or stride",
          4: "unknown layout", 5: "unknown block format", 6: "buffer too small",
          7: "CUDA runtime error", 8: "device fault reported"}


class ZdmmvError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_SIGS = {
    "zdmmv_status_str": ([_int], ctypes.c_char_p),
    "zdmmv_version": ([], ctypes.c_char_p),
    "zdmmv_block_bytes": ([_int], ctypes.c_size_t),
    "zdmmv_quantize_act_q8_0": ([_vp, _i64, _vp, _vp], _int),
    "zdmmv_q8_0": ([_vp, _int, _i64, _i64, _vp, _vp, _vp], _int),
    "zdmmv_q4_0": ([_vp, _int, _i64, _i64, _vp, _vp, _vp], _int),
    "zdmmv_q8_0_batched": ([_vp, _int, _i64, _i64, _vp, _int, _vp, _vp], _int),
    "zdmmv_q4_0_batched": ([_vp, _int, _i64, _i64, _vp, _int, _vp, _vp], _int),
    "zdmmv_dmmv_f32": ([_int, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp], _int),
    "zdmmv_dmmv_xf32": ([_int, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp], _int),
    "zdmmv_dmmv_acc": ([_int, _vp, _int, _i64, _i64, _vp, _vp, _vp, _vp], _int),
    "zdmmv_dmmv_argmax": ([_int, _vp, _int, _i64, _i64, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp], _int),
    "zdmmv_dmmv_argmax_noalloc": ([_int, _vp, _int, _i64, _i64, _vp, _vp, _vp, _vp], _int),
    "zdmmv_expert_gather": ([_int, _vp, _i64, _int, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp, _vp, _vp],
                            _int),
    "zdmmv_expert_gather_ready": ([_int, _vp, _i64, _int, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp, _vp,
                                   _vp], _int),
    "zdmmv_expert_gather_f32": ([_int, _vp, _i64, _int, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp, _vp,
                                 _int, _vp], _int),
    "zdmmv_expert_gather2": ([_int, _vp, _vp, _i64, _int, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp, _vp,
                              _vp, _vp], _int),
    "zdmmv_expert_swiglu": ([_int, _vp, _vp, _i64, _int, _i64, _i64, _vp, _int, _int, _vp, _i64, _vp, _vp,
                             _vp], _int),
    "zdmmv_expert_ffn_workspace_bytes": ([_int, _i64], ctypes.c_size_t),
    "zdmmv_expert_ffn": ([_int, _vp, _vp, _i64, _int, _vp, _i64, _i64, _i64, _vp, _int, _int, _vp, _vp, _vp,
                          ctypes.c_size_t, _vp, _vp], _int),
    "zdmmv_repacked_bytes": ([_int, _i64, _i64], ctypes.c_size_t),
    "zdmmv_repack": ([_int, _vp, _i64, _i64, _vp, ctypes.c_size_t, _vp], _int),
    "zdmmv_host_step_workspace_bytes": ([_i64, _i64, _int], ctypes.c_size_t),
    "zdmmv_host_step": ([_int, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp, ctypes.c_size_t, _vp], _int),
    "zdmmv_debug_block_sums": ([_int, _vp, _int, _i64, _i64, _vp, _vp, _vp], _int),
    "zdmmv_selftest_dp4a": ([_vp, _vp, _vp, _vp, _int, _vp], _int),
    "zdmmv_selftest_wait_timeout": ([_vp, _vp], _int),
    "zdmmv_device_status": ([ctypes.POINTER(ctypes.c_uint32), _int], _int),
}


def library_path() -> str:
    return _build.LIB


def lib(build: bool = True) -> ctypes.CDLL:
    """Load libzdmmv.so (building it first if it is stale) and declare its ABI."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/zdmmv.h."""
    import os
    hdr = os.path.join(_build.INCLUDE, "zdmmv.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zdmmv_[a-z0-9_]+)\s*\(", text)))


def _call(name: str, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise ZdmmvError(name, rc)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("zdmmv: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("zdmmv: expected a contiguous tensor")
    return t.data_ptr()


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


# ---------------------------------------------------------------- entry points
def quantize_act_q8_0(x: torch.Tensor, xq: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp32 activations (any shape, numel % 32 == 0) -> uint8 Q8_0 blocks."""
    k = x.numel()
    if x.dtype != torch.float32:
        raise ValueError("quantize_act_q8_0: x must be float32")
    if xq is None:
        xq = torch.empty(k // QK * 34, dtype=torch.uint8, device=x.device)
    elif _nbytes(xq) < k // QK * 34:
        raise ValueError("quantize_act_q8_0: xq too small")
    _call("zdmmv_quantize_act_q8_0", _ptr(x), k, _ptr(xq), _stream(stream))
    return xq


def _out(y, shape, device):
    if y is None:
        return torch.empty(shape, dtype=torch.float32, device=device)
    if y.dtype != torch.float32 or y.numel() < int(torch.tensor(shape).prod()):
        raise ValueError("output must be float32 with enough elements")
    return y


def q8_0(w, rows: int, cols: int, xq, y=None, layout: int = GGUF, stream=None):
    y = _out(y, (rows,), w.device)
    _call("zdmmv_q8_0", _ptr(w), layout, rows, cols, _ptr(xq), _ptr(y), _stream(stream))
    return y


def q4_0(w, rows: int, cols: int, xq, y=None, layout: int = GGUF, stream=None):
    y = _out(y, (rows,), w.device)
    _call("zdmmv_q4_0", _ptr(w), layout, rows, cols, _ptr(xq), _ptr(y), _stream(stream))
    return y


def q8_0_batched(w, rows: int, cols: int, xq, batch: int, y=None, layout: int = GGUF, stream=None):
    y = _out(y, (batch, rows), w.device)
    _call("zdmmv_q8_0_batched", _ptr(w), layout, rows, cols, _ptr(xq), batch, _ptr(y), _stream(stream))
    return y


def q4_0_batched(w, rows: int, cols: int, xq, batch: int, y=None, layout: int = GGUF, stream=None):
    y = _out(y, (batch, rows), w.device)
    _call("zdmmv_q4_0_batched", _ptr(w), layout, rows, cols, _ptr(xq), batch, _ptr(y), _stream(stream))
    return y


def dmmv(fmt: int, w, rows: int, cols: int, xq, y=None, layout: int = GGUF, stream=None):
    return (q8_0 if fmt == Q8_0 else q4_0)(w, rows, cols, xq, y=y, layout=layout, stream=stream)


def dmmv_batched(fmt: int, w, rows: int, cols: int, xq, batch: int, y=None, layout: int = GGUF, stream=None):
    f = q8_0_batched if fmt == Q8_0 else q4_0_batched
    return f(w, rows, cols, xq, batch, y=y, layout=layout, stream=stream)


def dmmv_f32(fmt: int, w, rows: int, cols: int, x, batch: int = 1, y=None, layout: int = GGUF,
             stream=None):
    """Fused decode step: quantize the fp32 activation x ([batch][cols]) and run
    the DMMV in one launch; identical to quantize_act_q8_0 followed by dmmv."""
    if x.dtype != torch.float32 or x.numel() != batch * cols:
        raise ValueError("dmmv_f32: x must be float32 [batch][cols]")
    y = _out(y, (batch, rows) if batch > 1 else (rows,), w.device)
    _call("zdmmv_dmmv_f32", fmt, _ptr(w), layout, rows, cols, _ptr(x), batch, _ptr(y), _stream(stream))
    return y


def dmmv_xf32(fmt: int, w, rows: int, cols: int, x, batch: int = 1, y=None, layout: int = GGUF, stream=None):
    """W.x with the fp32 activation taken as is (no quantization); x fp32 [batch][cols]."""
    if x.dtype != torch.float32:
        raise ValueError("dmmv_xf32: x must be float32")
    y = _out(y, (batch, rows) if batch > 1 else (rows,), w.device)
    _call("zdmmv_dmmv_xf32", fmt, _ptr(w), layout, rows, cols, _ptr(x), batch, _ptr(y), _stream(stream))
    return y


def dmmv_acc(fmt: int, w, rows: int, cols: int, xq, y, gate=None, layout: int = GGUF, stream=None):
    """y += s * W.x in place, s = sigmoid(gate[0]) for a device gate scalar, else 1."""
    _call("zdmmv_dmmv_acc", fmt, _ptr(w), layout, rows, cols, _ptr(xq), _ptr(gate), _ptr(y), _stream(stream))
    return y


def dmmv_argmax(fmt: int, w, rows: int, cols: int, xq, workspace=None, out=None, max_out=None,
                layout: int = GGUF, stream=None):
    """Index (int32 device tensor [1]) of the largest of W.x, without writing W.x."""
    if workspace is None:
        workspace = torch.empty(ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device=w.device)
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=w.device)
    _call("zdmmv_dmmv_argmax", fmt, _ptr(w), layout, rows, cols, _ptr(xq), _ptr(out), _ptr(max_out),
          _ptr(workspace), _nbytes(workspace), _stream(stream))
    return out


def dmmv_argmax_noalloc(fmt: int, w, rows: int, cols: int, xq, out=None, max_out=None, layout: int = GGUF,
                        stream=None):
    """The argmax DMMV without a workspace: for callers that cannot allocate
    device memory (see include/zdmmv.h). Overlapping calls race."""
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=w.device)
    _call("zdmmv_dmmv_argmax_noalloc", fmt, _ptr(w), layout, rows, cols, _ptr(xq), _ptr(out), _ptr(max_out),
          _stream(stream))
    return out


def expert_gather(fmt: int, w_stack, expert_stride: int, rows: int, cols: int, idx, n_experts: int, xq,
                  xq_stride: int, y=None, status=None, layout: int = GGUF, stream=None, idx_ready: bool = False):
    """idx_ready=True calls zdmmv_expert_gather_ready: an earlier expert call on
    the stream has read the same final index list (see include/zdmmv.h)."""
    n = idx.numel()
    if idx.dtype != torch.int32:
        raise ValueError("expert_gather: idx must be int32")
    y = _out(y, (n, rows), w_stack.device)
    _call("zdmmv_expert_gather_ready" if idx_ready else "zdmmv_expert_gather", fmt, _ptr(w_stack), expert_stride,
          layout, rows, cols, _ptr(idx), n, n_experts, _ptr(xq), xq_stride, _ptr(y), _ptr(status), _stream(stream))
    return y


def expert_gather_f32(fmt: int, w_stack, expert_stride: int, rows: int, cols: int, idx, n_experts: int, x,
                      x_stride: int, y=None, status=None, layout: int = GGUF, stream=None, idx_ready: bool = False):
    """Gather over fp32 activations (slot k: x + k*x_stride floats), quantized in the launch."""
    n = idx.numel()
    if idx.dtype != torch.int32:
        raise ValueError("expert_gather_f32: idx must be int32")
    if x.dtype != torch.float32:
        raise ValueError("expert_gather_f32: x must be float32")
    y = _out(y, (n, rows), w_stack.device)
    _call("zdmmv_expert_gather_f32", fmt, _ptr(w_stack), expert_stride, layout, rows, cols, _ptr(idx), n,
          n_experts, _ptr(x), x_stride, _ptr(y), _ptr(status), 1 if idx_ready else 0, _stream(stream))
    return y


def expert_gather2(fmt: int, w_stack_a, w_stack_b, expert_stride: int, rows: int, cols: int, idx,
                   n_experts: int, xq, xq_stride: int, y_a=None, y_b=None, status=None, layout: int = GGUF,
                   stream=None):
    """Two same-shaped expert stacks (e.g. gate and up) in one launch."""
    n = idx.numel()
    if idx.dtype != torch.int32:
        raise ValueError("expert_gather2: idx must be int32")
    y_a = _out(y_a, (n, rows), w_stack_a.device)
    y_b = _out(y_b, (n, rows), w_stack_a.device)
    _call("zdmmv_expert_gather2", fmt, _ptr(w_stack_a), _ptr(w_stack_b), expert_stride, layout, rows, cols,
          _ptr(idx), n, n_experts, _ptr(xq), xq_stride, _ptr(y_a), _ptr(y_b), _ptr(status), _stream(stream))
    return y_a, y_b


def expert_swiglu(fmt: int, w_gate, w_up, rows: int, cols: int, xq, idx=None, expert_stride: int = 0,
                  n_experts: int = 0, xq_stride: int = 0, h=None, status=None, layout: int = GGUF, stream=None):
    """h[k] = silu(G_idx[k] . x_k) * (U_idx[k] . x_k) in one launch; idx=None: one gate/up pair."""
    if idx is not None and idx.dtype != torch.int32:
        raise ValueError("expert_swiglu: idx must be int32")
    n = 1 if idx is None else idx.numel()
    h = _out(h, (n, rows), w_gate.device)
    _call("zdmmv_expert_swiglu", fmt, _ptr(w_gate), _ptr(w_up), expert_stride, layout, rows, cols, _ptr(idx), n,
          n_experts, _ptr(xq), xq_stride, _ptr(h), _ptr(status), _stream(stream))
    return h


def expert_ffn_workspace(n: int, ffn: int, device="cuda"):
    """A zero-filled workspace for expert_ffn (reusable across calls on one stream)."""
    nbytes = lib().zdmmv_expert_ffn_workspace_bytes(n, ffn)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def expert_ffn(fmt_gate_up: int, w_gate, w_up, gate_up_stride: int, fmt_down: int, w_down, down_stride: int,
               hidden: int, ffn: int, idx, n_experts: int, xq, y=None, workspace=None, status=None, stream=None):
    """The selected experts' gate/up DMMVs, SwiGLU and down DMMV in one launch:
    y[k] = D_idx[k] . q8_0(silu(G_idx[k] . x) * (U_idx[k] . x)). Returns (y, h)."""
    if idx.dtype != torch.int32:
        raise ValueError("expert_ffn: idx must be int32")
    n = idx.numel()
    y = _out(y, (n, hidden), w_gate.device)
    if workspace is None:
        workspace = expert_ffn_workspace(n, ffn, w_gate.device)
    _call("zdmmv_expert_ffn", fmt_gate_up, _ptr(w_gate), _ptr(w_up), gate_up_stride, fmt_down, _ptr(w_down),
          down_stride, hidden, ffn, _ptr(idx), n, n_experts, _ptr(xq), _ptr(y), _ptr(workspace),
          _nbytes(workspace), _ptr(status), _stream(stream))
    h = workspace[: 4 * n * ffn].view(torch.float32).view(n, ffn)
    return y, h


def repacked_bytes(fmt: int, rows: int, cols: int) -> int:
    return int(lib().zdmmv_repacked_bytes(fmt, rows, cols))


def repack(fmt: int, src, rows: int, cols: int, dst=None, stream=None):
    need = repacked_bytes(fmt, rows, cols)
    if dst is None:
        dst = torch.empty(need, dtype=torch.uint8, device=src.device)
    _call("zdmmv_repack", fmt, _ptr(src), rows, cols, _ptr(dst), _nbytes(dst), _stream(stream))
    return dst


def host_step_workspace_bytes(rows: int, cols: int, batch: int = 1) -> int:
    return int(lib().zdmmv_host_step_workspace_bytes(rows, cols, batch))


def host_step(fmt: int, w, rows: int, cols: int, x_host: torch.Tensor, y_host: torch.Tensor, workspace,
              batch: int = 1, layout: int = GGUF, stream=None):
    """One decode step from host activations to host outputs (asynchronous on
    the stream; synchronize before reading y_host)."""
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("host_step: x_host and y_host must be host tensors")
    _call("zdmmv_host_step", fmt, _ptr(w), layout, rows, cols, x_host.data_ptr(), batch, y_host.data_ptr(),
          _ptr(workspace), _nbytes(workspace), _stream(stream))
    return y_host


def debug_block_sums(fmt: int, w, rows: int, cols: int, xq, sums=None, layout: int = GGUF, stream=None):
    if sums is None:
        sums = torch.empty((rows, cols // QK), dtype=torch.int32, device=w.device)
    _call("zdmmv_debug_block_sums", fmt, _ptr(w), layout, rows, cols, _ptr(xq), _ptr(sums), _stream(stream))
    return sums


def selftest_dp4a(a, b, c, out=None, stream=None):
    if out is None:
        out = torch.empty_like(a)
    _call("zdmmv_selftest_dp4a", _ptr(a), _ptr(b), _ptr(c), _ptr(out), a.numel(), _stream(stream))
    return out


def selftest_wait_timeout(result=None, stream=None):
    """Run the failure-path self-test (a wait that can never complete, bounded)."""
    if result is None:
        result = torch.zeros(1, dtype=torch.int32, device="cuda")
    _call("zdmmv_selftest_wait_timeout", _ptr(result), _stream(stream))
    return result


def device_status(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _call("zdmmv_device_status", ctypes.byref(v), 1 if clear else 0)
    return int(v.value)
