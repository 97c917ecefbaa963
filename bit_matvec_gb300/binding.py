"""ctypes binding of libtq.so: the C ABI of include/tq.h under the same names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. Tensors must be CUDA tensors of the current device
(or of the device given by the first tensor argument, which is made current
for the call); sizes are passed through unchanged, and the library's status
codes become TQError. There is no CPU fallback: if libtq.so is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "tq.h")

TQ_OK = 0
TQ_ERR_SHAPE = -1
TQ_ERR_NULL = -2
TQ_ERR_ALIGN = -3
TQ_ERR_CUDA = -4
TQ_ERR_TIMEOUT = -5
TQ_ERR_ALIAS = -6
TQ_ERR_WORKSPACE = -7

QK_K = 256
GROUP = 128
PQ2_0_BYTES = 34
PTQ1_0_BYTES = 28
Q8K_BYTES = 292
TILE_ROWS = 32
TILE_BYTES = 1088
STATIC_WS_BYTES = 8 << 20   # TQ_STATIC_WS_BYTES: fixed workspace of tq_matmul_static_ws

_lock = threading.Lock()
_lib = None


class TQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        lib = _load()
        msg = lib.tq_strerror(code).decode()
        if code == TQ_ERR_CUDA:
            msg += f" (cudaError {lib.tq_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [{code}]")


def header_functions() -> list[str]:
    """Names of the functions include/tq.h declares."""
    with open(HEADER) as f:
        src = f.read()
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tq_\w+)\s*\(", src, flags=re.M)


def _load():
    global _lib
    if _lib is not None:   # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m bit_matvec_gb300.build, or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sig = {
            "tq_quantize_q8K": ([P, P, I64, I64, P], I),
            "tq_repacked_bytes": ([I64, I64], I64),
            "tq_repack": ([P, P, I64, I64, P], I),
            "tq_unrepack": ([P, P, I64, I64, P], I),
            "tq_ptq1_0_bytes": ([I64, I64], I64),
            "tq_repack_ptq1_0": ([P, P, I64, I64, P], I),
            "tq_matmul": ([P, P, P, I64, I64, I64, P], I),
            "tq_matmul_groupsums": ([P, P, P, I64, I64, I64, P], I),
            "tq_matmul_workspace_bytes": ([I64, I64, I64], I64),
            "tq_matmul_ws": ([P, P, P, I64, I64, I64, P, I64, P], I),
            "tq_matmul_groupsums_ws": ([P, P, P, I64, I64, I64, P, I64, P], I),
            "tq_matmul_static_ws": ([P, P, P, I64, I64, I64, P], I),
            "tq_matmul_host": ([P, P, P, P, P, P, I64, I64, I64, P, I64, P], I),
            "tq_quantize_matmul": ([P, P, P, P, I64, I64, I64, P, I64, P], I),
            "tq_strerror": ([I], ctypes.c_char_p),
            "tq_last_cuda_error": ([], I),
            "tq_device_status": ([], I),
            "tq_version": ([], ctypes.c_char_p),
            "tq_debug_stall_next_launch": ([I64], I),
            "tq_probe_read_sum": ([P, I64, P, I, P], I),
            "tq_ptq1_0_stream_bytes": ([I64, I64], I64),
            "tq_repack_ptq1_0_stream": ([P, P, I64, I64, P], I),
            "tq_matmul_ptq1_0_stream": ([P, P, P, I64, I64, I64, P], I),
            "tq_matmul_ptq1_0_stream_groupsums": ([P, P, P, I64, I64, I64, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def library() -> ctypes.CDLL:
    """The loaded libtq.so (raises if it has not been built)."""
    return _load()


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()   # an int; the declared argtypes make it a void*


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _call(name, device, *args):
    lib = _load()
    if device.index is None or device.index == torch.cuda.current_device():
        rc = getattr(lib, name)(*args)
    else:
        with torch.cuda.device(device):
            rc = getattr(lib, name)(*args)
    if rc != TQ_OK:
        raise TQError(rc, name)


# ---------------------------------------------------------------- allocation helpers

def q8K_nbytes(ntok: int, cols: int) -> int:
    return ntok * (cols // QK_K) * Q8K_BYTES


def q8K_empty(ntok: int, cols: int, device="cuda") -> torch.Tensor:
    """uint8 buffer for ntok x cols/256 q8_K blocks."""
    return torch.empty(q8K_nbytes(ntok, cols), dtype=torch.uint8, device=device)


def tq_repacked_bytes(rows: int, cols: int) -> int:
    n = _load().tq_repacked_bytes(rows, cols)
    if n < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_repacked_bytes")
    return int(n)


def repacked_empty(rows: int, cols: int, device="cuda") -> torch.Tensor:
    return torch.empty(tq_repacked_bytes(rows, cols), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- the C ABI

def tq_quantize_q8K(X: torch.Tensor, Xq: torch.Tensor, ntok: int, cols: int, stream=None):
    _call("tq_quantize_q8K", X.device, _ptr(X), _ptr(Xq), ntok, cols, _stream(stream, X.device))


def tq_repack(Wpq2: torch.Tensor, Wtq: torch.Tensor, rows: int, cols: int, stream=None):
    _call("tq_repack", Wpq2.device, _ptr(Wpq2), _ptr(Wtq), rows, cols,
          _stream(stream, Wpq2.device))


def tq_unrepack(Wtq: torch.Tensor, Wpq2: torch.Tensor, rows: int, cols: int, stream=None):
    _call("tq_unrepack", Wtq.device, _ptr(Wtq), _ptr(Wpq2), rows, cols,
          _stream(stream, Wtq.device))


def tq_ptq1_0_bytes(rows: int, cols: int) -> int:
    n = _load().tq_ptq1_0_bytes(rows, cols)
    if n < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_ptq1_0_bytes")
    return int(n)


def tq_repack_ptq1_0(Wpt: torch.Tensor, Wtq: torch.Tensor, rows: int, cols: int, stream=None):
    """ptq1_0 (1.75-bit) weights -> the tq layout, decoded once at load."""
    _call("tq_repack_ptq1_0", Wpt.device, _ptr(Wpt), _ptr(Wtq), rows, cols,
          _stream(stream, Wpt.device))


def tq_ptq1_0_stream_bytes(rows: int, cols: int) -> int:
    n = _load().tq_ptq1_0_stream_bytes(rows, cols)
    if n < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_ptq1_0_stream_bytes")
    return int(n)


def tq_repack_ptq1_0_stream(Wpt: torch.Tensor, Wt1: torch.Tensor, rows: int, cols: int,
                            stream=None):
    """ptq1_0 (1.75-bit) weights -> 32-row stream tiles, not decoded."""
    _call("tq_repack_ptq1_0_stream", Wpt.device, _ptr(Wpt), _ptr(Wt1), rows, cols,
          _stream(stream, Wpt.device))


def tq_matmul_ptq1_0_stream(Wt1: torch.Tensor, Xq: torch.Tensor, Y: torch.Tensor, rows: int,
                            cols: int, ntok: int, stream=None):
    _call("tq_matmul_ptq1_0_stream", Wt1.device, _ptr(Wt1), _ptr(Xq), _ptr(Y), rows, cols, ntok,
          _stream(stream, Wt1.device))


def tq_matmul_ptq1_0_stream_groupsums(Wt1: torch.Tensor, Xq: torch.Tensor, S: torch.Tensor,
                                      rows: int, cols: int, ntok: int, stream=None):
    _call("tq_matmul_ptq1_0_stream_groupsums", Wt1.device, _ptr(Wt1), _ptr(Xq), _ptr(S), rows,
          cols, ntok, _stream(stream, Wt1.device))


def tq_matmul(Wtq: torch.Tensor, Xq: torch.Tensor, Y: torch.Tensor, rows: int, cols: int,
              ntok: int, stream=None):
    _call("tq_matmul", Wtq.device, _ptr(Wtq), _ptr(Xq), _ptr(Y), rows, cols, ntok,
          _stream(stream, Wtq.device))


def tq_matmul_groupsums(Wtq: torch.Tensor, Xq: torch.Tensor, S: torch.Tensor, rows: int,
                        cols: int, ntok: int, stream=None):
    _call("tq_matmul_groupsums", Wtq.device, _ptr(Wtq), _ptr(Xq), _ptr(S), rows, cols, ntok,
          _stream(stream, Wtq.device))


def tq_matmul_workspace_bytes(rows: int, cols: int, ntok: int) -> int:
    n = _load().tq_matmul_workspace_bytes(rows, cols, ntok)
    if n < 0:
        raise TQError(TQ_ERR_SHAPE, "tq_matmul_workspace_bytes")
    return int(n)


def workspace_empty(rows: int, cols: int, ntok: int, device="cuda") -> torch.Tensor:
    """uint8 buffer for tq_matmul_ws (at least one byte, so it has an address)."""
    return torch.empty(max(1, tq_matmul_workspace_bytes(rows, cols, ntok)), dtype=torch.uint8,
                       device=device)


def tq_matmul_ws(Wtq: torch.Tensor, Xq: torch.Tensor, Y: torch.Tensor, rows: int, cols: int,
                 ntok: int, workspace: torch.Tensor, stream=None):
    _call("tq_matmul_ws", Wtq.device, _ptr(Wtq), _ptr(Xq), _ptr(Y), rows, cols, ntok,
          _ptr(workspace), workspace.numel(), _stream(stream, Wtq.device))


def tq_matmul_groupsums_ws(Wtq: torch.Tensor, Xq: torch.Tensor, S: torch.Tensor, rows: int,
                           cols: int, ntok: int, workspace: torch.Tensor, stream=None):
    _call("tq_matmul_groupsums_ws", Wtq.device, _ptr(Wtq), _ptr(Xq), _ptr(S), rows, cols, ntok,
          _ptr(workspace), workspace.numel(), _stream(stream, Wtq.device))


def tq_matmul_static_ws(Wtq: torch.Tensor, Xq: torch.Tensor, Y: torch.Tensor, rows: int,
                        cols: int, ntok: int, stream=None):
    """tq_matmul_ws with the library's fixed STATIC_WS_BYTES device array as
    its workspace, for callers that cannot allocate device memory. Calls share
    that array: calls that overlap on the GPU race, so keep them ordered."""
    _call("tq_matmul_static_ws", Wtq.device, _ptr(Wtq), _ptr(Xq), _ptr(Y), rows, cols, ntok,
          _stream(stream, Wtq.device))


def tq_quantize_matmul(Wtq: torch.Tensor, X: torch.Tensor, Xq: torch.Tensor, Y: torch.Tensor,
                       rows: int, cols: int, ntok: int, workspace: torch.Tensor, stream=None):
    """Xq = q8_K(X) and Y = Wtq x Xq in one call (one fused launch up to 3 tokens; from 4 to
    8, where the workspace size is not 0, a staging kernel and the GEMV)."""
    _call("tq_quantize_matmul", Wtq.device, _ptr(Wtq), _ptr(X), _ptr(Xq), _ptr(Y), rows, cols,
          ntok, _ptr(workspace), workspace.numel(), _stream(stream, Wtq.device))


def _host_ptr(t: torch.Tensor):
    if t.is_cuda:
        raise ValueError("tensor must live in host memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def tq_matmul_host(Wtq: torch.Tensor, X_host: torch.Tensor, X: torch.Tensor, Xq: torch.Tensor,
                   Y: torch.Tensor, Y_host: torch.Tensor, rows: int, cols: int, ntok: int,
                   workspace: torch.Tensor, stream=None):
    """Host f32 activations in, host f32 outputs out, in one enqueued step (copy
    in, quantize, matmul, copy out); X_host and Y_host should be pinned. Returns
    at once: synchronize the stream before reading Y_host."""
    _call("tq_matmul_host", Wtq.device, _ptr(Wtq), _host_ptr(X_host), _ptr(X), _ptr(Xq), _ptr(Y),
          _host_ptr(Y_host), rows, cols, ntok, _ptr(workspace), workspace.numel(),
          _stream(stream, Wtq.device))


def tq_strerror(code: int) -> str:
    return _load().tq_strerror(code).decode()


def tq_last_cuda_error() -> int:
    return int(_load().tq_last_cuda_error())


def tq_device_status(device=None) -> int:
    """Read and clear the device status word (synchronizes the device)."""
    lib = _load()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(lib.tq_device_status())


def tq_probe_read_sum(buf: torch.Tensor, out: torch.Tensor, early: bool = False, stream=None):
    """Adds buf's 32-bit words (mod 2^32) to out[0] (an int32 tensor) with the
    read-ceiling probe kernel: one streaming pass over buf and nothing else."""
    _call("tq_probe_read_sum", buf.device, _ptr(buf), buf.numel() * buf.element_size(), _ptr(out),
          1 if early else 0, _stream(stream, buf.device))


def tq_debug_stall_next_launch(wait_limit_ns: int):
    """Test facility: the next matmul kernel's first thread block requests no
    input copies, so its waits expire after wait_limit_ns and it reports
    TQ_ERR_TIMEOUT through tq_device_status (0 cancels)."""
    rc = _load().tq_debug_stall_next_launch(wait_limit_ns)
    if rc != TQ_OK:
        raise TQError(rc, "tq_debug_stall_next_launch")


def tq_version() -> str:
    return _load().tq_version().decode()
