"""ctypes wrapper of the plain C oracle (tq_ref.c).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg may import this package. The CUDA path never calls it, and it
never calls the CUDA path.

The shared library is built with gcc from tq_ref.c on first use (or by
build()): -O2, no fast-math, no floating-point contraction, so that the
quantizer's single IEEE division, multiplication and round-to-nearest-even
are exactly what the source says.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_ref.c")
_HDR = os.path.join(_HERE, "tq_ref.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libtq_ref.so")

QK_K = 256
GROUP = 128
PQ2_BYTES = 34
Q8K_BYTES = 292

# numpy view of one q8_K block, matching ref_block_q8K
Q8K_DTYPE = np.dtype([("d", "<f4"), ("qs", "i1", (256,)), ("bsums", "<i2", (16,))])
assert Q8K_DTYPE.itemsize == Q8K_BYTES

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile tq_ref.c into a shared library; returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-Wall", "-Wextra",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64 = ctypes.c_void_p, ctypes.c_int64
            lib.ref_fp16_to_f32.argtypes = [ctypes.c_uint16]
            lib.ref_fp16_to_f32.restype = ctypes.c_float
            lib.ref_quantize_q8K.argtypes = [P, I64, I64, P]
            lib.ref_decode_pq2_0.argtypes = [P, I64, I64, P, P]
            lib.ref_repacked_bytes.argtypes = [I64, I64]
            lib.ref_repacked_bytes.restype = I64
            lib.ref_repack.argtypes = [P, I64, I64, P]
            lib.ref_unrepack.argtypes = [P, I64, I64, P]
            lib.ref_groupsums.argtypes = [P, P, I64, I64, I64, P]
            lib.ref_matmul.argtypes = [P, P, I64, I64, I64, P, P]
            for f in ("ref_quantize_q8K", "ref_decode_pq2_0", "ref_repack",
                      "ref_unrepack", "ref_groupsums", "ref_matmul"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def fp16_to_f32(bits: int) -> float:
    return _load().ref_fp16_to_f32(int(bits) & 0xFFFF)


def quantize_q8K(x: np.ndarray) -> np.ndarray:
    """x f32 [ntok][cols] -> structured q8_K array [ntok][cols/256]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    ntok, cols = x.shape
    assert cols % QK_K == 0
    out = np.zeros((ntok, cols // QK_K), dtype=Q8K_DTYPE)
    _load().ref_quantize_q8K(_ptr(x), ntok, cols, _ptr(out))
    return out


def decode_pq2_0(wpq: np.ndarray, rows: int, cols: int):
    """pq2_0 bytes -> (ternary int8 w[rows][cols], fp16 scale bits[rows][cols/128])."""
    wpq = np.ascontiguousarray(wpq, dtype=np.uint8)
    assert wpq.size == rows * cols // GROUP * PQ2_BYTES
    w = np.empty((rows, cols), dtype=np.int8)
    sb = np.empty((rows, cols // GROUP), dtype=np.uint16)
    _load().ref_decode_pq2_0(_ptr(wpq), rows, cols, _ptr(w), _ptr(sb))
    return w, sb


def repacked_bytes(rows: int, cols: int) -> int:
    return int(_load().ref_repacked_bytes(rows, cols))


def repack(wpq: np.ndarray, rows: int, cols: int) -> np.ndarray:
    wpq = np.ascontiguousarray(wpq, dtype=np.uint8)
    assert wpq.size == rows * cols // GROUP * PQ2_BYTES
    out = np.empty(repacked_bytes(rows, cols), dtype=np.uint8)
    _load().ref_repack(_ptr(wpq), rows, cols, _ptr(out))
    return out


def unrepack(wtq: np.ndarray, rows: int, cols: int) -> np.ndarray:
    wtq = np.ascontiguousarray(wtq, dtype=np.uint8)
    assert wtq.size == repacked_bytes(rows, cols)
    out = np.empty(rows * cols // GROUP * PQ2_BYTES, dtype=np.uint8)
    _load().ref_unrepack(_ptr(wtq), rows, cols, _ptr(out))
    return out


def groupsums(wpq: np.ndarray, xq: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """int32 S[ntok][rows][cols/128]."""
    wpq = np.ascontiguousarray(wpq, dtype=np.uint8)
    xq = np.ascontiguousarray(xq)
    assert xq.dtype == Q8K_DTYPE and xq.shape[1] == cols // QK_K
    ntok = xq.shape[0]
    S = np.empty((ntok, rows, cols // GROUP), dtype=np.int32)
    _load().ref_groupsums(_ptr(wpq), _ptr(xq), rows, cols, ntok, _ptr(S))
    return S


def matmul(wpq: np.ndarray, xq: np.ndarray, rows: int, cols: int):
    """(y f32 [ntok][rows], abs_sum f64 [ntok][rows])."""
    wpq = np.ascontiguousarray(wpq, dtype=np.uint8)
    xq = np.ascontiguousarray(xq)
    assert xq.dtype == Q8K_DTYPE and xq.shape[1] == cols // QK_K
    ntok = xq.shape[0]
    y = np.empty((ntok, rows), dtype=np.float32)
    a = np.empty((ntok, rows), dtype=np.float64)
    _load().ref_matmul(_ptr(wpq), _ptr(xq), rows, cols, ntok, _ptr(y), _ptr(a))
    return y, a


def pq2_0_rows(wpq: np.ndarray, cols: int, row_ids) -> np.ndarray:
    """Gather whole pq2_0 rows (each row is cols/128 contiguous blocks)."""
    per_row = cols // GROUP * PQ2_BYTES
    w2 = np.asarray(wpq, dtype=np.uint8).reshape(-1, per_row)
    return np.ascontiguousarray(w2[np.asarray(row_ids)]).reshape(-1)
