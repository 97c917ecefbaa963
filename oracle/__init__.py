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
PTQ1_BYTES = 28
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
            lib.ref_ptq1_trit.argtypes = [ctypes.c_uint8, ctypes.c_int]
            lib.ref_ptq1_trit.restype = ctypes.c_int
            lib.ref_ptq1_byte.argtypes = [P]
            lib.ref_ptq1_byte.restype = ctypes.c_uint8
            lib.ref_encode_ptq1_0.argtypes = [P, P, I64, I64, P]
            lib.ref_ptq1_0_to_pq2_0.argtypes = [P, I64, I64, P]
            lib.ref_groupsums.argtypes = [P, P, I64, I64, I64, P]
            lib.ref_matmul.argtypes = [P, P, I64, I64, I64, P, P]
            for f in ("ref_quantize_q8K", "ref_decode_pq2_0", "ref_repack",
                      "ref_unrepack", "ref_groupsums", "ref_matmul", "ref_encode_ptq1_0",
                      "ref_ptq1_0_to_pq2_0"):
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


def ptq1_trit(b: int, n: int) -> int:
    """Trit n (0..4) of a ptq1_0 code byte b: the code u in {0, 1, 2}."""
    return int(_load().ref_ptq1_trit(b & 0xFF, n))


def ptq1_byte(trits) -> int:
    """The ptq1_0 code byte of five trits (each 0, 1 or 2)."""
    t = np.ascontiguousarray(np.asarray(trits, dtype=np.int32))
    assert t.shape == (5,)
    return int(_load().ref_ptq1_byte(_ptr(t)))


def encode_ptq1_0(w: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Ternary w int8 [rows][cols] and fp16 scale bits [rows][cols/128] ->
    flat ptq1_0 bytes (28 per 128 weights)."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    rows, cols = w.shape
    sb = np.ascontiguousarray(scale_bits, dtype=np.uint16)
    assert cols % GROUP == 0 and sb.shape == (rows, cols // GROUP)
    out = np.empty(rows * cols // GROUP * PTQ1_BYTES, dtype=np.uint8)
    _load().ref_encode_ptq1_0(_ptr(w), _ptr(sb), rows, cols, _ptr(out))
    return out


def ptq1_0_to_pq2_0(wpt: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """ptq1_0 bytes -> pq2_0 bytes of the same weights and scales."""
    wpt = np.ascontiguousarray(wpt, dtype=np.uint8)
    assert wpt.size == rows * cols // GROUP * PTQ1_BYTES
    out = np.empty(rows * cols // GROUP * PQ2_BYTES, dtype=np.uint8)
    _load().ref_ptq1_0_to_pq2_0(_ptr(wpt), rows, cols, _ptr(out))
    return out


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
