"""CPU oracle for row-wise ArgMax / ArgMin (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product (``row_wise_arg_gb300``) never does;
the two share no code.

The arithmetic lives in ``argreduce_oracle.c``: a plain sequential scan per
row that seeds the candidate with element 0 and replaces it only on a strictly
better value (onnxruntime PRs #32092 "Semantics" and #31694 "Semantics"); the
"max_last" / "min_last" ops replace it on a value that is not worse, which
makes ties go to the last index (ONNX select_last_index = 1).
This module compiles that file with the host C compiler and calls it through
ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "argreduce_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2, "f64": 3, "i32": 4, "i64": 5}
OP_CODE = {"max": 0, "min": 1, "max_last": 2, "min_last": 3}
RAW_NP = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "f64": np.float64, "i32": np.int32,
          "i64": np.int64}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (no fast-math: NaN and
    signed-zero comparisons must follow IEEE 754)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_argreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int, i64p, ctypes.c_void_p]
            lib.oracle_argreduce.restype = ctypes.c_int
            lib.oracle_argreduce_mt.argtypes = lib.oracle_argreduce.argtypes + [ctypes.c_int]
            lib.oracle_argreduce_mt.restype = ctypes.c_int
            lib.oracle_argreduce_axis.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int, i64p, ctypes.c_void_p]
            lib.oracle_argreduce_axis.restype = ctypes.c_int
            lib.oracle_cumreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int, i64p, ctypes.c_void_p]
            lib.oracle_cumreduce.restype = ctypes.c_int
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_f16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            _lib = lib
    return _lib


def argreduce(x: np.ndarray, dtype: str, op: str, threads: int = 1,
              want_val: bool = True) -> Tuple[np.ndarray, Optional[np.ndarray], int]:
    """Reduce each row of the 2-D raw array ``x`` (see ``workloads`` for the
    raw encodings). Returns ``(idx int64[rows], val raw[rows] or None,
    threads_used)``."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    if x.dtype != RAW_NP[dtype]:
        raise TypeError(f"{dtype} expects raw numpy dtype {RAW_NP[dtype]}, got {x.dtype}")
    rows, cols = x.shape
    idx = np.empty(rows, dtype=np.int64)
    val = np.empty(rows, dtype=x.dtype) if want_val else None
    args = (x.ctypes.data_as(ctypes.c_void_p), DTYPE_CODE[dtype], rows, cols, OP_CODE[op],
            idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            val.ctypes.data_as(ctypes.c_void_p) if val is not None else None)
    if threads <= 1:
        rc = lib.oracle_argreduce(*args)
        used = 1
    else:
        rc = used = lib.oracle_argreduce_mt(*args, threads)
    if rc < 0:
        raise ValueError(f"oracle rejected arguments: rows={rows} cols={cols} dtype={dtype} op={op}")
    return idx, val, used


def argreduce_axis(x: np.ndarray, dtype: str, op: str, want_val: bool = True):
    """Reduce the middle axis of the 3-D raw array ``x[outer, R, inner]``.
    Returns ``(idx int64[outer, inner], val raw[outer, inner] or None)``."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.ndim != 3:
        raise ValueError("x must be 3-D [outer, R, inner]")
    if x.dtype != RAW_NP[dtype]:
        raise TypeError(f"{dtype} expects raw numpy dtype {RAW_NP[dtype]}, got {x.dtype}")
    outer, R, inner = x.shape
    idx = np.empty((outer, inner), dtype=np.int64)
    val = np.empty((outer, inner), dtype=x.dtype) if want_val else None
    rc = lib.oracle_argreduce_axis(x.ctypes.data_as(ctypes.c_void_p), DTYPE_CODE[dtype], outer, R, inner,
                                   OP_CODE[op], idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   val.ctypes.data_as(ctypes.c_void_p) if val is not None else None)
    if rc < 0:
        raise ValueError(f"oracle rejected arguments: shape={x.shape} dtype={dtype} op={op}")
    return idx, val


def cumreduce(x: np.ndarray, dtype: str, op: str, want_val: bool = True):
    """cummax ("max") / cummin ("min") with indices along the last axis of the
    2-D raw array ``x``: for every prefix x[r, 0..j], the ArgMax (ArgMin) of
    that prefix (ties to the earlier index). Returns ``(idx int64[rows, cols],
    val raw[rows, cols] or None)``."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    if x.dtype != RAW_NP[dtype]:
        raise TypeError(f"{dtype} expects raw numpy dtype {RAW_NP[dtype]}, got {x.dtype}")
    rows, cols = x.shape
    idx = np.empty((rows, cols), dtype=np.int64)
    val = np.empty((rows, cols), dtype=x.dtype) if want_val else None
    rc = lib.oracle_cumreduce(x.ctypes.data_as(ctypes.c_void_p), DTYPE_CODE[dtype], rows, cols, OP_CODE[op],
                              idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                              val.ctypes.data_as(ctypes.c_void_p) if val is not None else None)
    if rc < 0:
        raise ValueError(f"oracle rejected arguments: shape={x.shape} dtype={dtype} op={op}")
    return idx, val


def decode_f16(bits: int) -> float:
    return _load().oracle_decode_f16(bits)


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)
