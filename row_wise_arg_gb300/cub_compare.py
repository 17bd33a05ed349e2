"""cub::DeviceReduce::ArgMax / ArgMin on one row, called as a library through
``libcubcompare.so`` (built by ``row_wise_arg_gb300.build``), for timing
comparisons only: the benchmark times it on the same inputs and in the same
way as argreduce(), and one GPU test checks that it finds the same indices on
NaN-free rows. It is not part of the argreduce API."""
from __future__ import annotations

import ctypes
import os

from ._lib import DTYPE_CODES, PKG

LIB_PATH = os.path.join(PKG, "libcubcompare.so")
OPS = {"max": 0, "min": 1}
_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with python -m row_wise_arg_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        lib.cubcmp_temp_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64]
        lib.cubcmp_temp_bytes.restype = ctypes.c_size_t
        lib.cubcmp_argreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        lib.cubcmp_argreduce.restype = ctypes.c_int
        _lib = lib
    return _lib


def temp_bytes(dtype: str, op: str, n: int) -> int:
    """Device temporary storage CUB needs for one row of n elements."""
    b = load().cubcmp_temp_bytes(DTYPE_CODES[dtype], OPS[op], n)
    if b == 0:
        raise ValueError(f"CUB rejected dtype={dtype} op={op} n={n}")
    return int(b)


def argreduce_raw(x_ptr: int, dtype: str, op: str, n: int, val_ptr: int, idx_ptr: int, temp_ptr: int,
                  temp_nbytes: int, stream_ptr: int) -> None:
    """Launch CUB's ArgMax/ArgMin of x[0..n) on the stream: the extremum into
    val_ptr, its int64 index into idx_ptr. Raises on a CUDA error code."""
    rc = load().cubcmp_argreduce(x_ptr, DTYPE_CODES[dtype], OPS[op], n, val_ptr, idx_ptr, temp_ptr, temp_nbytes,
                                 stream_ptr or None)
    if rc != 0:
        raise RuntimeError(f"cub::DeviceReduce::Arg{op.capitalize()} failed with CUDA error {rc}")
