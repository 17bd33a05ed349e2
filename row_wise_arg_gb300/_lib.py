"""ctypes binding of libargreduce.so (include/argreduce.h).

Argument marshalling only: every step of the reduction runs in the library's
CUDA kernels. PyTorch provides device memory and streams. There is no CPU
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Optional, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libargreduce.so")

ARGR_F32, ARGR_F16, ARGR_BF16, ARGR_F64, ARGR_I32, ARGR_I64 = 0, 1, 2, 3, 4, 5
ARGR_MAX, ARGR_MIN, ARGR_MAX_LAST, ARGR_MIN_LAST = 0, 1, 2, 3
(ARGR_OK, ARGR_EINVAL, ARGR_ESCRATCH, ARGR_EUNSUPPORTED, ARGR_ECUDA, ARGR_ETIMEOUT) = range(6)
ARGR_PATH_NONE, ARGR_PATH_ROWS, ARGR_PATH_SPLIT, ARGR_PATH_CLUSTER, ARGR_PATH_STREAM, ARGR_PATH_AXIS, \
    ARGR_PATH_CUM, ARGR_PATH_CUM_SPLIT, ARGR_PATH_CUM_STREAM = range(9)
ARGR_PLAN_PDL = 1
ARGR_PLAN_BULK = 2
ARGR_PLAN_TEST_EXPIRE = 4
ARGR_PLAN_STASH = 8
ARGR_PLAN_LOOKBACK = 16
ARGR_PLAN_PIPELINE = 32
ARGR_PLAN_PREFETCH = 64
ARGR_PLAN_PREFETCH_HEAD = 128

DTYPE_CODES = {"f32": ARGR_F32, "f16": ARGR_F16, "bf16": ARGR_BF16, "f64": ARGR_F64, "i32": ARGR_I32,
               "i64": ARGR_I64}
OP_CODES = {"max": ARGR_MAX, "min": ARGR_MIN, "max_last": ARGR_MAX_LAST, "min_last": ARGR_MIN_LAST}
PATH_NAMES = {ARGR_PATH_NONE: "none", ARGR_PATH_ROWS: "rows", ARGR_PATH_SPLIT: "split",
              ARGR_PATH_CLUSTER: "cluster", ARGR_PATH_STREAM: "stream", ARGR_PATH_AXIS: "axis",
              ARGR_PATH_CUM: "cum", ARGR_PATH_CUM_SPLIT: "cum_split", ARGR_PATH_CUM_STREAM: "cum_stream"}

# Every function the header declares (checked by the tests).
EXPORTS = (
    "argreduce_scratch_bytes", "argreduce_scratch_init", "argreduce", "argreduce_plan",
    "argreduce_with_plan", "argreduce_plan_scratch_bytes", "argreduce_read_error",
    "argreduce_device_caps", "argreduce_status_string", "argreduce_version", "argreduce_noalloc",
    "argreduce_axis", "argreduce_axis_plan", "argreduce_axis_with_plan", "argreduce_cum", "argreduce_cum_plan",
    "argreduce_cum_with_plan", "argreduce_cum_scratch_bytes", "argreduce_plan_check",
)


class argr_caps(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("max_threads_per_sm", ctypes.c_int32),
                ("max_cluster", ctypes.c_int32), ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32)]


class argr_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("block", ctypes.c_int32), ("group", ctypes.c_int32),
                ("vec", ctypes.c_int32), ("unroll", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("stages", ctypes.c_int32), ("stage_bytes", ctypes.c_int32),
                ("reserved", ctypes.c_int32),
                ("blocks_per_row", ctypes.c_int64), ("grid_rows", ctypes.c_int64),
                ("scratch_bytes", ctypes.c_uint64)]

    def as_dict(self) -> Dict[str, int]:
        d = {f: int(getattr(self, f)) for f, _ in self._fields_}
        d["path_name"] = PATH_NAMES.get(d["path"], "?")
        return d

    def __repr__(self) -> str:
        return f"argr_plan({self.as_dict()})"


class ArgreduceError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}" if what else status_string(status))


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libargreduce.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m row_wise_arg_gb300.build` "
                               "(or __graft_entry__.build()); there is no fallback implementation")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.argreduce_scratch_bytes.argtypes = [i64, i64, i32, i32]
        lib.argreduce_scratch_bytes.restype = sz
        lib.argreduce_scratch_init.argtypes = [vp, sz, vp]
        lib.argreduce_scratch_init.restype = i32
        lib.argreduce.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp, sz, vp]
        lib.argreduce.restype = i32
        lib.argreduce_plan.argtypes = [i64, i64, i32, i32, ctypes.POINTER(argr_caps), ctypes.POINTER(argr_plan)]
        lib.argreduce_plan.restype = i32
        lib.argreduce_with_plan.argtypes = [ctypes.POINTER(argr_plan), vp, i32, i64, i64, i32, vp, vp, vp, sz, vp]
        lib.argreduce_with_plan.restype = i32
        lib.argreduce_plan_check.argtypes = [ctypes.POINTER(argr_plan), i64, i64, i32, ctypes.POINTER(argr_caps), i32]
        lib.argreduce_plan_check.restype = i32
        lib.argreduce_plan_scratch_bytes.argtypes = [ctypes.POINTER(argr_plan), i64]
        lib.argreduce_plan_scratch_bytes.restype = sz
        lib.argreduce_read_error.argtypes = [vp, vp]
        lib.argreduce_read_error.restype = i32
        lib.argreduce_device_caps.argtypes = [i32, ctypes.POINTER(argr_caps)]
        lib.argreduce_device_caps.restype = i32
        lib.argreduce_status_string.argtypes = [i32]
        lib.argreduce_status_string.restype = ctypes.c_char_p
        lib.argreduce_axis.argtypes = [vp, i32, i64, i64, i64, i32, vp, vp, vp, sz, vp]
        lib.argreduce_axis.restype = i32
        lib.argreduce_axis_plan.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(argr_caps),
                                            ctypes.POINTER(argr_plan)]
        lib.argreduce_axis_plan.restype = i32
        lib.argreduce_axis_with_plan.argtypes = [ctypes.POINTER(argr_plan), vp, i32, i64, i64, i64, i32, vp, vp, vp,
                                                 sz, vp]
        lib.argreduce_axis_with_plan.restype = i32
        lib.argreduce_cum.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp, sz, vp]
        lib.argreduce_cum.restype = i32
        lib.argreduce_cum_plan.argtypes = [i64, i64, i32, i32, ctypes.POINTER(argr_caps), ctypes.POINTER(argr_plan)]
        lib.argreduce_cum_plan.restype = i32
        lib.argreduce_cum_with_plan.argtypes = [ctypes.POINTER(argr_plan), vp, i32, i64, i64, i32, vp, vp, vp, sz,
                                                vp]
        lib.argreduce_cum_with_plan.restype = i32
        lib.argreduce_cum_scratch_bytes.argtypes = [i64, i64, i32, i32]
        lib.argreduce_cum_scratch_bytes.restype = sz
        lib.argreduce_noalloc.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp]
        lib.argreduce_noalloc.restype = i32
        lib.argreduce_version.argtypes = []
        lib.argreduce_version.restype = ctypes.c_char_p
        del i64p
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# Thin wrappers with the C names (plain integers and pointers).
# ---------------------------------------------------------------------------
def status_string(status: int) -> str:
    return load().argreduce_status_string(status).decode()


def argreduce_status_string(status: int) -> str:
    return status_string(status)


def argreduce_version() -> str:
    return load().argreduce_version().decode()


def _code(table: Dict[str, int], v) -> int:
    return table[v] if isinstance(v, str) else int(v)


def argreduce_scratch_bytes(rows: int, cols: int, dtype, op) -> int:
    return int(load().argreduce_scratch_bytes(rows, cols, _code(DTYPE_CODES, dtype), _code(OP_CODES, op)))


def argreduce_scratch_init(scratch_ptr: int, nbytes: int, stream_ptr: int = 0) -> int:
    return load().argreduce_scratch_init(scratch_ptr or None, nbytes, stream_ptr or None)


def argreduce_raw(x_ptr: int, dtype, rows: int, cols: int, op, out_idx_ptr: int, out_val_ptr: int,
                  scratch_ptr: int, scratch_bytes: int, stream_ptr: int) -> int:
    """The C call argreduce() with integer pointers; returns the status."""
    return load().argreduce(x_ptr or None, _code(DTYPE_CODES, dtype), rows, cols, _code(OP_CODES, op),
                            out_idx_ptr or None, out_val_ptr or None, scratch_ptr or None, scratch_bytes,
                            stream_ptr or None)


def argreduce_noalloc_raw(x_ptr: int, dtype, rows: int, cols: int, op, out_idx_ptr: int, out_val_ptr: int,
                         stream_ptr: int) -> int:
    """The C call argreduce_noalloc(): no scratch argument, allocates nothing;
    its scratch is an array inside the library shared by every call."""
    return load().argreduce_noalloc(x_ptr or None, _code(DTYPE_CODES, dtype), rows, cols, _code(OP_CODES, op),
                                    out_idx_ptr or None, out_val_ptr or None, stream_ptr or None)


def argreduce_with_plan_raw(plan: argr_plan, x_ptr: int, dtype, rows: int, cols: int, op, out_idx_ptr: int,
                            out_val_ptr: int, scratch_ptr: int, scratch_bytes: int, stream_ptr: int) -> int:
    return load().argreduce_with_plan(ctypes.byref(plan), x_ptr or None, _code(DTYPE_CODES, dtype), rows, cols,
                                      _code(OP_CODES, op), out_idx_ptr or None, out_val_ptr or None,
                                      scratch_ptr or None, scratch_bytes, stream_ptr or None)


def argreduce_plan(rows: int, cols: int, dtype, op, caps: Optional[argr_caps] = None) -> argr_plan:
    p = argr_plan()
    st = load().argreduce_plan(rows, cols, _code(DTYPE_CODES, dtype), _code(OP_CODES, op),
                               ctypes.byref(caps) if caps is not None else None, ctypes.byref(p))
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_plan")
    return p


def argreduce_plan_check(plan: argr_plan, rows: int, cols: int, dtype, caps: argr_caps,
                         rows_aligned: bool = True) -> int:
    """Status argreduce_with_plan() would give this plan on a device with `caps`
    (no GPU needed)."""
    return load().argreduce_plan_check(ctypes.byref(plan), rows, cols, _code(DTYPE_CODES, dtype),
                                       ctypes.byref(caps), 1 if rows_aligned else 0)


def argreduce_axis_raw(x_ptr: int, dtype, outer: int, reduce: int, inner: int, op, out_idx_ptr: int,
                       out_val_ptr: int, scratch_ptr: int, scratch_bytes: int, stream_ptr: int,
                       plan: Optional[argr_plan] = None) -> int:
    """argreduce_axis() (or argreduce_axis_with_plan() when a plan is given)."""
    args = (x_ptr or None, _code(DTYPE_CODES, dtype), outer, reduce, inner, _code(OP_CODES, op),
            out_idx_ptr or None, out_val_ptr or None, scratch_ptr or None, scratch_bytes, stream_ptr or None)
    if plan is None:
        return load().argreduce_axis(*args)
    return load().argreduce_axis_with_plan(ctypes.byref(plan), *args)


def argreduce_axis_plan(outer: int, reduce: int, inner: int, dtype, op, caps: Optional[argr_caps] = None) -> argr_plan:
    p = argr_plan()
    st = load().argreduce_axis_plan(outer, reduce, inner, _code(DTYPE_CODES, dtype), _code(OP_CODES, op),
                                    ctypes.byref(caps) if caps is not None else None, ctypes.byref(p))
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_axis_plan")
    return p


def argreduce_cum_raw(x_ptr: int, dtype, rows: int, cols: int, op, out_idx_ptr: int, out_val_ptr: int,
                      scratch_ptr: int, scratch_bytes: int, stream_ptr: int, plan: Optional[argr_plan] = None) -> int:
    """argreduce_cum() (or argreduce_cum_with_plan() when a plan is given)."""
    args = (x_ptr or None, _code(DTYPE_CODES, dtype), rows, cols, _code(OP_CODES, op), out_idx_ptr or None,
            out_val_ptr or None, scratch_ptr or None, scratch_bytes, stream_ptr or None)
    if plan is None:
        return load().argreduce_cum(*args)
    return load().argreduce_cum_with_plan(ctypes.byref(plan), *args)


def argreduce_cum_plan(rows: int, cols: int, dtype, op, caps: Optional[argr_caps] = None) -> argr_plan:
    p = argr_plan()
    st = load().argreduce_cum_plan(rows, cols, _code(DTYPE_CODES, dtype), _code(OP_CODES, op),
                                   ctypes.byref(caps) if caps is not None else None, ctypes.byref(p))
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_cum_plan")
    return p


def argreduce_cum_scratch_bytes(rows: int, cols: int, dtype, op) -> int:
    return int(load().argreduce_cum_scratch_bytes(rows, cols, _code(DTYPE_CODES, dtype), _code(OP_CODES, op)))


def argreduce_plan_scratch_bytes(plan: argr_plan, rows: int) -> int:
    return int(load().argreduce_plan_scratch_bytes(ctypes.byref(plan), rows))


def argreduce_read_error(scratch_ptr: int, stream_ptr: int = 0) -> int:
    return load().argreduce_read_error(scratch_ptr or None, stream_ptr or None)


def argreduce_device_caps(device: int = 0) -> argr_caps:
    c = argr_caps()
    st = load().argreduce_device_caps(device, ctypes.byref(c))
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_device_caps")
    return c


def make_caps(sm_count: int, max_threads_per_sm: int = 2048, max_cluster: int = 16, cc: Tuple[int, int] = (10, 3)):
    return argr_caps(sm_count, max_threads_per_sm, max_cluster, cc[0], cc[1])
