"""Row-wise ArgMax / ArgMin over the last axis on a GB300 (sm_103a).

The reduction runs in hand-written CUDA kernels behind the C ABI of
``libargreduce.so`` (``include/argreduce.h``). This package is the thin Python
binding: it takes torch tensors for device memory and streams and passes raw
pointers to the library. It has no CPU fallback.

Semantics (onnxruntime #32092 and #31694, Semantics sections): one int64 index
per row; ties resolve to the lowest index; a leading NaN gives index 0; later
NaNs never win; rows entirely -inf, +inf or NaN give index 0.
"""
from __future__ import annotations

import threading
from typing import Dict, Optional, Tuple

from . import _lib
from ._lib import (ARGR_BF16, ARGR_F16, ARGR_F32, ARGR_F64, ARGR_MAX, ARGR_MIN,  # noqa: F401
                   ARGR_OK, ArgreduceError, DTYPE_CODES, OP_CODES, argr_caps, argr_plan, argreduce_axis_plan,
                   argreduce_cum_plan, argreduce_cum_scratch_bytes,
                   argreduce_device_caps,
                   argreduce_plan, argreduce_plan_check, argreduce_plan_scratch_bytes, argreduce_read_error,
                   argreduce_scratch_bytes,
                   argreduce_scratch_init, argreduce_status_string, argreduce_version, load, make_caps)

__all__ = [
    "argreduce", "argreduce_axis", "argreduce_axis_plan", "argreduce_cum", "argreduce_cum_plan",
    "argreduce_cum_scratch_bytes", "cummax", "cummin",
    "argmax", "argmin", "argreduce_with_plan", "argreduce_plan", "argreduce_plan_check", "argreduce_scratch_bytes",
    "argreduce_scratch_init", "argreduce_read_error", "argreduce_device_caps", "argreduce_status_string",
    "argreduce_version", "argreduce_plan_scratch_bytes", "ArgreduceError", "Scratch", "make_caps",
]


def _torch():
    import torch
    return torch


_ELEM_SIZE = {ARGR_F32: 4, ARGR_F16: 2, ARGR_BF16: 2, ARGR_F64: 8, _lib.ARGR_I32: 4, _lib.ARGR_I64: 8}
_tensor_codes: Optional[dict] = None
_raw_stream = None


def dtype_code(t, dtype: Optional[str]) -> int:
    """Element type code for a tensor; raw 16-bit tensors need ``dtype``."""
    global _tensor_codes
    if dtype is not None:
        code = DTYPE_CODES[dtype]
        if t.element_size() != _ELEM_SIZE[code]:
            raise TypeError(f"dtype {dtype} does not match element size {t.element_size()}")
        return code
    if _tensor_codes is None:
        torch = _torch()
        _tensor_codes = {torch.float32: ARGR_F32, torch.float16: ARGR_F16, torch.bfloat16: ARGR_BF16,
                         torch.float64: ARGR_F64, torch.int32: _lib.ARGR_I32, torch.int64: _lib.ARGR_I64}
    code = _tensor_codes.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported tensor dtype {t.dtype}; pass dtype= for raw 16-bit storage")
    return code


def _stream_ptr(stream, device_index: int) -> int:
    """The cudaStream_t to launch on: `stream` (a torch stream or a raw
    handle), else torch's current stream on the device."""
    global _raw_stream
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    if _raw_stream is None:
        torch = _torch()
        f = getattr(torch._C, "_cuda_getCurrentRawStream", None)  # no Stream object per call
        _raw_stream = f if f is not None else (lambda d: torch.cuda.current_stream(d).cuda_stream)
    return _raw_stream(device_index)


class Scratch:
    """Device scratch for one stream, grown on demand and prepared with
    argreduce_scratch_init() whenever it is (re)allocated; the preparation has
    completed when the constructor or ensure() returns, so the buffer may be
    used on any stream. Two calls that can run concurrently on the GPU must
    use different Scratch objects.

    A buffer, once handed to a call, stays allocated for the lifetime of the
    Scratch even after a larger one replaces it: a CUDA graph captured with
    the smaller buffer still holds its address, so it must not go back to
    torch's allocator while the graph may be replayed."""

    def __init__(self, device=None, nbytes: int = 0):
        torch = _torch()
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self.buf = None
        self.nbytes = 0
        self.retired = []  # buffers replaced by larger ones, kept alive (see above)
        if nbytes:
            self.ensure(nbytes, torch.cuda.current_stream(self.device).cuda_stream)

    def ensure(self, nbytes: int, stream_ptr: int):
        if nbytes <= self.nbytes:
            return
        torch = _torch()
        if torch.cuda.is_current_stream_capturing():
            # the preparing memset would be recorded into the graph instead of
            # running now, leaving the new buffer unprepared for eager calls
            raise RuntimeError("argreduce scratch must grow before a CUDA graph capture: make one call of the "
                               "largest problem (or pass a Scratch of enough bytes) before capturing")
        n = max(nbytes, 4096, 2 * self.nbytes)  # geometric growth: few buffers are ever retired
        buf = torch.empty(n, dtype=torch.uint8, device=self.device)
        st = argreduce_scratch_init(buf.data_ptr(), n, stream_ptr)
        if st != ARGR_OK:
            raise ArgreduceError(st, "argreduce_scratch_init")
        # The buffer may be used next on another stream (torch's streams do not
        # wait for each other): let the preparing memset finish first. Growth
        # is rare (geometric) and never happens inside a capture.
        torch.cuda.synchronize(self.device)
        if self.buf is not None:
            self.retired.append(self.buf)
        self.buf = buf
        self.nbytes = n

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() if self.buf is not None else 0


_scratch_lock = threading.Lock()
_scratch: Dict[Tuple[int, int], Scratch] = {}


def _default_scratch(device_index: int, stream_ptr: int) -> Scratch:
    key = (device_index, stream_ptr)
    with _scratch_lock:
        s = _scratch.get(key)
        if s is None:
            s = _scratch[key] = Scratch(device_index)
        return s


_need_lock = threading.Lock()
_need_cache: Dict[Tuple[int, int, int, int, int, bool], int] = {}


def _scratch_need(device_index: int, rows: int, cols: int, code: int, opc: int, cum: bool = False) -> int:
    """Scratch bytes of the planner's plan for this problem on this device,
    asked once per (device, shape, type, op): the planner is a pure function
    of them and the device's properties."""
    if rows == 0:
        return 0
    key = (device_index, rows, cols, code, opc, cum)
    need = _need_cache.get(key)
    if need is None:
        need = (argreduce_cum_scratch_bytes if cum else argreduce_scratch_bytes)(rows, cols, code, opc)
        with _need_lock:
            if len(_need_cache) > 4096:
                _need_cache.clear()
            _need_cache[key] = need
    return need


def _prepare(x, op, dtype, with_values, out_idx, out_val):
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (the library has no CPU path)")
    shape = x.shape
    if len(shape) == 0:
        raise ValueError("x must have at least one dimension")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous (row-major, reduced over its last axis)")
    cols = shape[-1]
    rows = x.numel() // cols if cols else 0
    code = dtype_code(x, dtype)
    opc = OP_CODES[op] if isinstance(op, str) else int(op)
    if out_idx is None or (with_values and out_val is None):
        torch = _torch()
        if out_idx is None:
            out_idx = torch.empty(shape[:-1], dtype=torch.int64, device=x.device)
        if with_values and out_val is None:
            out_val = torch.empty(shape[:-1], dtype=x.dtype, device=x.device)
    return rows, cols, code, opc, out_idx, out_val


def argreduce(x, op="max", *, dtype: Optional[str] = None, with_values: bool = False, out_idx=None, out_val=None,
              scratch: Optional[Scratch] = None, stream=None):
    """Reduce the last axis of a contiguous CUDA tensor.

    Returns ``(indices, values)``: int64 indices of shape ``x.shape[:-1]`` and,
    if ``with_values`` (or ``out_val``) is given, the raw elements
    ``x[..., index]`` (else ``None``). Runs on ``stream`` (default: torch's
    current stream) without synchronising.
    """
    rows, cols, code, opc, out_idx, out_val = _prepare(x, op, dtype, with_values, out_idx, out_val)
    dev = x.get_device()
    st_ptr = _stream_ptr(stream, dev)
    need = _scratch_need(dev, rows, cols, code, opc)
    if scratch is None and need:
        scratch = _default_scratch(dev, st_ptr)
    if need:
        scratch.ensure(need, st_ptr)
    st = _lib.load().argreduce(x.data_ptr(), code, rows, cols, opc, out_idx.data_ptr(),
                               out_val.data_ptr() if out_val is not None else None,
                               scratch.ptr if scratch is not None else None,
                               scratch.nbytes if scratch is not None else 0, st_ptr or None)
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce")
    return out_idx, out_val


def argreduce_with_plan(plan: argr_plan, x, op="max", *, dtype: Optional[str] = None, with_values: bool = False,
                        out_idx=None, out_val=None, scratch: Optional[Scratch] = None, stream=None):
    """argreduce() with an explicit (possibly forced) plan."""
    torch = _torch()
    rows, cols, code, opc, out_idx, out_val = _prepare(x, op, dtype, with_values, out_idx, out_val)
    st_ptr = _stream_ptr(stream, x.get_device())
    need = argreduce_plan_scratch_bytes(plan, rows)
    if scratch is None and need:
        scratch = _default_scratch(x.device.index, st_ptr)
    if need:
        scratch.ensure(need, st_ptr)
    st = _lib.argreduce_with_plan_raw(plan, x.data_ptr(), code, rows, cols, opc, out_idx.data_ptr(),
                                      out_val.data_ptr() if out_val is not None else 0,
                                      scratch.ptr if scratch is not None else 0,
                                      scratch.nbytes if scratch is not None else 0, st_ptr)
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_with_plan")
    return out_idx, out_val


def argreduce_axis(x, dim: int, op="max", *, dtype: Optional[str] = None, with_values: bool = False,
                   out_idx=None, out_val=None, scratch: Optional[Scratch] = None, stream=None, plan=None):
    """Reduce dimension ``dim`` of a contiguous CUDA tensor. The tensor is
    viewed as [outer, reduce, inner] around ``dim``; results have the shape of
    ``x`` without ``dim``. Ties and NaNs follow the same rules as argreduce()."""
    torch = _torch()
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    dim = dim % x.dim()
    outer = 1
    for d in x.shape[:dim]:
        outer *= d
    inner = 1
    for d in x.shape[dim + 1:]:
        inner *= d
    reduce = x.shape[dim]
    code = dtype_code(x, dtype)
    opc = _lib._code(OP_CODES, op)
    shape = tuple(x.shape[:dim]) + tuple(x.shape[dim + 1:])
    if out_idx is None:
        out_idx = torch.empty(shape, dtype=torch.int64, device=x.device)
    if with_values and out_val is None:
        out_val = torch.empty(shape, dtype=x.dtype, device=x.device)
    st_ptr = _stream_ptr(stream, x.get_device())
    need = 0
    if inner == 1 and outer > 0 and reduce > 0:
        need = argreduce_plan_scratch_bytes(plan, outer) if plan is not None else \
            argreduce_scratch_bytes(outer, reduce, code, opc)
    if scratch is None and need:
        scratch = _default_scratch(x.device.index, st_ptr)
    if need:
        scratch.ensure(need, st_ptr)
    st = _lib.argreduce_axis_raw(x.data_ptr(), code, outer, reduce, inner, opc, out_idx.data_ptr(),
                                 out_val.data_ptr() if out_val is not None else 0,
                                 scratch.ptr if scratch is not None else 0,
                                 scratch.nbytes if scratch is not None else 0, st_ptr, plan)
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_axis")
    return out_idx, out_val


def argreduce_cum(x, op="max", *, dtype: Optional[str] = None, with_values: bool = True, out_idx=None,
                  out_val=None, scratch: Optional[Scratch] = None, stream=None, plan=None):
    """cummax ("max") / cummin ("min") with indices along the last axis of a
    contiguous CUDA tensor: for every position, the ArgMax/ArgMin of the prefix
    up to it (ties keep the earlier index). Returns (indices, values) shaped
    like x (values None unless with_values or out_val). Runs on ``stream``
    without synchronising; the split scan uses ``scratch`` (default: the
    stream's own Scratch)."""
    torch = _torch()
    if not x.is_cuda or not x.is_contiguous() or x.dim() == 0:
        raise ValueError("x must be a contiguous CUDA tensor with at least one dimension")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    code = dtype_code(x, dtype)
    if out_idx is None:
        out_idx = torch.empty(x.shape, dtype=torch.int64, device=x.device)
    if with_values and out_val is None:
        out_val = torch.empty_like(x)
    st_ptr = _stream_ptr(stream, x.get_device())
    if rows == 0:
        need = 0
    elif plan is None:
        need = _scratch_need(x.device.index, rows, cols, code, _lib._code(OP_CODES, op), cum=True)
    else:
        need = argreduce_plan_scratch_bytes(plan, rows)
    if scratch is None and need:
        scratch = _default_scratch(x.device.index, st_ptr)
    if need:
        scratch.ensure(need, st_ptr)
    st = _lib.argreduce_cum_raw(x.data_ptr(), code, rows, cols, op, out_idx.data_ptr(),
                                out_val.data_ptr() if out_val is not None else 0,
                                scratch.ptr if scratch is not None else 0,
                                scratch.nbytes if scratch is not None else 0, st_ptr, plan)
    if st != ARGR_OK:
        raise ArgreduceError(st, "argreduce_cum")
    return out_idx, out_val


def cummax(x, **kw):
    return argreduce_cum(x, "max", **kw)


def cummin(x, **kw):
    return argreduce_cum(x, "min", **kw)


def argmax(x, **kw):
    return argreduce(x, "max", **kw)[0]


def argmin(x, **kw):
    return argreduce(x, "min", **kw)[0]
