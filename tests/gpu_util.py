"""Helpers for the GPU tests: move seeded raw inputs to the device, call the
library through its C ABI, bring results back as raw numpy arrays."""
import numpy as np

import row_wise_arg_gb300 as A
from row_wise_arg_gb300 import _lib

ES = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8}
NP_VIEW = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64}


def torch():
    import torch as t
    return t


def to_device(x: np.ndarray, dtype: str, offset: int = 0, guard: int = 0):
    """Copy raw rows to the device. `offset` elements of padding before the
    data make the base pointer unaligned; `guard` elements after it are filled
    with a sentinel. Returns (tensor view [rows, cols], backing buffer)."""
    t = torch()
    flat = np.ascontiguousarray(x).view(NP_VIEW[dtype]).reshape(-1)
    host = t.from_numpy(flat)
    buf = t.empty(flat.size + offset + guard, dtype=host.dtype, device="cuda")
    if offset:
        buf[:offset].fill_(0)
    if guard:
        buf[offset + flat.size:].fill_(0)
    buf[offset:offset + flat.size].copy_(host)
    view = buf[offset:offset + flat.size].view(x.shape)
    return view, buf


def alloc_out(rows: int, dtype: str, guard: int = 16):
    """Output buffers with sentinel guard bands on both sides."""
    t = torch()
    idx_buf = t.full((rows + 2 * guard,), -7777, dtype=t.int64, device="cuda")
    vt = {"f32": t.int32, "f16": t.int16, "bf16": t.int16, "f64": t.int64}[dtype]
    val_buf = t.full((rows + 2 * guard,), 0x3C3C, dtype=vt, device="cuda")
    return idx_buf, val_buf, guard


def check_guards(idx_buf, val_buf, guard: int, rows: int):
    ib = idx_buf.cpu().numpy()
    vb = val_buf.cpu().numpy()
    assert (ib[:guard] == -7777).all() and (ib[guard + rows:] == -7777).all(), "out_idx guard band overwritten"
    assert (vb[:guard] == 0x3C3C).all() and (vb[guard + rows:] == 0x3C3C).all(), "out_val guard band overwritten"


def run(x: np.ndarray, dtype: str, op: str, plan=None, offset: int = 0, scratch=None, want_val: bool = True):
    """Run the CUDA path on raw rows; returns (idx int64, val raw) numpy."""
    t = torch()
    rows, cols = x.shape
    xd, _keep = to_device(x, dtype, offset=offset, guard=64)
    idx_buf, val_buf, g = alloc_out(rows, dtype)
    out_idx = idx_buf[g:g + rows]
    out_val = val_buf[g:g + rows] if want_val else None
    if plan is None:
        A.argreduce(xd, op, dtype=dtype, out_idx=out_idx, out_val=out_val, scratch=scratch)
    else:
        A.argreduce_with_plan(plan, xd, op, dtype=dtype, out_idx=out_idx, out_val=out_val, scratch=scratch)
    t.cuda.synchronize()
    check_guards(idx_buf, val_buf, g, rows)
    idx = out_idx.cpu().numpy()
    val = None
    if want_val:
        raw_t = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "f64": np.float64}[dtype]
        val = out_val.cpu().numpy().view(raw_t)
    return idx, val


def forced_plan(path: str, **kw):
    p = _lib.argr_plan()
    p.block = kw.get("block", 256)
    p.unroll = kw.get("unroll", 4)
    p.flags = _lib.ARGR_PLAN_PDL if kw.get("pdl", True) else 0
    if path == "rows":
        p.path = _lib.ARGR_PATH_ROWS
        p.group = kw["group"]
        p.vec = kw.get("vec", 0)
        p.unroll = kw.get("unroll", 4)
        p.grid_rows = kw.get("grid", 64)
        p.blocks_per_row = 1
        if kw.get("pipeline"):
            p.flags |= _lib.ARGR_PLAN_PIPELINE
    elif path == "split":
        p.path = _lib.ARGR_PATH_SPLIT
        p.blocks_per_row = kw["bpr"]
        p.grid_rows = kw["grid_rows"]
    elif path == "stream":
        p.path = _lib.ARGR_PATH_STREAM
        p.group = kw["group"]
        p.stages = kw.get("stages", 2)
        p.stage_bytes = kw.get("stage_bytes", 8192)
        p.grid_rows = kw.get("grid", 8)
        p.blocks_per_row = 1
        p.vec = 1
        if kw.get("expire"):
            p.flags |= _lib.ARGR_PLAN_TEST_EXPIRE
    elif path == "cluster":
        p.path = _lib.ARGR_PATH_CLUSTER
        if kw.get("bulk"):
            p.flags |= _lib.ARGR_PLAN_BULK
        p.cluster = kw["cluster"]
        p.blocks_per_row = kw["cluster"]
        p.grid_rows = kw["grid_rows"]
    else:
        raise ValueError(path)
    if kw.get("prefetch"):
        p.flags |= _lib.ARGR_PLAN_PREFETCH
    if kw.get("prefetch_head"):
        p.flags |= _lib.ARGR_PLAN_PREFETCH | _lib.ARGR_PLAN_PREFETCH_HEAD
    return p


def raw_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return a.shape == b.shape and bool((a.view(np.uint8) == b.view(np.uint8)).all())


def run_axis(x3: np.ndarray, dtype: str, op: str, plan=None, offset: int = 0):
    """Reduce the middle axis of raw [outer, R, inner] data on the device
    through argreduce_axis(); returns (idx [outer, inner], val raw)."""
    t = torch()
    outer, R, inner = x3.shape
    xd, _keep = to_device(x3.reshape(outer, R * inner), dtype, offset=offset, guard=64)
    n = outer * inner
    idx_buf, val_buf, g = alloc_out(n, dtype)
    out_idx = idx_buf[g:g + n]
    out_val = val_buf[g:g + n]
    A.argreduce_axis(xd.view(outer, R, inner), 1, op, dtype=dtype, out_idx=out_idx, out_val=out_val, plan=plan)
    t.cuda.synchronize()
    check_guards(idx_buf, val_buf, g, n)
    raw_t = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "f64": np.float64}[dtype]
    return out_idx.cpu().numpy().reshape(outer, inner), out_val.cpu().numpy().view(raw_t).reshape(outer, inner)


def axis_plan(cluster=1, warps=4, vec=1, unroll=8, grid=None, outer=1, pdl=True, cg=32):
    p = _lib.argr_plan()
    p.path = _lib.ARGR_PATH_AXIS
    p.group = cg
    p.block = 32 * warps
    p.vec = vec
    p.unroll = unroll
    p.cluster = cluster
    p.blocks_per_row = cluster
    p.grid_rows = grid if grid is not None else outer
    p.flags = _lib.ARGR_PLAN_PDL if pdl else 0
    return p
