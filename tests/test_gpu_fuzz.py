"""Seeded random GPU parity: problem shapes, element types, ops, base offsets
and forced plans drawn from every path and parameter range (the planner's
own choice included), each call compared with the CPU oracle bit for bit.
Plans the library rejects are skipped and counted; most draws must run."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import _lib  # noqa: E402

from gpu_util import forced_plan, raw_equal, run  # noqa: E402

VIEW = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64, "i32": np.int32, "i64": np.int64}


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def random_rows(rng, dtype, rows, cols):
    if dtype in ("i32", "i64"):
        info = np.iinfo(VIEW[dtype])
        x = rng.integers(-3, 4, size=(rows, cols)).astype(np.int64)
        x = np.where(rng.random((rows, cols)) < 0.02, info.max, x)
        x = np.where(rng.random((rows, cols)) < 0.02, info.min, x)
        return x.astype(VIEW[dtype])
    return W.fuzz_rows(dtype, rows, cols, seed=int(rng.integers(1 << 30)), p_special=float(rng.choice([0.0, 0.01, 0.3])))


def test_fuzz_argreduce():
    rng = np.random.Generator(np.random.PCG64(20260))
    ran = skipped = 0
    for it in range(600):
        dtype = str(rng.choice(W.DTYPES))
        op = str(rng.choice(W.ALL_OPS))
        rows = int(rng.choice([1, 2, 3, 7, 33, 300]))
        cols = int(rng.choice([1, 2, 5, 31, 64, 257, 1000, 4099, 20011, 65537]))
        x = random_rows(rng, dtype, rows, cols)
        kind = str(rng.choice(["planner", "rows", "split", "cluster"]))
        block = int(rng.choice([32, 64, 128, 256, 512, 1024]))
        unroll = int(rng.choice([1, 2, 4, 8]))
        if kind == "planner":
            plan = None
        elif kind == "rows":
            group, vec = int(rng.choice([1, 2, 4, 8, 16, 32])), int(rng.integers(2))
            plan = forced_plan("rows", group=group, vec=vec, block=block, unroll=int(rng.choice([4, 8])),
                               grid=int(rng.integers(1, 200)),
                               pipeline=group >= 16 and vec == 1 and block <= 256 and it % 2 == 0)
        elif kind == "split":
            bpr = int(rng.choice([1, 2, 3, 8, 40]))
            plan = forced_plan("split", bpr=bpr, grid_rows=rows if bpr > 1 else int(rng.integers(1, rows + 1)),
                               block=block, unroll=unroll, pdl=bool(rng.integers(2)))
        else:
            plan = forced_plan("cluster", cluster=int(rng.choice([2, 4, 8, 16])), grid_rows=rows, block=block,
                               unroll=unroll, bulk=bool(rng.integers(2)))
        offset = int(rng.choice([0, 0, 1, 3]))
        try:
            idx, val = run(x, dtype, op, plan=plan, offset=offset)
        except A.ArgreduceError as e:
            assert e.status in (_lib.ARGR_EINVAL, _lib.ARGR_EUNSUPPORTED), (it, e)
            skipped += 1
            continue
        eidx, evalue, _ = oracle.argreduce(x, dtype, op)
        assert (idx == eidx).all(), (it, dtype, op, rows, cols, kind, plan.as_dict() if plan else None)
        assert raw_equal(val, evalue), (it, dtype, op, kind)
        ran += 1
    assert ran >= 400, (ran, skipped)


def test_fuzz_cum():
    rng = np.random.Generator(np.random.PCG64(20261))
    ran = skipped = 0
    sc = A.Scratch()
    for it in range(400):
        dtype = str(rng.choice(["f32", "f16", "bf16", "f64", "i32", "i64"]))
        op = str(rng.choice(["max", "min"]))
        rows = int(rng.choice([1, 2, 5, 40]))
        cols = int(rng.choice([1, 3, 100, 1793, 7000, 40001]))
        x = random_rows(rng, dtype, rows, cols)
        kind = str(rng.choice(["planner", "cta", "cluster", "split", "lookback", "stash", "stream"]))
        block = int(rng.choice([32, 64, 128, 256, 512, 1024]))
        p = _lib.argr_plan()
        p.block, p.flags = block, int(rng.integers(2))
        if kind == "planner":
            p = None
        elif kind in ("cta", "cluster"):
            c = 1 if kind == "cta" else int(rng.choice([2, 4, 8, 16]))
            p.path, p.cluster, p.blocks_per_row = _lib.ARGR_PATH_CUM, c, c
            p.grid_rows = rows if c > 1 else int(rng.integers(1, rows + 1))
        elif kind == "stream":
            p.path, p.cluster = _lib.ARGR_PATH_CUM_STREAM, 1
            p.blocks_per_row = -(-cols // (block * 7))
            p.grid_rows = int(rng.choice([1, 5, 152, 999]))
        else:
            p.path, p.cluster, p.grid_rows = _lib.ARGR_PATH_CUM_SPLIT, 1, rows
            p.blocks_per_row = int(rng.choice([1, 2, 7, 64, 600]))
            p.flags |= {"split": 0, "lookback": _lib.ARGR_PLAN_LOOKBACK, "stash": _lib.ARGR_PLAN_STASH}[kind]
        flat = np.ascontiguousarray(x).view(VIEW[dtype]).reshape(-1)
        off = int(rng.choice([0, 1]))
        buf = torch.zeros(flat.size + off, dtype=getattr(torch, str(flat.dtype)), device="cuda")
        buf[off:] = torch.from_numpy(flat).cuda()
        try:
            idx, val = A.argreduce_cum(buf[off:].view(x.shape), op, dtype=dtype, plan=p, scratch=sc)
            torch.cuda.synchronize()
        except A.ArgreduceError as e:
            assert e.status in (_lib.ARGR_EINVAL, _lib.ARGR_EUNSUPPORTED), (it, e)
            skipped += 1
            continue
        eidx, evalue = oracle.cumreduce(x, dtype, op)
        got = idx.cpu().numpy()
        assert (got == eidx).all(), (it, dtype, op, rows, cols, kind, p.as_dict() if p else None)
        assert raw_equal(val.cpu().numpy().view(oracle.RAW_NP[dtype]), evalue), (it, kind)
        ran += 1
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    assert ran >= 250, (ran, skipped)


def test_fuzz_axis():
    from gpu_util import run_axis
    rng = np.random.Generator(np.random.PCG64(20262))
    for it in range(200):
        dtype = str(rng.choice(W.DTYPES))
        op = str(rng.choice(W.ALL_OPS))
        outer = int(rng.choice([1, 2, 9]))
        R = int(rng.choice([1, 2, 31, 700, 5000]))
        inner = int(rng.choice([1, 2, 3, 8, 33, 256, 1000]))
        x = random_rows(rng, dtype, outer, R * inner).reshape(outer, R, inner)
        idx, val = run_axis(x, dtype, op, offset=int(rng.choice([0, 1])))
        eidx, evalue = oracle.argreduce_axis(x, dtype, op)
        assert (idx == eidx).all(), (it, dtype, op, x.shape)
        assert raw_equal(val, evalue), (it, dtype, op, x.shape)
