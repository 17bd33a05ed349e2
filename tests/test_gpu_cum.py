"""GPU parity of cummax / cummin with indices (argreduce_cum) against the CPU
oracle, bit for bit: the Paddle-issue workloads at full size, and every
forced geometry (one CTA per row with row loops, clusters of 2..16 CTAs per
row, tile widths from 32 to 1024 threads) on special-value rows of every
element type, including leading NaNs and the integer extremes."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import _lib  # noqa: E402

from gpu_util import raw_equal  # noqa: E402

VIEW = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64, "i32": np.int32, "i64": np.int64}
CUM_DTYPES = ("f32", "f16", "bf16", "f64", "i32", "i64")


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def cum_plan(cluster=1, block=256, grid=1, pdl=True):
    p = _lib.argr_plan()
    p.path = _lib.ARGR_PATH_CUM
    p.block = block
    p.cluster = cluster
    p.blocks_per_row = cluster
    p.grid_rows = grid
    p.flags = _lib.ARGR_PLAN_PDL if pdl else 0
    return p


def run_cum(x, dtype, op, plan=None):
    xd = torch.from_numpy(np.ascontiguousarray(x).view(VIEW[dtype])).cuda()
    idx, val = A.argreduce_cum(xd, op, dtype=dtype, plan=plan)
    torch.cuda.synchronize()
    raw_t = oracle.RAW_NP[dtype]
    return idx.cpu().numpy(), val.cpu().numpy().view(raw_t)


def check_cum(x, dtype, op, plan=None):
    idx, val = run_cum(x, dtype, op, plan)
    eidx, evalue = oracle.cumreduce(x, dtype, op)
    bad = np.argwhere(idx != eidx)
    assert bad.size == 0, f"{len(bad)} outputs differ, first {bad[:3].tolist()}: got {idx[tuple(bad[0])]} " \
                          f"want {eidx[tuple(bad[0])]}"
    assert raw_equal(val, evalue), "value bits differ"


def cum_rows(dtype, rows, cols, seed):
    if dtype in ("i32", "i64"):
        rng = np.random.Generator(np.random.PCG64(seed))
        info = np.iinfo(VIEW[dtype])
        x = rng.integers(-4, 5, size=(rows, cols)).astype(np.int64)
        x = np.where(rng.random((rows, cols)) < 0.03, info.max, x)
        x = np.where(rng.random((rows, cols)) < 0.03, info.min, x)
        return x.astype(VIEW[dtype])
    return W.fuzz_rows(dtype, rows, cols, seed=seed, p_special=0.1)


@pytest.mark.parametrize("case", W.config_cases(7), ids=lambda c: c.name)
def test_cum_workload_full_size(case):
    x = W.make(case)
    check_cum(x, case.dtype, case.op)
    check_cum(x, case.dtype, "min" if case.op == "max" else "max")


@pytest.mark.parametrize("dtype", CUM_DTYPES)
def test_cum_forced_geometries(dtype):
    for rows, cols in [(1, 1), (1, 2), (3, 7), (2, 1000), (1, 20011), (5, 4099), (33, 300)]:
        x = cum_rows(dtype, rows, cols, seed=rows * 100 + cols)
        for op in ("max", "min"):
            check_cum(x, dtype, op)
            for cluster, block in ((1, 32), (1, 1024), (2, 64), (5, 256), (16, 32), (16, 128)):
                check_cum(x, dtype, op, plan=cum_plan(cluster, block, grid=rows, pdl=cluster != 5))
            check_cum(x, dtype, op, plan=cum_plan(1, 128, grid=1))  # one CTA loops over every row


def test_cum_leading_nan_and_extremes():
    x = W.fuzz_rows("f32", 6, 5000, seed=3, p_special=0.3)
    x[0, 0] = np.nan
    x[1, :] = np.nan
    x[2, :] = -np.inf
    for op in ("max", "min"):
        check_cum(x, "f32", op)
        check_cum(x, "f32", op, plan=cum_plan(4, 128, grid=6))
        idx, _ = run_cum(x, "f32", op)
        assert (idx[0] == 0).all() and (idx[1] == 0).all()


def test_cum_last_element_is_argreduce():
    x = W.fuzz_rows("bf16", 40, 3001, seed=9)
    for op in ("max", "min"):
        idx, _ = run_cum(x, "bf16", op)
        eidx, _, _ = oracle.argreduce(x, "bf16", op)
        assert (idx[:, -1] == eidx).all()


def test_cum_rejections():
    x = torch.zeros(4, 100, device="cuda")
    with pytest.raises(A.ArgreduceError) as e:
        A.argreduce_cum(x, "max_last")
    assert e.value.status == _lib.ARGR_EUNSUPPORTED
    with pytest.raises(A.ArgreduceError):
        A.argreduce_cum(x, "max", plan=cum_plan(2, 256, grid=1))  # a cluster plan may not loop over rows
    xi = torch.zeros(4, 100, dtype=torch.int64, device="cuda")
    with pytest.raises(A.ArgreduceError) as e:
        A.argreduce(xi, "max")  # the integer types are for the scan only
    assert e.value.status == _lib.ARGR_EUNSUPPORTED
