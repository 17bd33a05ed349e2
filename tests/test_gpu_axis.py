"""GPU parity of ArgMax/ArgMin over a non-last axis (argreduce_axis) against
the CPU oracle, bit for bit: the strided-axis workloads at full size in both
tie modes, and every forced geometry (vector or scalar columns, warps along
the reduced axis, clusters of CTAs along it, unroll, outer loops) on
special-value tensors with ragged column tiles and misaligned bases."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import _lib  # noqa: E402

from gpu_util import axis_plan, raw_equal, run_axis  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def check_axis(x3, dtype, op, **kw):
    idx, val = run_axis(x3, dtype, op, **kw)
    eidx, evalue = oracle.argreduce_axis(x3, dtype, op)
    bad = np.argwhere(idx != eidx)
    assert bad.size == 0, f"{len(bad)} outputs differ, first {bad[:3].tolist()}: got {idx[tuple(bad[0])]} " \
                          f"want {eidx[tuple(bad[0])]}"
    assert raw_equal(val, evalue), "value bits differ"


@pytest.mark.parametrize("case", W.config_cases(6), ids=lambda c: c.name)
def test_axis_workload_full_size(case):
    x = W.make(case)
    check_axis(x, case.dtype, case.op)
    check_axis(x, case.dtype, case.op + "_last")


def fuzz3(dtype, outer, R, inner, seed):
    return W.fuzz_rows(dtype, outer * R, inner, seed=seed, p_special=0.15).reshape(outer, R, inner)


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_axis_forced_geometries(dtype):
    v = 2 if dtype == "f64" else 4
    for outer, R, inner in [(1, 1, 5), (3, 2, 3), (2, 17, 33), (1, 300, 128), (3, 64, 130), (2, 1000, 8),
                            (1, 33, 1000), (5, 7, 256)]:
        x = fuzz3(dtype, outer, R, inner, seed=outer * 1000 + R + inner)
        for op in W.ALL_OPS:
            check_axis(x, dtype, op)  # the planner's choice
            for cluster, warps, unroll, cg in ((1, 1, 4, 32), (1, 4, 8, 8), (2, 3, 4, 1), (5, 2, 4, 4),
                                               (16, 1, 8, 16), (3, 2, 8, 2)):
                check_axis(x, dtype, op, plan=axis_plan(cluster, warps, vec=0, unroll=unroll, outer=outer, cg=cg))
                if inner % v == 0:
                    check_axis(x, dtype, op, plan=axis_plan(cluster, warps, vec=1, unroll=unroll, outer=outer,
                                                            pdl=cluster != 2, cg=cg))
            if outer > 1:  # fewer outer slots than outer: the CTAs loop
                check_axis(x, dtype, op, plan=axis_plan(1, 2, vec=0, unroll=4, grid=1, cg=4))
            check_axis(x, dtype, op, offset=1)  # base not aligned: scalar columns


def test_axis_inner_one_is_last_axis():
    x = W.fuzz_rows("f32", 20, 3000, seed=5).reshape(20, 3000, 1)
    for op in W.ALL_OPS:
        check_axis(x, "f32", op)
        check_axis(x, "f32", op, plan=axis_plan(3, 2, vec=0, unroll=8, outer=20))


def test_axis_plan_validation():
    x = torch.randn(4, 100, 6, device="cuda")
    for bad in (axis_plan(cluster=2, warps=2, vec=0, outer=4, grid=2),  # a cluster plan may not loop over outer
                axis_plan(cluster=17, outer=4),
                axis_plan(cluster=1, unroll=3, outer=4),
                axis_plan(cluster=1, unroll=2, outer=4),
                axis_plan(cluster=1, outer=4, cg=3),
                axis_plan(cluster=1, vec=1, outer=4)):                    # inner 6 is not a multiple of 4
        with pytest.raises(A.ArgreduceError):
            A.argreduce_axis(x, 1, "max", plan=bad)
    p = A.argreduce_plan(4, 100, "f32", "max")  # a last-axis plan with inner != 1
    with pytest.raises(A.ArgreduceError):
        A.argreduce_axis(x, 1, "max", plan=p)
