"""GPU parity: the CUDA path against the CPU oracle, bit for bit (index and
raw value bits, tolerance 0), through the C ABI.

* every workload case at full size, in the planner's launch configuration
  (the one the benchmark times);
* every kernel path forced (thread/group/warp per row, vector and scalar
  loads, one or many CTAs per row with the global merge, clusters of 2..16)
  on special-value fuzz rows whose widths span several tiles and ragged tails,
  with unaligned base pointers;
* the test shapes described by onnxruntime #31694 and #32092 (Testing).
"""
import json
import os

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

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def check(x, dtype, op, **kw):
    idx, val = run(x, dtype, op, **kw)
    eidx, evalue, _ = oracle.argreduce(x, dtype, op)
    bad = np.nonzero(idx != eidx)[0]
    assert bad.size == 0, f"{bad.size} rows differ, first rows {bad[:5]}: got {idx[bad[:5]]} want {eidx[bad[:5]]}"
    assert raw_equal(val, evalue), "value bits differ"


# ---------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", [c for _, c in W.all_cases()], ids=lambda c: c.name)
def test_workload_full_size(case):
    x = W.make(case)
    check(x, case.dtype, case.op)
    check(x, case.dtype, case.op + "_last")  # the same rows with ties to the last index


def test_narrow_matches_thread_per_row():
    """Narrow rows: the planner's path and a forced one-thread-per-row scan
    give the same bits (and both equal the oracle)."""
    for c in W.config_cases(5):
        x = W.make(c)
        check(x, c.dtype, c.op)
        check(x, c.dtype, c.op, plan=forced_plan("rows", group=1, vec=0, grid=1024))


# ---------------------------------------------------------------------------
# Every path forced, on fuzz rows.
# ---------------------------------------------------------------------------
WIDTHS = [1, 2, 3, 7, 8, 9, 31, 32, 33, 127, 128, 129, 255, 256, 257, 1000, 4099, 20011]


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("group", [1, 2, 4, 8, 16, 32])
def test_rows_path(dtype, group):
    es = W.ELEM_SIZE[dtype]
    for cols in WIDTHS[:-1]:
        rows = 37 if cols < 2000 else 5
        x = W.fuzz_rows(dtype, rows, cols, seed=cols * 31 + group)
        for op in W.ALL_OPS:
            check(x, dtype, op, plan=forced_plan("rows", group=group, vec=0, grid=3, pdl=False))
            check(x, dtype, op, plan=forced_plan("rows", group=group, vec=0, grid=64, unroll=8), offset=1)
            if (cols * es) % 16 == 0:
                check(x, dtype, op, plan=forced_plan("rows", group=group, vec=1, grid=5))
                check(x, dtype, op, plan=forced_plan("rows", group=group, vec=1, grid=7, unroll=8, pdl=False))
                if group >= 16:  # software-pipelined loads
                    check(x, dtype, op, plan=forced_plan("rows", group=group, vec=1, grid=5, block=64,
                                                         pipeline=True))
                    check(x, dtype, op, plan=forced_plan("rows", group=group, vec=1, grid=2, unroll=8,
                                                         pipeline=True, pdl=False))


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("bpr", [1, 2, 5, 64])
def test_split_path(dtype, bpr):
    for cols in WIDTHS:
        rows = 3 if cols > 4000 else 9
        x = W.fuzz_rows(dtype, rows, cols, seed=cols * 7 + bpr)
        for op in W.ALL_OPS:
            for block, unroll in ((256, 4), (32, 1), (1024, 8), (64, 2)):
                check(x, dtype, op, plan=forced_plan("split", bpr=bpr, grid_rows=rows, block=block,
                                                     unroll=unroll, pdl=block != 32))
            for off in (1, 3):
                check(x, dtype, op, plan=forced_plan("split", bpr=bpr, grid_rows=rows), offset=off)
            if bpr == 1:  # row loop: fewer row slots than rows
                check(x, dtype, op, plan=forced_plan("split", bpr=1, grid_rows=2))


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("cluster", [2, 4, 8, 16])
def test_cluster_path(dtype, cluster):
    """One row per CTA (row slots >= rows): every warp pushes its candidate
    into CTA 0 (st.async on an mbarrier); fewer row slots than rows: CTAs loop
    over rows and merge through a cluster barrier."""
    caps = A.argreduce_device_caps(torch.cuda.current_device())
    if caps.max_cluster < cluster:
        pytest.skip("cluster size not supported")
    for cols in WIDTHS:
        rows = 3 if cols > 4000 else 7
        x = W.fuzz_rows(dtype, rows, cols, seed=cols * 13 + cluster)
        for op in W.ALL_OPS:
            check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=rows))
            check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=2, unroll=1, pdl=False),
                  offset=1)
            check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=rows, block=512, unroll=8))
            # more row slots than rows: the barrier merge with idle clusters
            check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=rows + 3, block=96, unroll=2),
                  offset=3)
            if cols * W.ELEM_SIZE[dtype] // 16 <= cluster * 8192:  # share fits the 128 KiB bulk buffer
                check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=rows, bulk=True))
                check(x, dtype, op, plan=forced_plan("cluster", cluster=cluster, grid_rows=2, bulk=True, block=128),
                      offset=1)


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_prefetch_paths(dtype):
    """ARGR_PLAN_PREFETCH (L2 prefetch of each CTA's first share before the
    dependency wait) on the rows, split, cluster and streaming paths, and its
    16 KiB head variant on the rows path, with aligned and unaligned bases,
    ragged tails, row loops and shares wider than what one CTA prefetches."""
    es = W.ELEM_SIZE[dtype]
    caps = A.argreduce_device_caps(torch.cuda.current_device())
    for cols in (1, 9, 257, 4099, 20011, 300001):
        rows = 2 if cols > 100000 else 5 if cols > 4000 else 37
        x = W.fuzz_rows(dtype, rows, cols, seed=cols * 3 + es)
        for op in W.ALL_OPS:
            for off in (0, 1):
                check(x, dtype, op, offset=off, plan=forced_plan("rows", group=32, vec=0, grid=3, prefetch=True))
                check(x, dtype, op, offset=off, plan=forced_plan("rows", group=32, vec=0, grid=3, prefetch_head=True))
                check(x, dtype, op, offset=off, plan=forced_plan("split", bpr=1, grid_rows=2, prefetch=True))
                check(x, dtype, op, offset=off, plan=forced_plan("split", bpr=7, grid_rows=rows, prefetch=True))
                if caps.max_cluster >= 16:
                    check(x, dtype, op, offset=off, plan=forced_plan("cluster", cluster=16, grid_rows=2,
                                                                     block=512, unroll=8, prefetch=True))
            if (cols * es) % 16 == 0:
                for g in (4, 32):
                    check(x, dtype, op, plan=forced_plan("rows", group=g, vec=1, grid=5, prefetch=True))
                    check(x, dtype, op, plan=forced_plan("rows", group=g, vec=1, grid=5, prefetch_head=True))
                check(x, dtype, op, plan=forced_plan("rows", group=32, vec=1, grid=2, unroll=8, pipeline=True,
                                                     prefetch=True))
                check(x, dtype, op, plan=forced_plan("cluster", cluster=4, grid_rows=rows, prefetch=True))
                check(x, dtype, op, plan=forced_plan("stream", group=32, stages=2, stage_bytes=8192, grid=3,
                                                     block=128, prefetch=True))


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("group", [1, 4, 32])
def test_stream_path(dtype, group):
    """Per-warp bulk-copy streaming: rows that fit a stage (whole rows, G
    lanes per row) and rows cut into pieces (whole warp); warps with many rows,
    one row and none."""
    es = W.ELEM_SIZE[dtype]
    for cols in [16 // es, 32 // es, 64, 256, 1000 - 1000 % (16 // es), 2048, 4096, 20008, 100000]:
        for rows in (1, 7, 300):
            if rows * cols > 3_000_000:
                continue
            x = W.fuzz_rows(dtype, rows, cols, seed=rows * 7 + cols + group)
            row_bytes = cols * es
            for stages, stage_bytes, block, grid in ((2, 8192, 256, 3), (4, 4096, 128, 40), (1, 1024, 1024, 1),
                                                     (3, 65536, 32, 2)):
                if row_bytes > stage_bytes and group != 32:
                    continue
                for op in W.ALL_OPS:
                    check(x, dtype, op, plan=forced_plan("stream", group=group, stages=stages,
                                                         stage_bytes=stage_bytes, block=block, grid=grid))


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_exhaustive_alphabet_rows(dtype):
    """All 8**4 rows of length 4 over the special alphabet, on every path."""
    x = W.exhaustive_rows(dtype, 4)
    rows = x.shape[0]
    for op in W.ALL_OPS:
        check(x, dtype, op)
        check(x, dtype, op, plan=forced_plan("rows", group=4, vec=0, grid=100))
        check(x, dtype, op, plan=forced_plan("split", bpr=1, grid_rows=min(rows, 1000), block=32))
        if W.ELEM_SIZE[dtype] * 4 % 16 == 0:
            check(x, dtype, op, plan=forced_plan("stream", group=1, stages=2, stage_bytes=4096, grid=50))
        for r0 in range(0, rows, 2048):  # a multi-CTA split has at most 2048 row slots
            xs = np.ascontiguousarray(x[r0:r0 + 2048])
            check(xs, dtype, op, plan=forced_plan("split", bpr=3, grid_rows=xs.shape[0], block=32))


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_planner_default_on_fuzz(dtype):
    for rows, cols in [(1, 1), (1, 5), (3, 100000), (2000, 33), (500, 3000), (64, 70000), (1, 300001)]:
        x = W.fuzz_rows(dtype, rows, cols, seed=rows + cols)
        for op in W.ALL_OPS:
            check(x, dtype, op)
            check(x, dtype, op, offset=1)


# ---------------------------------------------------------------------------
# The pages' test shapes.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", W.DTYPES)
def test_golden_long_axis_300x4(dtype):
    with open(os.path.join(GOLDEN, "onnxruntime_31694_long_axis_300x4.json")) as f:
        fx = json.load(f)
    x = W.encode(np.array(fx["rows"], dtype=np.float64), dtype)
    for op in W.OPS:
        idx, _ = run(x, dtype, op)
        assert list(idx) == fx["expected"][op]
        for bpr in (1, 2):
            idx, _ = run(x, dtype, op, plan=forced_plan("split", bpr=bpr, grid_rows=4))
            assert list(idx) == fx["expected"][op]


def test_golden_first_index_65536():
    with open(os.path.join(GOLDEN, "onnxruntime_31694_first_index_65536.json")) as f:
        fx = json.load(f)
    rng = np.random.Generator(np.random.PCG64(fx["seed"]))
    row = rng.standard_normal(fx["cols"]).astype(np.float32)
    row[fx["inf_positions"]] = np.inf
    idx, _ = run(row.reshape(1, -1), "f32", "max")
    assert idx[0] == fx["expected_max"]


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_golden_last_index(dtype):
    with open(os.path.join(GOLDEN, "onnx_select_last_index.json")) as f:
        fx = json.load(f)
    from test_oracle import _token
    raw_t = oracle.RAW_NP[dtype]
    for case in fx["cases"]:
        x = np.array([[_token(t, dtype) for t in case["row"]]], dtype=raw_t)
        for op in W.LAST_OPS:
            for plan in (None, forced_plan("split", bpr=2, grid_rows=1, block=32),
                         forced_plan("rows", group=4, vec=0, grid=1)):
                idx, _ = run(x, dtype, op, plan=plan)
                assert idx[0] == case[op], (case["what"], op, plan)


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_operator_shapes(dtype):
    """#32092 Testing: {3, 40000} and {2, 202048}; #31694 Testing: lengths on
    both sides of a 256-wide block and rows 1..300."""
    for rows, cols in [(3, 40000), (2, 202048)]:
        for op in W.OPS:
            check(W.fuzz_rows(dtype, rows, cols, seed=rows, p_special=0.001), dtype, op)
    for cols in (1, 2, 255, 256, 257, 1000, 129280):
        for rows in (1, 300):
            if rows * cols > 4_000_000:
                continue
            for op in W.OPS:
                check(W.fuzz_rows(dtype, rows, cols, seed=cols, p_special=0.01), dtype, op)
