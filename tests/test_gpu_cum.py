"""GPU parity of cummax / cummin with indices (argreduce_cum) against the CPU
oracle, bit for bit: the Paddle-issue workloads at full size, and every
forced geometry (one CTA per row with row loops, clusters of 2..16 CTAs per
row, split scans of 2..1024 chunks exchanging aggregates through scratch,
tile widths from 32 to 1024 threads) on special-value rows of every element
type, including leading NaNs and the integer extremes; plus the split scan's
scratch handling (shared with argreduce, graph replay, a forced expiry)."""
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


def split_plan(chunks, block=256, rows=1, flags=_lib.ARGR_PLAN_PDL):
    p = _lib.argr_plan()
    p.path = _lib.ARGR_PATH_CUM_SPLIT
    p.block = block
    p.cluster = 1
    p.blocks_per_row = chunks
    p.grid_rows = rows
    p.flags = flags
    return p


STASH = 8  # ARGR_PLAN_STASH


def stream_plan(cols, block=256, rows=1, grid=16, flags=_lib.ARGR_PLAN_PDL):
    p = _lib.argr_plan()
    p.path = _lib.ARGR_PATH_CUM_STREAM
    p.block = block
    p.cluster = 1
    p.blocks_per_row = -(-cols // (block * 7))  # tiles per row
    p.grid_rows = grid  # CTAs
    p.flags = flags
    return p
LOOKBACK = 16  # ARGR_PLAN_LOOKBACK


def run_cum(x, dtype, op, plan=None, scratch=None, offset=0):
    """The scan of x on the GPU; `offset` elements of padding in front move
    the base pointer off its allocation's alignment."""
    flat = np.ascontiguousarray(x).view(VIEW[dtype]).reshape(-1)
    buf = torch.zeros(flat.size + offset, dtype=getattr(torch, str(flat.dtype)), device="cuda")
    buf[offset:] = torch.from_numpy(flat).cuda()
    xd = buf[offset:].view(x.shape)
    idx, val = A.argreduce_cum(xd, op, dtype=dtype, plan=plan, scratch=scratch)
    torch.cuda.synchronize()
    raw_t = oracle.RAW_NP[dtype]
    return idx.cpu().numpy(), val.cpu().numpy().view(raw_t)


def check_cum(x, dtype, op, plan=None, scratch=None, offset=0):
    idx, val = run_cum(x, dtype, op, plan, scratch, offset)
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


@pytest.mark.parametrize("case", W.config_cases(7) + W.config_cases(8), ids=lambda c: c.name)
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
            for chunks, block in ((2, 32), (3, 1024), (7, 64), (64, 256)):
                if rows * chunks <= 1024:  # chunks > cols leaves some chunks empty
                    check_cum(x, dtype, op, plan=split_plan(chunks, block, rows, flags=chunks % 2))
            # streaming scan: tiles in ticket order over a fixed grid (1 CTA walks every tile)
            for block, grid in ((32, 1), (128, 3), (1024, 16), (64, 304)):
                check_cum(x, dtype, op, plan=stream_plan(cols, block, rows, grid, flags=grid % 2))
            # decoupled look-back (inclusive prefixes), chunks of up to a tile and beyond
            for chunks, block in ((2, 64), (3, 1024), (9, 32), (100, 128)):
                if rows * chunks * 2 <= 65536:
                    check_cum(x, dtype, op, plan=split_plan(chunks, block, rows, flags=(chunks % 2) | LOOKBACK))
            # stashed chunks (bulk copies of the aligned middle, plain loads of the ends)
            for chunks, block, off in ((1, 512, 0), (3, 128, 1), (5, 1024, 3), (64, 64, 2)):
                if -(-cols // chunks) * W.ELEM_SIZE[dtype] <= 80 * 1024:
                    check_cum(x, dtype, op, plan=split_plan(chunks, block, rows, flags=1 | STASH), offset=off)


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


def test_cum_split_many_chunks():
    # the planner's split at the pages' lengths, and the largest record count
    for n, dtype in ((65536, "i64"), (131072, "i64"), (1 << 20, "f32"), (5 << 20, "bf16")):
        x = cum_rows(dtype, 1, n, seed=n)
        assert A.argreduce_cum_plan(1, n, dtype, "max").as_dict()["path_name"] == "cum_split"
        check_cum(x, dtype, "max")
    x = cum_rows("f64", 2, 300001, seed=5)
    check_cum(x, "f64", "min", plan=split_plan(512, 128, rows=2))
    x = cum_rows("f16", 1, 300001, seed=7)
    check_cum(x, "f16", "max", plan=split_plan(1024, 32, rows=1))
    x = cum_rows("i32", 1024, 40, seed=6)
    check_cum(x, "i32", "max", plan=split_plan(1, 32, rows=1024))


def test_cum_split_scratch_shared_with_argreduce_and_graphs():
    """One scratch buffer serves argreduce's split path (per-row counters that
    must stay zero between calls) and the split scan (records in the same
    region, cleared by each launch's last CTA) one call after the other, on
    one stream, eagerly and replayed from CUDA graphs."""
    from gpu_util import forced_plan
    sc = A.Scratch()
    xs = cum_rows("f32", 3, 70001, seed=11)
    xr = W.fuzz_rows("f32", 3, 3_000_000, seed=12)
    er, _, _ = oracle.argreduce(xr, "f32", "max")
    xrd = torch.from_numpy(xr).cuda()
    rplan = forced_plan("split", bpr=8, grid_rows=3)
    xsd = torch.from_numpy(xs).cuda()
    eidx, _ = oracle.cumreduce(xs, "f32", "min")
    splan = split_plan(40, 256, rows=3)
    for _ in range(3):
        idx, _ = A.argreduce_cum(xsd, "min", plan=splan, scratch=sc, with_values=False)
        got, _ = A.argreduce_with_plan(rplan, xrd, "max", scratch=sc)
        torch.cuda.synchronize()
        assert (idx.cpu().numpy() == eidx).all() and (got.cpu().numpy() == er).all()
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    s = torch.cuda.Stream()
    out_i = torch.empty(3, 70001, dtype=torch.int64, device="cuda")
    out_r = torch.empty(3, dtype=torch.int64, device="cuda")
    with torch.cuda.stream(s):
        A.argreduce_cum(xsd, "min", plan=splan, scratch=sc, out_idx=out_i, with_values=False, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            A.argreduce_cum(xsd, "min", plan=splan, scratch=sc, out_idx=out_i, with_values=False, stream=s)
            A.argreduce_with_plan(rplan, xrd, "max", scratch=sc, out_idx=out_r, stream=s)
            A.argreduce_cum(xsd, "min", scratch=sc, out_idx=out_i, with_values=False, stream=s)
        for _ in range(5):
            out_i.zero_()
            out_r.zero_()
            g.replay()
            s.synchronize()
            assert (out_i.cpu().numpy() == eidx).all() and (out_r.cpu().numpy() == er).all()
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK


def test_cum_split_bounded_wait_expires():
    """Chunk 0 never publishes its record (test flag): every other CTA's wait
    for it gives up after 2 ms, the expiry is reported as ARGR_ETIMEOUT, and
    the counters and records are left clean, so the next call is exact."""
    sc = A.Scratch()
    x = cum_rows("i64", 2, 50000, seed=13)
    xd = torch.from_numpy(x).cuda()
    A.argreduce_cum(xd, "max", plan=split_plan(9, 128, rows=2, flags=_lib.ARGR_PLAN_TEST_EXPIRE), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_ETIMEOUT
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK  # cleared
    check_cum(x, "i64", "max", plan=split_plan(9, 128, rows=2), scratch=sc)
    check_cum(x, "i64", "max", plan=split_plan(5, 256, rows=2), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK


def test_cum_split_rejections():
    x = torch.zeros(4, 100000, device="cuda")
    o = torch.empty(4, 100000, dtype=torch.int64, device="cuda")
    p = split_plan(8, 256, rows=4)
    assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, 0, 0, 0, p) == \
        _lib.ARGR_ESCRATCH  # no scratch
    sc = A.Scratch(nbytes=4096)
    assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, sc.ptr + 8, 4000, 0,
                                  p) == _lib.ARGR_ESCRATCH  # misaligned
    assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, sc.ptr, 200, 0,
                                  p) == _lib.ARGR_ESCRATCH  # too small
    # more than 1024 chunks keep their records 1 MiB into the scratch buffer
    assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, sc.ptr, 4096, 0,
                                  split_plan(257, 256, rows=4)) == _lib.ARGR_ESCRATCH
    for bad in (split_plan(16385, 256, rows=4), split_plan(8, 256, rows=3), split_plan(8, 48, rows=4),
                split_plan(8, 256, rows=4, flags=_lib.ARGR_PLAN_BULK),
                split_plan(1, 256, rows=4, flags=STASH)):  # a 400 KB chunk does not fit the stash
        assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, sc.ptr, 4096, 0,
                                      bad) == _lib.ARGR_EINVAL
    bad = split_plan(8, 256, rows=4)
    bad.cluster = 2
    assert _lib.argreduce_cum_raw(x.data_ptr(), "f32", 4, 100000, "max", o.data_ptr(), 0, sc.ptr, 4096, 0,
                                  bad) == _lib.ARGR_EINVAL
    torch.cuda.synchronize()


def test_cum_int_max_row_f16():
    """[1, INT32_MAX] fp16, the widest admitted row (4 GiB in, 16 GiB of
    indices, 4 GiB of values): zeros with a planted ladder of maxima and two
    minima, so every output is known by construction; checked at the ladder's
    edges, the last element and random positions, under the planner's split
    scan, a 1024-chunk split, a cluster and a single CTA."""
    free, _ = torch.cuda.mem_get_info()
    if free < 30 * 2**30:
        pytest.skip("needs ~26 GiB of device memory")
    n = 2**31 - 1
    p1, p2, p3 = 1000, 2**30 + 7, n - 2
    q1 = 5
    x = torch.zeros((1, n), dtype=torch.float16, device="cuda")
    x[0, p1], x[0, p2], x[0, p3] = 1.0, 2.0, 3.0
    x[0, q1], x[0, n - 1] = -1.0, -2.0
    out_i = torch.empty((1, n), dtype=torch.int64, device="cuda")
    out_v = torch.empty((1, n), dtype=torch.float16, device="cuda")
    rng = np.random.Generator(np.random.PCG64(2**31))
    pos = np.unique(np.concatenate([rng.integers(0, n, size=2000),
                                    [0, 1, q1 - 1, q1, q1 + 1, p1 - 1, p1, p1 + 1, p2 - 1, p2, p2 + 1,
                                     p3 - 1, p3, p3 + 1, n - 2, n - 1]]))
    pos = pos[(pos >= 0) & (pos < n)]
    pos_t = torch.from_numpy(pos).cuda()

    def want(op):
        if op == "max":
            return np.select([pos < p1, pos < p2, pos < p3], [0, p1, p2], p3)
        return np.select([pos < q1, pos < n - 1], [0, q1], n - 1)

    vals = {0: 0.0, p1: 1.0, p2: 2.0, p3: 3.0, q1: -1.0, n - 1: -2.0}
    plans = [None, split_plan(1024, 512, rows=1), cum_plan(16, 1024, grid=1), cum_plan(1, 1024, grid=1)]
    for plan in plans:
        for op in ("max", "min"):
            out_i.fill_(-7)
            A.argreduce_cum(x, op, out_idx=out_i, out_val=out_v, plan=plan)
            torch.cuda.synchronize()
            got = out_i[0, pos_t].cpu().numpy()
            w = want(op)
            assert (got == w).all(), (plan.as_dict() if plan is not None else "planner", op,
                                      pos[got != w][:5], got[got != w][:5], w[got != w][:5])
            gv = out_v[0, pos_t].float().cpu().numpy()
            assert (gv == np.array([vals[int(i)] for i in w], dtype=np.float32)).all()
    del x, out_i, out_v
    torch.cuda.empty_cache()


def test_cum_stash_and_large_record_region():
    """Split scans of more than 1024 chunks keep their records 1 MiB into the
    scratch buffer: with and without stashed chunks, from misaligned bases,
    alternating with argreduce's split path on one buffer, and 80 KiB
    stashes of a 96 MiB row."""
    from gpu_util import forced_plan
    sc = A.Scratch()
    x = cum_rows("f32", 2, 300001, seed=21)
    for plan in (split_plan(1000, 128, rows=2, flags=1 | STASH), split_plan(1000, 64, rows=2),
                 split_plan(2500, 32, rows=2, flags=STASH), split_plan(16, 512, rows=2, flags=STASH)):
        for off in (0, 1):
            check_cum(x, "f32", "max", plan=plan, scratch=sc, offset=off)
    xr = W.fuzz_rows("bf16", 4, 1_000_000, seed=22)
    er, _, _ = oracle.argreduce(xr, "bf16", "min")
    xrd = torch.from_numpy(xr.view(np.int16)).cuda()
    rplan = forced_plan("split", bpr=16, grid_rows=4)
    for _ in range(2):
        check_cum(x, "f32", "min", plan=split_plan(1500, 128, rows=2, flags=STASH), scratch=sc)
        got, _ = A.argreduce_with_plan(rplan, xrd, "min", dtype="bf16", scratch=sc)
        torch.cuda.synchronize()
        assert (got.cpu().numpy() == er).all()
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    # stashed 80 KiB chunks of 12M int64 elements (96 MiB, 1229 chunks) in one row, from an odd base
    n = 12 << 20
    big = cum_rows("i64", 1, n, seed=23)
    check_cum(big, "i64", "max", plan=split_plan(1229, 512, rows=1, flags=1 | STASH), offset=1)
    # the forced expiry with stashed chunks
    # (16 chunks of a 300001-element f32 row: 75 KB each, within the 80 KiB stash)
    A.argreduce_cum(torch.from_numpy(x).cuda(), "max", plan=split_plan(16, 256, rows=2, flags=STASH | 4),
                    scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_ETIMEOUT
    check_cum(x, "f32", "max", plan=split_plan(16, 256, rows=2, flags=STASH), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK


def test_split_partials_stay_below_the_scan_records():
    """argreduce's split partials may not reach 1 MiB into the scratch
    buffer, where large split scans keep their records."""
    from gpu_util import forced_plan
    x = torch.zeros(2048, 100000, device="cuda")
    o = torch.empty(2048, dtype=torch.int64, device="cuda")
    sc = A.Scratch(nbytes=4 << 20)
    ok = forced_plan("split", bpr=31, grid_rows=2048)   # 63488 partials: below 1 MiB
    bad = forced_plan("split", bpr=32, grid_rows=2048)  # 65536 partials: beyond
    assert _lib.argreduce_with_plan_raw(ok, x.data_ptr(), "f32", 2048, 100000, "max", o.data_ptr(), 0, sc.ptr,
                                        sc.nbytes, 0) == _lib.ARGR_OK
    assert _lib.argreduce_with_plan_raw(bad, x.data_ptr(), "f32", 2048, 100000, "max", o.data_ptr(), 0, sc.ptr,
                                        sc.nbytes, 0) == _lib.ARGR_EINVAL
    torch.cuda.synchronize()


def test_cum_lookback_long_rows_and_scratch():
    """The decoupled look-back at large chunk counts (windows of one chunk per
    thread, several windows back), one-tile chunks of long rows, the forced
    expiry, and one scratch buffer shared with argreduce's split path."""
    from gpu_util import forced_plan
    sc = A.Scratch()
    x = cum_rows("f32", 2, 300001, seed=31)
    for chunks, block in ((4096, 32), (1000, 64), (300, 128)):
        for off in (0, 3):
            check_cum(x, "f32", "max", plan=split_plan(chunks, block, rows=2, flags=1 | LOOKBACK), scratch=sc,
                      offset=off)
    for dtype, n, block in (("i64", 1 << 20, 512), ("f64", 3 << 20, 256), ("bf16", 1 << 24, 512)):
        big = cum_rows(dtype, 1, n, seed=n % 1000)
        chunks = -(-n // (block * 7))  # one tile per chunk
        check_cum(big, dtype, "min", plan=split_plan(chunks, block, rows=1, flags=1 | LOOKBACK), scratch=sc)
    xi = cum_rows("i32", 16, 70000, seed=32)
    check_cum(xi, "i32", "max", plan=split_plan(1024, 64, rows=16, flags=LOOKBACK), scratch=sc)
    xr = W.fuzz_rows("f32", 3, 2_000_000, seed=33)
    er, _, _ = oracle.argreduce(xr, "f32", "max")
    got, _ = A.argreduce_with_plan(forced_plan("split", bpr=12, grid_rows=3), torch.from_numpy(xr).cuda(), "max",
                                   scratch=sc)
    torch.cuda.synchronize()
    assert (got.cpu().numpy() == er).all()
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    A.argreduce_cum(torch.from_numpy(x).cuda(), "max", plan=split_plan(600, 128, rows=2, flags=LOOKBACK | 4),
                    scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_ETIMEOUT
    check_cum(x, "f32", "max", plan=split_plan(600, 128, rows=2, flags=LOOKBACK), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    assert _lib.argreduce_cum_raw(0x10000, "f32", 2, 300001, "max", 0x10000, 0, sc.ptr, sc.nbytes, 0,
                                  split_plan(8, 128, rows=2, flags=LOOKBACK | STASH)) == _lib.ARGR_EINVAL


def test_cum_stream_long_rows_graphs_and_scratch():
    """The streaming scan on long rows of every width class, from misaligned
    bases, in CUDA-graph replays (the ticket counter must come back to zero
    after every launch), through a forced expiry, and on one scratch buffer
    with argreduce's split path and the split scan."""
    from gpu_util import forced_plan
    sc = A.Scratch()
    for dtype, rows, n, block, grid in (("i64", 1, 1 << 20, 512, 304), ("f64", 2, 3 << 20, 256, 608),
                                        ("bf16", 1, 1 << 24, 512, 304), ("f32", 7, 300001, 128, 1000),
                                        ("i32", 3, 1 << 20, 1024, 152)):
        x = cum_rows(dtype, rows, n, seed=n % 997 + rows)
        check_cum(x, dtype, "min" if rows % 2 else "max", plan=stream_plan(n, block, rows, grid), scratch=sc,
                  offset=rows % 3)
    x = cum_rows("f32", 2, 400001, seed=41)
    xd = torch.from_numpy(x).cuda()
    eidx, _ = oracle.cumreduce(x, "f32", "max")
    xr = W.fuzz_rows("f32", 3, 2_000_000, seed=42)
    er, _, _ = oracle.argreduce(xr, "f32", "max")
    xrd = torch.from_numpy(xr).cuda()
    rplan = forced_plan("split", bpr=12, grid_rows=3)
    s = torch.cuda.Stream()
    out_i = torch.empty(2, 400001, dtype=torch.int64, device="cuda")
    out_r = torch.empty(3, dtype=torch.int64, device="cuda")
    plan = stream_plan(400001, 256, rows=2, grid=300)
    with torch.cuda.stream(s):
        A.argreduce_cum(xd, "max", plan=plan, scratch=sc, out_idx=out_i, with_values=False, stream=s)
        A.argreduce_with_plan(rplan, xrd, "max", scratch=sc, out_idx=out_r, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            A.argreduce_cum(xd, "max", plan=plan, scratch=sc, out_idx=out_i, with_values=False, stream=s)
            A.argreduce_with_plan(rplan, xrd, "max", scratch=sc, out_idx=out_r, stream=s)
            A.argreduce_cum(xd, "max", plan=split_plan(40, 128, rows=2), scratch=sc, out_idx=out_i,
                            with_values=False, stream=s)
            A.argreduce_cum(xd, "max", plan=plan, scratch=sc, out_idx=out_i, with_values=False, stream=s)
        for _ in range(5):
            out_i.zero_()
            out_r.zero_()
            g.replay()
            s.synchronize()
            assert (out_i.cpu().numpy() == eidx).all() and (out_r.cpu().numpy() == er).all()
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    A.argreduce_cum(xd, "max", plan=stream_plan(400001, 256, rows=2, grid=64, flags=4), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_ETIMEOUT
    check_cum(x, "f32", "max", plan=stream_plan(400001, 256, rows=2, grid=64), scratch=sc)
    assert A.argreduce_read_error(sc.ptr, 0) == _lib.ARGR_OK
    bad = stream_plan(400001, 256, rows=2, grid=64)
    bad.blocks_per_row += 1  # not the row's tile count
    assert _lib.argreduce_cum_raw(xd.data_ptr(), "f32", 2, 400001, "max", out_i.data_ptr(), 0, sc.ptr, sc.nbytes, 0,
                                  bad) == _lib.ARGR_EINVAL


def test_scratch_prepared_before_use_on_another_stream():
    """A Scratch made (and zeroed) on torch's current stream and used at once
    on a different stream: torch's streams do not wait for each other, so the
    binding lets the preparing memset finish before it hands the buffer out.
    A split scan (tickets, a done counter, records) and a split reduction
    both depend on that; every call is exact and no wait expires."""
    x = np.random.Generator(np.random.PCG64(44)).integers(-500, 500, size=(1, 1 << 21)).astype(np.int64)
    xd = torch.from_numpy(x).cuda()
    eidx, _ = oracle.cumreduce(x, "i64", "max", want_val=False)
    plan = A.argreduce_cum_plan(1, 1 << 21, "i64", "max")
    assert plan.path == _lib.ARGR_PATH_CUM_SPLIT
    for k in range(3):
        sc = A.Scratch(nbytes=2 << 20)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            idx, _ = A.argreduce_cum(xd, "max", scratch=sc, stream=s, with_values=False)
        assert A.argreduce_read_error(sc.ptr, s.cuda_stream) == _lib.ARGR_OK
        assert (idx.cpu().numpy() == eidx).all(), k


def structured_rows(dtype, rows, cols, kind, seed):
    """Rows whose chunks are all dominated by their carry-in (decreasing,
    constant, an early maximum), none (increasing), or some (steps with ties
    at and around chunk boundaries)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    j = np.arange(cols, dtype=np.float64)
    if kind == "increasing":
        v = j / 8.0
    elif kind == "decreasing":
        v = -j / 8.0
    elif kind == "constant":
        v = np.zeros(cols)
    elif kind == "early_max":
        v = rng.integers(-50, 50, size=cols).astype(np.float64)
        v[3] = 1000.0
    else:  # steps: a new maximum every ~cols/13 elements, repeated ties in between
        v = np.floor(j / max(1, cols // 13)) + (rng.random(cols) < 0.5) * 0.0
    v = np.broadcast_to(v, (rows, cols)) + np.arange(rows)[:, None] * 0.0
    if dtype in ("i32", "i64"):
        return np.ascontiguousarray(np.clip(np.round(v * 8), -2**30, 2**30)).astype(VIEW[dtype])
    if dtype == "f16":
        v = np.clip(v, -60000, 60000)
    return np.ascontiguousarray(W.encode(v, dtype))


@pytest.mark.parametrize("dtype", CUM_DTYPES)
def test_cum_dominated_chunks(dtype):
    """Phase B writes the carry-in without reading a chunk again when the
    carry is at least as good as the chunk's best element, and scans it
    otherwise: rows where every chunk, no chunk, or some chunks are dominated,
    for the split scan (all its variants) and the cluster scan."""
    for kind in ("increasing", "decreasing", "constant", "early_max", "steps"):
        for rows, cols in ((1, 40000), (3, 20011)):
            x = structured_rows(dtype, rows, cols, kind, seed=cols + len(kind))
            for op in ("max", "min"):
                check_cum(x, dtype, op)
                for chunks, block in ((2, 64), (13, 128), (40, 256)):
                    check_cum(x, dtype, op, plan=split_plan(chunks, block, rows))
                    check_cum(x, dtype, op, plan=split_plan(chunks, block, rows, flags=1 | LOOKBACK))
                stash_chunks = 3 if -(-cols // 3) * W.ELEM_SIZE[dtype] <= 80 * 1024 else 6
                check_cum(x, dtype, op, plan=split_plan(stash_chunks, 128, rows, flags=1 | STASH))
                for cluster in (2, 7, 16):
                    check_cum(x, dtype, op, plan=cum_plan(cluster, 128, grid=rows))
                check_cum(x, dtype, op, plan=cum_plan(4, 64, grid=rows + 2))  # spare row slots
