"""GPU checks of the boundary's contract: scratch validation, self-resetting
counters, a dirtied partials region, CUDA graph capture and replay, streams,
empty and maximal inputs (onnxruntime #32092 Testing: undersized and unaligned
buffers, a dirtied intermediate buffer, graph capture with repeated replay,
and a [1, INT_MAX] fp16 row)."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import _lib  # noqa: E402

from gpu_util import forced_plan, raw_equal, run, to_device  # noqa: E402

INT_MAX = 2**31 - 1


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def test_bounded_wait_expires_and_is_reported():
    """A bulk copy whose barrier never completes (test flag): the kernel's
    bounded wait runs out, the kernel returns, the host reads ARGR_ETIMEOUT,
    and the next call is unaffected."""
    x = torch.randn(64, 4096, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert A.argreduce_read_error(0, s) == _lib.ARGR_OK
    plan = forced_plan("stream", group=32, stages=2, stage_bytes=16384, block=128, grid=4, expire=True)
    A.argreduce_with_plan(plan, x, "max")
    assert A.argreduce_read_error(0, s) == _lib.ARGR_ETIMEOUT
    assert A.argreduce_read_error(0, s) == _lib.ARGR_OK  # cleared
    idx, _ = A.argreduce_with_plan(forced_plan("stream", group=32, stages=2, stage_bytes=16384, block=128, grid=4),
                                   x, "max")
    torch.cuda.synchronize()
    assert (idx.cpu().numpy() == oracle.argreduce(x.cpu().numpy(), "f32", "max")[0]).all()
    assert A.argreduce_read_error(0, s) == _lib.ARGR_OK


def test_stream_plan_validation():
    x = torch.randn(4, 1001, device="cuda")  # rows not 16-byte aligned
    with pytest.raises(A.ArgreduceError):
        A.argreduce_with_plan(forced_plan("stream", group=32), x, "max")
    y = torch.randn(4, 8192, device="cuda")
    for bad in (dict(group=4, stage_bytes=8192),        # a row wider than a stage needs the whole warp
                dict(group=32, stages=5),
                dict(group=32, stage_bytes=1000),
                dict(group=32, stage_bytes=65536, stages=4, block=512)):  # too much shared memory
        with pytest.raises(A.ArgreduceError):
            A.argreduce_with_plan(forced_plan("stream", **bad), y, "max")
    split = forced_plan("split", bpr=1, grid_rows=4)
    split.flags |= _lib.ARGR_PLAN_TEST_EXPIRE
    with pytest.raises(A.ArgreduceError):  # the test flag only exists on the stream path
        A.argreduce_with_plan(split, y, "max")


def test_rows_zero_and_one_col():
    x = torch.empty((0, 17), dtype=torch.float32, device="cuda")
    idx, _ = A.argreduce(x, "max")
    assert idx.shape == (0,)
    x = W.fuzz_rows("f32", 1000, 1, seed=1)
    i, v = run(x, "f32", "max")
    assert (i == 0).all() and raw_equal(v, x[:, 0])


def test_scratch_errors():
    rows, cols = 2, 3_000_000  # too wide for one cluster: split over the device, with scratch
    x = torch.randn(rows, cols, device="cuda")
    out = torch.empty(rows, dtype=torch.int64, device="cuda")
    need = A.argreduce_scratch_bytes(rows, cols, "f32", "max")
    assert need > 0
    buf = torch.zeros(need + 64, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    f = _lib.argreduce_raw
    assert f(x.data_ptr(), "f32", rows, cols, "max", out.data_ptr(), 0, 0, 0, s) == _lib.ARGR_ESCRATCH
    assert f(x.data_ptr(), "f32", rows, cols, "max", out.data_ptr(), 0, buf.data_ptr(), need - 1, s) == \
        _lib.ARGR_ESCRATCH
    assert f(x.data_ptr(), "f32", rows, cols, "max", out.data_ptr(), 0, buf.data_ptr() + 8, need, s) == \
        _lib.ARGR_ESCRATCH
    assert A.argreduce_scratch_init(buf.data_ptr(), need, s) == _lib.ARGR_OK
    assert f(x.data_ptr(), "f32", rows, cols, "max", out.data_ptr(), 0, buf.data_ptr(), need, s) == _lib.ARGR_OK
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == oracle.argreduce(x.cpu().numpy(), "f32", "max")[0]).all()
    assert A.argreduce_read_error(buf.data_ptr(), s) == _lib.ARGR_OK


def test_forced_plan_validation():
    x = torch.randn(4, 1000, device="cuda")
    bad = [
        forced_plan("rows", group=3),                       # not a power of two
        forced_plan("rows", group=4, vec=1),                # unroll 5 (set below) is not offered
        forced_plan("split", bpr=4, grid_rows=2),           # split rows may not loop
        forced_plan("split", bpr=0, grid_rows=4),
        forced_plan("split", bpr=2, grid_rows=4, block=48),  # not a multiple of 32
        forced_plan("split", bpr=2, grid_rows=4, unroll=3),
        forced_plan("cluster", cluster=17, grid_rows=4),
        forced_plan("cluster", cluster=1, grid_rows=4),
        forced_plan("rows", group=8, vec=1, pipeline=True),             # pipelined: 16 or 32 lanes per row
        forced_plan("rows", group=32, vec=0, pipeline=True),            # pipelined: vector loads only
        forced_plan("rows", group=32, vec=1, block=512, pipeline=True),  # pipelined: at most 256 threads
        forced_plan("split", bpr=1, grid_rows=4),                       # pipelined: rows path only (set below)
    ]
    bad[1].unroll = 5
    bad[-1].flags |= _lib.ARGR_PLAN_PIPELINE
    for p in bad:
        with pytest.raises(A.ArgreduceError) as e:
            A.argreduce_with_plan(p, x, "max")
        assert e.value.status in (_lib.ARGR_EINVAL, _lib.ARGR_EUNSUPPORTED)
    # vector loads on rows that are not 16-byte aligned are refused
    x2 = torch.randn(4, 1001, device="cuda")
    with pytest.raises(A.ArgreduceError):
        A.argreduce_with_plan(forced_plan("rows", group=4, vec=1), x2, "max")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f64"])
def test_dirtied_partials_and_repeat(dtype):
    """Counters reset themselves; garbage in the partials region is harmless."""
    rows, cols = 4, 2_500_000  # split over the device: partials and counters in scratch
    c = W.Case("t", rows, cols, dtype, "max", "batch_logits", 3001)
    x = W.make(c)
    eidx, _, _ = oracle.argreduce(x, dtype, "max")
    xd, _k = to_device(x, dtype)
    plan = A.argreduce_plan(rows, cols, dtype, "max")
    assert plan.blocks_per_row > 1
    scratch = A.Scratch(nbytes=plan.scratch_bytes)
    from row_wise_arg_gb300._lib import argreduce_plan_scratch_bytes
    # partials start after the 256-byte header and 2048 row-slot counters
    off = 256 + 4 * 2048
    assert argreduce_plan_scratch_bytes(plan, rows) <= scratch.nbytes
    for it in range(5):
        scratch.buf[off:].fill_(0xFF if it % 2 else 0xA5)  # dirty the partials only
        idx, _ = A.argreduce(xd, "max", dtype=dtype, scratch=scratch)
        torch.cuda.synchronize()
        assert (idx.cpu().numpy() == eidx).all()
    # the counters are back at zero after every call
    counters = scratch.buf[256:256 + 4 * plan.grid_rows].cpu()
    assert (counters == 0).all()


def test_shared_scratch_across_plans():
    """Calls with different split plans share one scratch buffer; a call's
    partials never disturb another call's arrival counters."""
    shapes = [(1, 300000), (500, 3000), (7, 90001), (1200, 5000), (1, 33), (300, 20000)]
    data = [W.fuzz_rows("f32", r, c, seed=r * 7 + c, p_special=0.01) for r, c in shapes]
    exp = [oracle.argreduce(x, "f32", "max")[0] for x in data]
    dev = [to_device(x, "f32")[0] for x in data]
    scratch = A.Scratch()
    for rep in range(3):
        for k in (list(range(len(shapes))) if rep % 2 == 0 else list(reversed(range(len(shapes))))):
            idx, _ = A.argreduce(dev[k], "max", scratch=scratch)
            torch.cuda.synchronize()
            assert (idx.cpu().numpy() == exp[k]).all(), (rep, shapes[k])


@pytest.mark.parametrize("path", ["planner", "split", "cluster", "rows"])
def test_graph_capture_replay(path):
    """Capture one call into a CUDA graph and replay it 100 times with new
    input contents each time; every replay matches the oracle."""
    rows, cols = 6, 150001
    dtype = "f32"
    if path == "planner":
        plan = A.argreduce_plan(rows, cols, dtype, "max")
    elif path == "split":
        plan = forced_plan("split", bpr=40, grid_rows=rows)
    elif path == "cluster":
        plan = forced_plan("cluster", cluster=8, grid_rows=rows)
    else:
        plan = forced_plan("rows", group=32, vec=0, grid=2)
    xs = [W.fuzz_rows(dtype, rows, cols, seed=900 + k, p_special=0.001) for k in range(4)]
    exp = [oracle.argreduce(x, dtype, "max")[0] for x in xs]
    xd = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    out = torch.empty(rows, dtype=torch.int64, device="cuda")
    scratch = A.Scratch(nbytes=max(4096, plan.scratch_bytes))
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        A.argreduce_with_plan(plan, xd, "max", out_idx=out, scratch=scratch, stream=stream)  # warm-up
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            A.argreduce_with_plan(plan, xd, "max", out_idx=out, scratch=scratch, stream=stream)
    host = [torch.from_numpy(x) for x in xs]
    for k in range(100):
        xd.copy_(host[k % 4])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert (out.cpu().numpy() == exp[k % 4]).all(), f"replay {k}"


def test_push_merge_wait_expires_and_is_reported():
    """The push merge's CTA 0 waits (bounded) for the cluster's candidates.
    Under the test flag its barrier expects 16 bytes more than arrive: the
    wait runs out after 2 ms, the kernel returns, the host reads
    ARGR_ETIMEOUT, and the next call is exact."""
    x = W.fuzz_rows("f32", 3, 50000, seed=5, p_special=0.001)
    xd, _keep = to_device(x, "f32")
    s = torch.cuda.current_stream().cuda_stream
    assert A.argreduce_read_error(0, s) == _lib.ARGR_OK
    plan = forced_plan("cluster", cluster=4, grid_rows=3)
    plan.flags |= _lib.ARGR_PLAN_TEST_EXPIRE
    A.argreduce_with_plan(plan, xd, "max")
    assert A.argreduce_read_error(0, s) == _lib.ARGR_ETIMEOUT
    assert A.argreduce_read_error(0, s) == _lib.ARGR_OK  # cleared
    idx, _ = run(x, "f32", "max", plan=forced_plan("cluster", cluster=4, grid_rows=3))
    assert (idx == oracle.argreduce(x, "f32", "max")[0]).all()
    bad = forced_plan("cluster", cluster=4, grid_rows=2)  # rows loop: no push wait to expire
    bad.flags |= _lib.ARGR_PLAN_TEST_EXPIRE
    with pytest.raises(A.ArgreduceError):
        A.argreduce_with_plan(bad, xd, "max")


def test_default_scratch_graph_after_growth():
    """A graph captured with the stream's default scratch stays valid after a
    larger call on the same stream grows that scratch: the old buffer is kept
    alive, so 100 replays (new inputs each time) all match the oracle."""
    rows, cols, dtype = 4, 120001, "f32"
    stream = torch.cuda.Stream()
    xs = [W.fuzz_rows(dtype, rows, cols, seed=700 + k, p_special=0.001) for k in range(4)]
    exp = [oracle.argreduce(x, dtype, "max")[0] for x in xs]
    xd = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    out = torch.empty(rows, dtype=torch.int64, device="cuda")
    plan = forced_plan("split", bpr=20, grid_rows=rows)  # a split plan: uses scratch
    with torch.cuda.stream(stream):
        xd.copy_(torch.from_numpy(xs[0]))
        A.argreduce_with_plan(plan, xd, "max", out_idx=out, stream=stream)  # default scratch, warm-up
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            A.argreduce_with_plan(plan, xd, "max", out_idx=out, stream=stream)
        # a larger problem on the same stream grows the default scratch
        big_rows = 1500
        big = W.fuzz_rows(dtype, big_rows, 40000, seed=77, p_special=0.001)
        bigd = torch.from_numpy(big).cuda()
        big_plan = forced_plan("split", bpr=12, grid_rows=big_rows)
        assert big_plan.grid_rows * big_plan.blocks_per_row * 16 > 4 * plan.grid_rows * plan.blocks_per_row * 16
        bi, _ = A.argreduce_with_plan(big_plan, bigd, "max", stream=stream)
        # had the first buffer gone back to the allocator, one of these would
        # likely take its place and fill its counters with junk
        junk = [torch.full((16384,), 0x7F, dtype=torch.uint8, device="cuda") for _ in range(64)]
        stream.synchronize()
    assert (bi.cpu().numpy() == oracle.argreduce(big, dtype, "max")[0]).all()
    host = [torch.from_numpy(x) for x in xs]
    for k in range(100):
        xd.copy_(host[k % 4])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert (out.cpu().numpy() == exp[k % 4]).all(), f"replay {k}"
    del junk


def test_scratch_growth_refused_inside_capture():
    """Growing a Scratch inside a capture would record its preparing memset
    into the graph; the binding refuses with a clear error instead."""
    s = A.Scratch()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with pytest.raises(RuntimeError, match="before a CUDA graph capture"):
            with torch.cuda.graph(g, stream=stream):
                s.ensure(1 << 16, stream.cuda_stream)


def test_streams_independent():
    """Two streams with their own scratch run concurrently and both match."""
    a = W.fuzz_rows("f32", 16, 300000, seed=3, p_special=0.001)
    b = W.fuzz_rows("f32", 16, 300000, seed=4, p_special=0.001)
    da, _ka = to_device(a, "f32")
    db, _kb = to_device(b, "f32")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    sa, sb = A.Scratch(), A.Scratch()
    torch.cuda.synchronize()
    for _ in range(20):
        ia, _ = A.argreduce(da, "max", scratch=sa, stream=s1)
        ib, _ = A.argreduce(db, "max", scratch=sb, stream=s2)
    torch.cuda.synchronize()
    assert (ia.cpu().numpy() == oracle.argreduce(a, "f32", "max")[0]).all()
    assert (ib.cpu().numpy() == oracle.argreduce(b, "f32", "max")[0]).all()


def test_int_max_row_f16():
    """[1, INT_MAX] fp16 (4 GiB): a property check at the widest admitted row.
    Zeros with planted values near both ends; the expected indices follow
    from the construction."""
    free, _ = torch.cuda.mem_get_info()
    if free < 6 * 2**30:
        pytest.skip("needs ~5 GiB of device memory")
    n = INT_MAX
    x = torch.zeros((1, n), dtype=torch.float16, device="cuda")
    x[0, n - 3] = 1.0
    x[0, n - 1] = 1.0
    x[0, 5] = -1.0
    x[0, n - 2] = -1.0
    plans = [None, forced_plan("split", bpr=3, grid_rows=1, block=1024, unroll=8),
             forced_plan("split", bpr=1, grid_rows=1)]
    for p in plans:
        for op, want in (("max", n - 3), ("min", 5)):
            if p is None:
                idx, val = A.argreduce(x, op, with_values=True)
            else:
                idx, val = A.argreduce_with_plan(p, x, op, with_values=True)
            torch.cuda.synchronize()
            assert int(idx[0]) == want, (p, op)
    x[0, 0] = float("nan")
    idx, _ = A.argreduce(x, "max")
    torch.cuda.synchronize()
    assert int(idx[0]) == 0
    del x
    torch.cuda.empty_cache()


def test_concurrent_host_threads():
    """Four host threads call the library at once (ctypes releases the GIL),
    each on its own stream and scratch: cluster launches with their
    co-scheduling check, raised shared-memory limits (bulk cluster plans, the
    stashed scan) and split scans share the per-device launch records without
    corrupting them or each other's results."""
    import threading
    xs = [W.fuzz_rows("f32", 3, 200001 + 17 * k, seed=70 + k) for k in range(4)]
    want = [oracle.argreduce(x, "f32", "max")[0] for x in xs]
    want_cum = [oracle.cumreduce(np.ascontiguousarray(x[:, :50000]), "f32", "min")[0] for x in xs]
    dev = [torch.from_numpy(x).cuda() for x in xs]
    dev_cum = [torch.from_numpy(np.ascontiguousarray(x[:, :50000])).cuda() for x in xs]
    errors = []

    def stash_plan():
        p = _lib.argr_plan()
        p.path, p.block, p.cluster, p.blocks_per_row, p.grid_rows, p.flags = _lib.ARGR_PATH_CUM_SPLIT, 256, 1, 8, 3, 1 | 8
        return p

    def worker(k):
        try:
            s = torch.cuda.Stream()
            sc = A.Scratch()
            plans = [None, forced_plan("cluster", cluster=16, block=512, unroll=8, grid_rows=3),
                     forced_plan("cluster", cluster=8, block=256, unroll=4, grid_rows=3, bulk=True)]
            with torch.cuda.stream(s):
                for it in range(20):
                    p = plans[(it + k) % 3]
                    if p is None:
                        idx, _ = A.argreduce(dev[k], "max", scratch=sc, stream=s)
                    else:
                        idx, _ = A.argreduce_with_plan(p, dev[k], "max", scratch=sc, stream=s)
                    ci, _ = A.argreduce_cum(dev_cum[k], "min", scratch=sc, stream=s, with_values=False,
                                            plan=stash_plan() if it % 2 else None)
                    s.synchronize()
                    if not (idx.cpu().numpy() == want[k]).all() or not (ci.cpu().numpy() == want_cum[k]).all():
                        errors.append((k, it))
                        return
        except Exception as e:  # surfaced below
            errors.append((k, repr(e)))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
