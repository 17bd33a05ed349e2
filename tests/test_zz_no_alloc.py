"""GPU test of argreduce_noalloc(), the entry point that allocates nothing.

Some callers cannot call cudaMalloc: a plugin running inside an inference
engine that owns all device memory and gives the plugin no allocator, a
real-time path that may not make a call that can synchronise the device or
take an unbounded time, or a service that fixes its memory footprint at
start-up. For them argreduce_noalloc() keeps the split-row kernel's scratch in
an array inside the library. This test calls it through the C ABI twice in a
row per problem and requires the CPU oracle's bits (indices and raw values)
on both calls, and the same bits as argreduce() with caller-provided scratch.

It lives in its own file, named to be collected last, and must pass both
alone in a fresh process and after the other GPU tests.
"""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import _lib  # noqa: E402

VIEW = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64}
VAL_T = {"f32": torch.int32, "f16": torch.int16, "bf16": torch.int16, "f64": torch.int64}
RAW = {"f32": np.uint32, "f16": np.uint16, "bf16": np.uint16, "f64": np.uint64}

CASES = [
    (1, 202048, "f32", "max"),        # one row over the whole device
    (8, 202048, "bf16", "min"),       # a batch of rows, each over many CTAs
    (3, 1_000_003, "f64", "max"),     # rows that do not start on 16-byte boundaries
    (2, 40000, "f16", "min"),
    (5, 123457, "f32", "max_last"),   # ties to the last index, ragged tails
    (4, 77777, "bf16", "min_last"),
    (1, 5, "f32", "max"),             # one CTA per row: no scratch used
    (3000, 100, "f32", "min"),        # more rows than one wave: one CTA per row
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def make_rows(rows, cols, dtype, seed):
    """Fuzz rows with special values plus planted ties: every row holds its
    extreme twice, far apart, so first- and last-index ties differ."""
    x = W.fuzz_rows(dtype, rows, cols, seed=seed, p_special=0.001)
    if cols >= 8:
        rng = np.random.Generator(np.random.PCG64(seed + 1))
        big = W.encode(np.array([1e4, -1e4]), dtype)
        for r in range(rows):
            p = np.sort(rng.choice(cols - 1, size=2, replace=False) + 1)
            x[r, p] = big[0] if r % 2 == 0 else big[1]
    return x


def noalloc(xd, rows, cols, dtype, op, stream):
    out_idx = torch.full((rows,), -1, dtype=torch.int64, device="cuda")
    out_val = torch.zeros(rows, dtype=VAL_T[dtype], device="cuda")
    st = _lib.argreduce_noalloc_raw(xd.data_ptr(), dtype, rows, cols, op, out_idx.data_ptr(), out_val.data_ptr(),
                                    stream)
    assert st == _lib.ARGR_OK, _lib.status_string(st)
    return out_idx, out_val


def existing(xd, rows, cols, dtype, op):
    """The existing entry point argreduce() with its own scratch."""
    out_idx = torch.empty(rows, dtype=torch.int64, device="cuda")
    out_val = torch.empty(rows, dtype=VAL_T[dtype], device="cuda")
    need = A.argreduce_scratch_bytes(rows, cols, dtype, op)
    scratch = A.Scratch(nbytes=max(need, 4096))
    stream = torch.cuda.current_stream().cuda_stream
    st = _lib.argreduce_raw(xd.data_ptr(), dtype, rows, cols, op, out_idx.data_ptr(), out_val.data_ptr(),
                            scratch.ptr, scratch.nbytes, stream)
    assert st == _lib.ARGR_OK, _lib.status_string(st)
    torch.cuda.synchronize()
    return out_idx.cpu().numpy(), out_val.cpu().numpy()


@pytest.mark.parametrize("rows,cols,dtype,op", CASES, ids=[f"{r}x{c}_{d}_{o}" for r, c, d, o in CASES])
def test_noalloc_matches_oracle_twice(rows, cols, dtype, op):
    x = make_rows(rows, cols, dtype, seed=rows * 31 + cols)
    eidx, evalue, _ = oracle.argreduce(x, dtype, op)
    xd = torch.from_numpy(x.view(VIEW[dtype])).cuda()
    have_idx, have_val = existing(xd, rows, cols, dtype, op)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out_idx, out_val = noalloc(xd, rows, cols, dtype, op, stream)
        torch.cuda.synchronize()
        got_idx = out_idx.cpu().numpy()
        got_val = out_val.cpu().numpy()
        assert (got_idx == eidx).all(), f"call {call}: indices differ from the oracle"
        assert (got_val.view(RAW[dtype]) == evalue.view(RAW[dtype])).all(), f"call {call}: value bits differ"
        assert (got_idx == have_idx).all() and (got_val == have_val).all(), f"call {call}: differs from argreduce()"


def test_noalloc_graph_replays():
    """Calls after the first may be captured: the counters are back at zero
    after every launch, so each replay of one captured call is exact."""
    rows, cols, dtype, op = 6, 150001, "f32", "max"
    xs = [make_rows(rows, cols, dtype, seed=900 + k) for k in range(3)]
    want = [oracle.argreduce(x, dtype, op)[0] for x in xs]
    xd = torch.from_numpy(xs[0]).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out_idx, _ = noalloc(xd, rows, cols, dtype, op, s.cuda_stream)  # warm-up call outside the capture
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            _lib.argreduce_noalloc_raw(xd.data_ptr(), dtype, rows, cols, op, out_idx.data_ptr(), 0, s.cuda_stream)
    for k in range(6):
        xd.copy_(torch.from_numpy(xs[k % 3]))
        out_idx.fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert (out_idx.cpu().numpy() == want[k % 3]).all(), f"replay {k}"


def test_noalloc_rejects_bad_arguments():
    x = torch.zeros(4, 100, device="cuda")
    out = torch.empty(4, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert _lib.argreduce_noalloc_raw(0, "f32", 4, 100, "max", out.data_ptr(), 0, s) == _lib.ARGR_EINVAL
    assert _lib.argreduce_noalloc_raw(x.data_ptr(), "f32", 4, 0, "max", out.data_ptr(), 0, s) == _lib.ARGR_EINVAL
    assert _lib.argreduce_noalloc_raw(x.data_ptr(), "i32", 4, 100, "max", out.data_ptr(), 0, s) == \
        _lib.ARGR_EUNSUPPORTED
    assert _lib.argreduce_noalloc_raw(x.data_ptr(), "i64", 4, 50, "max", out.data_ptr(), 0, s) == \
        _lib.ARGR_EUNSUPPORTED
    assert _lib.argreduce_noalloc_raw(x.data_ptr(), "f32", 0, 100, "max", out.data_ptr(), 0, s) == _lib.ARGR_OK
