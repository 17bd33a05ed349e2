"""The benchmark's comparison point, cub::DeviceReduce::ArgMax / ArgMin called
as a library, computes the same thing as argreduce() on the rows it is timed
on: on NaN-free single rows (planted unique and duplicated extremes, heavy
ties, the wide-row lengths) its index equals the oracle's first index."""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

import row_wise_arg_gb300 as A  # noqa: E402
from row_wise_arg_gb300 import cub_compare  # noqa: E402

VIEW = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64}


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_wise_arg_gb300.build import build
    build()


def cub_index(x, dtype, op):
    xd = torch.from_numpy(np.ascontiguousarray(x).view(VIEW[dtype])).cuda().reshape(-1)
    n = xd.numel()
    temp = torch.empty(max(cub_compare.temp_bytes(dtype, op, n), 16), dtype=torch.uint8, device="cuda")
    val = torch.empty(16, dtype=torch.uint8, device="cuda")
    idx = torch.empty(1, dtype=torch.int64, device="cuda")
    cub_compare.argreduce_raw(xd.data_ptr(), dtype, op, n, val.data_ptr(), idx.data_ptr(), temp.data_ptr(),
                              temp.numel(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return int(idx.item())


def test_cub_matches_on_the_timed_rows():
    for c in W.config_cases(1) + W.config_cases(2):
        x = W.make(c)
        e, _, _ = oracle.argreduce(x, c.dtype, c.op)
        assert cub_index(x, c.dtype, c.op) == int(e[0]), c.name


@pytest.mark.parametrize("dtype", ("f32", "f16", "bf16", "f64"))
def test_cub_first_index_on_ties(dtype):
    rng = np.random.Generator(np.random.PCG64(32092))
    for n in (1, 2, 255, 256, 257, 1000, 129280, 1 << 22):
        v = rng.integers(-3, 4, size=(1, n)).astype(np.float64)  # many ties, exact in every type
        x = W.encode(v, dtype)
        for op in ("max", "min"):
            e, _, _ = oracle.argreduce(x, dtype, op)
            got, _ = A.argreduce(torch.from_numpy(x.view(VIEW[dtype])).cuda(), op, dtype=dtype)
            assert cub_index(x, dtype, op) == int(e[0]) == int(got.item()), (n, op)
