"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:

* its binary16 / bfloat16 decoders against numpy's conversions, for every one
  of the 65536 bit patterns of each type;
* the sequential scan against an independent closed form, exhaustively over
  every row of length 1..5 on the special-value alphabet of the randomized
  fuzz in onnxruntime PR #32092 (Testing);
* numpy.argmax / numpy.argmin (documented to return the first occurrence) on
  NaN-free rows, including heavy ties;
* invariants planted by construction (unique and duplicated extremes);
* golden rows built to the pages' own test descriptions (tests/golden/);
* a mutation check: plausible mistakes planted into the oracle's C source
  must each be caught by at least one of these pins.
"""
import json
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent decoding (numpy) and the closed form.
# ---------------------------------------------------------------------------
def np_decode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Decode raw elements to float64 with numpy's own conversions."""
    if dtype == "f32":
        return x.astype(np.float64)
    if dtype == "f64":
        return x.astype(np.float64)
    if dtype == "f16":
        return x.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):  # signalling NaN patterns stay NaN
            return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def closed_form(x: np.ndarray, dtype: str, op: str) -> np.ndarray:
    """Second formulation of the result: 0 when element 0 is NaN, otherwise the
    smallest j (largest j for the last-index ops) whose value is not NaN and
    equals the max (min) over the non-NaN values of the row."""
    v = np_decode(x, dtype)
    rows, cols = v.shape
    out = np.zeros(rows, dtype=np.int64)
    nan = np.isnan(v)
    lead_nan = nan[:, 0]
    is_max = op.startswith("max")
    fill = -np.inf if is_max else np.inf
    w = np.where(nan, fill, v)
    m = w.max(axis=1) if is_max else w.min(axis=1)
    hit = (~nan) & (v == m[:, None])
    if op.endswith("_last"):
        pick = cols - 1 - np.argmax(hit[:, ::-1], axis=1)
    else:
        pick = np.argmax(hit, axis=1)
    out[:] = np.where(lead_nan, 0, pick)
    return out


def raw_equal(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality of raw element arrays (NaN payloads included)."""
    ua = a.view(np.uint8)
    ub = b.view(np.uint8)
    return ua.shape == ub.shape and bool((ua == ub).all())


def take_rows(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    return x[np.arange(x.shape[0]), idx]


# ---------------------------------------------------------------------------
# Decoders.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decoder_exhaustive(dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = np_decode(bits.reshape(1, -1), dtype)[0]
    dec = oracle.decode_f16 if dtype == "f16" else oracle.decode_bf16
    got = np.array([dec(int(b)) for b in bits], dtype=np.float64)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # signs of zeros and infinities survive decoding
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


# ---------------------------------------------------------------------------
# Exhaustive brute force over the special-value alphabet.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("op", W.ALL_OPS)
def test_exhaustive_alphabet(dtype, op):
    for length in range(1, 6):
        x = W.exhaustive_rows(dtype, length)
        idx, val, _ = oracle.argreduce(x, dtype, op)
        exp = closed_form(x, dtype, op)
        bad = np.nonzero(idx != exp)[0]
        assert bad.size == 0, (length, x[bad[:5]], idx[bad[:5]], exp[bad[:5]])
        assert raw_equal(val, take_rows(x, idx))


def test_brute_force_python_loop():
    """A third formulation on a small random sample: pure Python, pairwise
    'is any earlier element at least as good / any element strictly better'."""
    for dtype in W.DTYPES:
        x = W.fuzz_rows(dtype, 400, 9, seed=77, p_special=0.4)
        v = np_decode(x, dtype)
        for op in W.ALL_OPS:
            idx, _, _ = oracle.argreduce(x, dtype, op)
            is_max = op.startswith("max")
            order = range(x.shape[1] - 1, -1, -1) if op.endswith("_last") else range(x.shape[1])
            for r in range(x.shape[0]):
                row = v[r]
                if np.isnan(row[0]):
                    exp = 0
                else:
                    exp = None
                    for j in order:
                        if np.isnan(row[j]):
                            continue
                        beats_all = all(
                            np.isnan(row[k]) or (row[j] >= row[k] if is_max else row[j] <= row[k])
                            for k in range(len(row)))
                        if beats_all:
                            exp = j
                            break
                assert idx[r] == exp, (dtype, op, r, row)


# ---------------------------------------------------------------------------
# numpy special case: NaN-free rows.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", W.DTYPES)
def test_numpy_nan_free(dtype):
    rng = np.random.Generator(np.random.PCG64(123))
    g = W.encode(rng.standard_normal((64, 3001)) * 3.0, dtype)
    t = W.encode(rng.integers(0, 8, size=(64, 1000)).astype(np.float64), dtype)
    for x in (g, t):
        v = np_decode(x, dtype)
        assert not np.isnan(v).any()
        for op in W.OPS:
            idx, val, _ = oracle.argreduce(x, dtype, op)
            exp = np.argmax(v, axis=1) if op == "max" else np.argmin(v, axis=1)
            assert (idx == exp).all()
            assert raw_equal(val, take_rows(x, idx))
        # last occurrence: numpy's first occurrence on the reversed row
        cols = v.shape[1]
        for op in W.LAST_OPS:
            idx, val, _ = oracle.argreduce(x, dtype, op)
            rv = v[:, ::-1]
            first_rev = np.argmax(rv, axis=1) if op == "max_last" else np.argmin(rv, axis=1)
            assert (idx == cols - 1 - first_rev).all()
            assert raw_equal(val, take_rows(x, idx))


def test_mt_wrapper_matches_single():
    x = W.fuzz_rows("f32", 1000, 77, seed=5)
    for op in W.OPS:
        a, va, _ = oracle.argreduce(x, "f32", op, threads=1)
        b, vb, used = oracle.argreduce(x, "f32", op, threads=7)
        assert used == 7
        assert (a == b).all() and raw_equal(va, vb)


def test_invalid_arguments():
    x = np.zeros((2, 0), dtype=np.float32)
    with pytest.raises(ValueError):
        oracle.argreduce(x, "f32", "max")


# ---------------------------------------------------------------------------
# Invariants by construction on the workload recipes (reduced sizes).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", W.OPS)
def test_planted_extreme(dtype, op):
    for variant in ("unique", "dup"):
        c = W.Case("t", 3, 20011, dtype, op, "planted", 99, variant)
        x = W.make(c)
        v = np_decode(x, dtype)
        target = 64.0 if op == "max" else -64.0
        idx, _, _ = oracle.argreduce(x, dtype, op)
        for r in range(c.rows):
            pos = np.nonzero(v[r] == target)[0]
            assert len(pos) == (1 if variant == "unique" else 2)
            assert idx[r] == pos[0]


def test_small_ints_first_seven():
    c = W.Case("t", 512, 64, "f32", "max", "small_ints", 5001)
    x = W.make(c)
    idx, _, _ = oracle.argreduce(x, "f32", "max")
    for r in range(c.rows):
        row = list(x[r])
        assert idx[r] == row.index(max(row))
    idx, _, _ = oracle.argreduce(x, "f32", "min")
    for r in range(c.rows):
        row = list(x[r])
        assert idx[r] == row.index(min(row))


@pytest.mark.parametrize("dtype", ["f32", "f64"])
@pytest.mark.parametrize("op", W.OPS)
def test_uniform_special_classes(dtype, op):
    c = W.Case("t", 200, 301, dtype, op, "uniform_special", 4001)
    x = W.make(c)
    v = np_decode(x, dtype)
    idx, val, _ = oracle.argreduce(x, dtype, op)
    cls = np.arange(c.rows) % W.N_ROW_CLASSES
    for r in range(c.rows):
        k = cls[r]
        row = v[r]
        if k in (0, 4, 6):  # all-equal, leading NaN, all -inf
            assert idx[r] == 0
        elif k == 7:  # -0.0 then +0.0, everything else worse than zero
            z = np.nonzero(row == 0.0)[0]
            assert len(z) == 2 and np.signbit(row[z[0]]) and not np.signbit(row[z[1]])
            assert idx[r] == z[0]
        elif k == 5:  # a NaN mid-row is never chosen
            assert not np.isnan(row[idx[r]])
        if k == 1 and op == "max":
            assert np.isposinf(row[idx[r]])
        if k == 2 and op == "min":
            assert np.isneginf(row[idx[r]])
    assert raw_equal(val, take_rows(x, idx))


# ---------------------------------------------------------------------------
# Golden rows built to the pages' test descriptions.
# ---------------------------------------------------------------------------
def _token(tok, dtype):
    sv = W.special_values(dtype)
    if isinstance(tok, (int, float)):
        return W.encode(np.array([float(tok)]), dtype)[0]
    m = {"nan": "nan", "inf": "pinf", "-inf": "ninf", "-0": "nzero", "denorm": "denorm"}
    if tok in m:
        return sv[m[tok]]
    if tok in ("lowest", "highest"):
        if dtype == "f16":
            return np.uint16(0xFBFF if tok == "lowest" else 0x7BFF)
        if dtype == "bf16":
            return np.uint16(0xFF7F if tok == "lowest" else 0x7F7F)
        ft = np.float32 if dtype == "f32" else np.float64
        return np.finfo(ft).min if tok == "lowest" else np.finfo(ft).max
    raise ValueError(tok)


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_golden_semantics(dtype):
    with open(os.path.join(GOLDEN, "onnxruntime_32092_semantics.json")) as f:
        fx = json.load(f)
    raw_t = oracle.RAW_NP[dtype]
    for case in fx["cases"]:
        x = np.array([[_token(t, dtype) for t in case["row"]]], dtype=raw_t)
        for op in W.OPS:
            idx, val, _ = oracle.argreduce(x, dtype, op)
            assert idx[0] == case[op], (case["what"], op)
            assert raw_equal(val, x[0, idx])


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_golden_semantics_last_index(dtype):
    with open(os.path.join(GOLDEN, "onnx_select_last_index.json")) as f:
        fx = json.load(f)
    raw_t = oracle.RAW_NP[dtype]
    for case in fx["cases"]:
        x = np.array([[_token(t, dtype) for t in case["row"]]], dtype=raw_t)
        for op in W.LAST_OPS:
            idx, val, _ = oracle.argreduce(x, dtype, op)
            assert idx[0] == case[op], (case["what"], op)
            assert raw_equal(val, x[0, idx])


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_golden_long_axis(dtype):
    with open(os.path.join(GOLDEN, "onnxruntime_31694_long_axis_300x4.json")) as f:
        fx = json.load(f)
    x = W.encode(np.array(fx["rows"], dtype=np.float64), dtype)
    for op in W.OPS:
        idx, _, _ = oracle.argreduce(x, dtype, op)
        assert list(idx) == fx["expected"][op]


def test_golden_first_index_65536():
    with open(os.path.join(GOLDEN, "onnxruntime_31694_first_index_65536.json")) as f:
        fx = json.load(f)
    rng = np.random.Generator(np.random.PCG64(fx["seed"]))
    row = rng.standard_normal(fx["cols"]).astype(np.float32)
    row[fx["inf_positions"]] = np.inf
    idx, _, _ = oracle.argreduce(row.reshape(1, -1), "f32", "max")
    assert idx[0] == fx["expected_max"]


# ---------------------------------------------------------------------------
# Mutation check: each planted mistake must fail a pin.
# ---------------------------------------------------------------------------
MUTANTS = [
    ("first-index ties become last", "case ORACLE_MAX: return a > b;", "case ORACLE_MAX: return a >= b;"),
    ("min ties become last", "case ORACLE_MIN: return a < b;", "case ORACLE_MIN: return a <= b;"),
    ("ops swapped", "case ORACLE_MAX: return a > b;", "case ORACLE_MAX: return a < b;"),
    ("NaN wins", "case ORACLE_MAX: return a > b;", "case ORACLE_MAX: return !(a <= b);"),
    ("element 1 skipped", "for (int64_t j = 1; j < cols; ++j)", "for (int64_t j = 2; j < cols; ++j)"),
    ("last element skipped", "for (int64_t j = 1; j < cols; ++j)", "for (int64_t j = 1; j + 1 < cols; ++j)"),
    ("value from wrong index", "row + (size_t)best_j * es, es);", "row, es);"),
    ("f16 subnormal scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("f16 implicit bit", "ldexp((double)(1024 + f), e - 25)", "ldexp((double)(f), e - 15)"),
    ("bf16 fraction width", "ldexp((double)(128 + f), e - 134)", "ldexp((double)(256 + f), e - 135)"),
    ("bf16 sign dropped", "    return sign ? -v : v;\n}\n\nstatic size_t", "    return v;\n}\n\nstatic size_t"),
    ("row stride", "(size_t)r * (size_t)cols * es", "(size_t)r * (size_t)cols"),
    ("last-index ties dropped", "case ORACLE_MAX_LAST: return a >= b;", "case ORACLE_MAX_LAST: return a > b;"),
    ("last-index lets NaN in", "default: return a <= b;", "default: return !(a > b);"),
]


def _pin_suite_passes(lib_path: str) -> bool:
    """Run a compact version of the pins above against another build."""
    import ctypes
    saved = oracle._lib
    try:
        oracle._lib = None
        lib = ctypes.CDLL(lib_path)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_argreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, i64p, ctypes.c_void_p]
        lib.oracle_argreduce_mt.argtypes = lib.oracle_argreduce.argtypes + [ctypes.c_int]
        for name in ("oracle_decode_f16", "oracle_decode_bf16"):
            getattr(lib, name).argtypes = [ctypes.c_uint16]
            getattr(lib, name).restype = ctypes.c_double
        oracle._lib = lib
        try:
            for dtype in ("f16", "bf16"):
                test_decoder_exhaustive(dtype)
            for dtype in W.DTYPES:
                for op in W.ALL_OPS:
                    test_exhaustive_alphabet(dtype, op)
                test_numpy_nan_free(dtype)
                test_golden_semantics(dtype)
                test_golden_semantics_last_index(dtype)
                test_golden_long_axis(dtype)
        except AssertionError:
            return False
        return True
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mutated = src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "libm_oracle.so")
        with open(c, "w") as f:
            f.write(mutated)
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", c, "-o", so, "-lm"],
                       check=True)
        assert not _pin_suite_passes(so), f"mutant '{name}' survived the pins"


def test_unmutated_passes_pin_suite():
    assert _pin_suite_passes(oracle.build())


# ---------------------------------------------------------------------------
# Reduction over a non-last (strided) axis: x[outer, R, inner] over R.
# ---------------------------------------------------------------------------
def closed_form_axis(x3, dtype, op):
    """The closed form applied to every (o, i) column: move R last, reuse the
    2-D closed form on the [outer*inner, R] view."""
    outer, R, inner = x3.shape
    cols = np.ascontiguousarray(np.transpose(x3, (0, 2, 1))).reshape(outer * inner, R)
    return closed_form(cols, dtype, op).reshape(outer, inner)


@pytest.mark.parametrize("dtype", W.DTYPES)
@pytest.mark.parametrize("op", W.ALL_OPS)
def test_axis_exhaustive_alphabet(dtype, op):
    # every length-4 column over the alphabet, laid out with inner = 8, 64, 512
    rows = W.exhaustive_rows(dtype, 4)  # [4096, 4]
    for inner in (8, 64, 512):
        x3 = np.ascontiguousarray(rows.reshape(-1, inner, 4).transpose(0, 2, 1))  # [outer, R=4, inner]
        idx, val = oracle.argreduce_axis(x3, dtype, op)
        assert (idx == closed_form_axis(x3, dtype, op)).all()
        gathered = np.take_along_axis(x3, idx[:, None, :], axis=1)[:, 0, :]
        assert raw_equal(val, np.ascontiguousarray(gathered))


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_axis_numpy_nan_free(dtype):
    rng = np.random.Generator(np.random.PCG64(9))
    for shape in ((3, 1000, 17), (1, 257, 64), (5, 2, 3), (2, 1, 9), (4, 33, 1)):
        x3 = W.encode(rng.integers(-4, 5, size=shape).astype(np.float64), dtype)
        v = np_decode(x3.reshape(-1, 1), dtype).reshape(shape)
        idx, _ = oracle.argreduce_axis(x3, dtype, "max")
        assert (idx == np.argmax(v, axis=1)).all()
        idx, _ = oracle.argreduce_axis(x3, dtype, "min")
        assert (idx == np.argmin(v, axis=1)).all()
        idx, _ = oracle.argreduce_axis(x3, dtype, "max_last")
        assert (idx == shape[1] - 1 - np.argmax(v[:, ::-1, :], axis=1)).all()


def test_axis_brute_force_loops():
    """Pure-Python loops over (o, r, i) on a small special-value tensor."""
    for dtype in ("f32", "bf16"):
        x = W.fuzz_rows(dtype, 6, 5 * 7, seed=3, p_special=0.4).reshape(6, 5, 7)
        v = np_decode(x.reshape(-1, 1), dtype).reshape(x.shape)
        for op in W.ALL_OPS:
            idx, _ = oracle.argreduce_axis(x, dtype, op)
            for o in range(6):
                for i in range(7):
                    col = [v[o, r, i] for r in range(5)]
                    if np.isnan(col[0]):
                        exp = 0
                    else:
                        ok = [r for r in range(5) if not np.isnan(col[r]) and all(
                            np.isnan(col[k]) or (col[r] >= col[k] if op.startswith("max") else col[r] <= col[k])
                            for k in range(5))]
                        exp = ok[-1] if op.endswith("_last") else ok[0]
                    assert idx[o, i] == exp, (op, o, i, col)


AXIS_MUTANTS = [
    ("column stride", "const size_t stride = (size_t)inner * es;", "const size_t stride = es;"),
    ("outer offset", "(size_t)o * (size_t)R * (size_t)inner + (size_t)i", "(size_t)o * (size_t)inner + (size_t)i"),
    ("output position", "out_idx[o * inner + i] = best_r;", "out_idx[i * outer + o] = best_r;"),
    ("first r skipped", "for (int64_t r = 1; r < R; ++r) {", "for (int64_t r = 2; r < R; ++r) {"),
]


@pytest.mark.parametrize("name,old,new", AXIS_MUTANTS, ids=[m[0] for m in AXIS_MUTANTS])
def test_axis_mutant_is_caught(name, old, new):
    import ctypes
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, old
    with tempfile.TemporaryDirectory() as d:
        c, so = os.path.join(d, "m.c"), os.path.join(d, "libm.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", c, "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        lib.oracle_argreduce_axis.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                              ctypes.c_void_p]
        saved = oracle._lib
        try:
            class Shim:
                pass
            shim = Shim()
            shim.oracle_argreduce_axis = lib.oracle_argreduce_axis
            oracle._lib = shim
            caught = False
            try:
                for dtype in ("f32", "f64"):
                    test_axis_numpy_nan_free(dtype)
                    for op in W.ALL_OPS:
                        test_axis_exhaustive_alphabet(dtype, op)
            except AssertionError:
                caught = True
            assert caught, f"axis mutant '{name}' survived"
        finally:
            oracle._lib = saved


# ---------------------------------------------------------------------------
# cummax / cummin with indices (prefix ArgMax / ArgMin).
# ---------------------------------------------------------------------------
CUM_DTYPES = ("f32", "f16", "bf16", "f64", "i32", "i64")


def cum_rows(dtype, rows, cols, seed):
    if dtype in ("i32", "i64"):
        rng = np.random.Generator(np.random.PCG64(seed))
        info = np.iinfo(np.int32 if dtype == "i32" else np.int64)
        x = rng.integers(-5, 6, size=(rows, cols)).astype(np.int64)
        ext = rng.random((rows, cols)) < 0.05
        x = np.where(ext, np.where(rng.random((rows, cols)) < 0.5, info.min, info.max), x)
        big = rng.random((rows, cols)) < 0.05
        x = np.where(big, info.max - rng.integers(0, 3, size=(rows, cols)), x)  # values a double cannot tell apart
        return x.astype(np.int32 if dtype == "i32" else np.int64)
    return W.fuzz_rows(dtype, rows, cols, seed=seed, p_special=0.2)


@pytest.mark.parametrize("dtype", CUM_DTYPES)
@pytest.mark.parametrize("op", ("max", "min"))
def test_cumreduce_prefix_equals_argreduce(dtype, op):
    """Column j of the scan is the oracle's ArgMax/ArgMin of the prefix 0..j
    (for the floating types), and a direct running scan in Python (ints)."""
    x = cum_rows(dtype, 30, 41, seed=7)
    idx, val = oracle.cumreduce(x, dtype, op)
    assert raw_equal(val, np.take_along_axis(x, idx, axis=1))
    if dtype in ("i32", "i64"):
        for r in range(x.shape[0]):
            best = 0
            for j in range(x.shape[1]):
                v, b = int(x[r, j]), int(x[r, best])
                if (v > b) if op == "max" else (v < b):
                    best = j
                assert idx[r, j] == best
    else:
        for j in range(x.shape[1]):
            pidx, _, _ = oracle.argreduce(np.ascontiguousarray(x[:, :j + 1]), dtype, op)
            assert (idx[:, j] == pidx).all()
            assert (idx[:, j] == closed_form(np.ascontiguousarray(x[:, :j + 1]), dtype, op)).all()


def test_cumreduce_numpy_accumulate():
    """NaN-free floats and ints: the values are numpy's maximum/minimum
    accumulate, and each index is the first position reaching that value."""
    rng = np.random.Generator(np.random.PCG64(11))
    for dtype in ("f32", "f64", "i64", "i32"):
        x = rng.integers(-50, 50, size=(20, 333)).astype(oracle.RAW_NP[dtype])
        for op, acc in (("max", np.maximum), ("min", np.minimum)):
            idx, val = oracle.cumreduce(x, dtype, op)
            assert (val == acc.accumulate(x, axis=1)).all()
            for r in range(x.shape[0]):
                first = {}
                for j, v in enumerate(x[r]):
                    first.setdefault(v, j)
                assert all(idx[r, j] == first[val[r, j]] for j in range(x.shape[1]))


def test_cumreduce_golden_two_pass():
    """Paddle issue #79670 (Possible fixes): a tiled two-pass cummax (cummax
    inside tiles, cummax of the tile maxima, carry folded back) is bit-equal to
    the one-pass scan. Built here with numpy on int64 data."""
    rng = np.random.Generator(np.random.PCG64(79670))
    x = rng.integers(-1000, 1000, size=(1, 65536)).astype(np.int64)
    _, val = oracle.cumreduce(x, "i64", "max")
    part = np.maximum.accumulate(x.reshape(512, 128), axis=1)
    carry = np.maximum.accumulate(part[:, -1])
    two_pass = np.maximum(part, np.concatenate([[np.iinfo(np.int64).min], carry[:-1]])[:, None]).reshape(1, -1)
    assert (val == two_pass).all()


CUM_MUTANTS = [
    ("int ties to last", "take = op == ORACLE_MAX ? v > best_i : v < best_i;",
     "take = op == ORACLE_MAX ? v >= best_i : v <= best_i;"),
    ("int compared as double", "const int64_t v = read_int(row + (size_t)j * es, dtype);",
     "const int64_t v = (int64_t)(double)read_int(row + (size_t)j * es, dtype);"),
    ("output one late", "out_idx[(size_t)r * (size_t)cols + (size_t)j] = best_j;",
     "out_idx[(size_t)r * (size_t)cols + (size_t)j] = j > 0 && j == best_j ? j - 1 : best_j;"),
]


@pytest.mark.parametrize("name,old,new", CUM_MUTANTS, ids=[m[0] for m in CUM_MUTANTS])
def test_cum_mutant_is_caught(name, old, new):
    import ctypes
    if shutil.which("gcc") is None:
        pytest.skip("no host C compiler")
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, old
    with tempfile.TemporaryDirectory() as d:
        c, so = os.path.join(d, "m.c"), os.path.join(d, "libm.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", c, "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_cumreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                         i64p, ctypes.c_void_p]
        lib.oracle_argreduce.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int, i64p, ctypes.c_void_p]
        saved = oracle._lib
        try:
            class Shim:
                pass
            shim = Shim()
            shim.oracle_cumreduce = lib.oracle_cumreduce
            shim.oracle_argreduce = saved.oracle_argreduce if saved else oracle._load().oracle_argreduce
            oracle._lib = shim
            caught = False
            try:
                for dtype in CUM_DTYPES:
                    for op in ("max", "min"):
                        test_cumreduce_prefix_equals_argreduce(dtype, op)
                test_cumreduce_numpy_accumulate()
            except AssertionError:
                caught = True
            assert caught, f"cum mutant '{name}' survived"
        finally:
            oracle._lib = saved
