"""Seeded synthetic inputs for row-wise ArgMax/ArgMin.

This module only *makes inputs*. It holds none of the reduction's arithmetic:
no comparison, no scan, no expected index. Both the CPU oracle (under
``oracle/``) and the CUDA path are fed the exact same bytes from here, and the
tests compare their outputs.

Every array is a contiguous row-major ``[rows, cols]`` numpy array of the raw
element type:

* ``f32`` -> ``np.float32``
* ``f64`` -> ``np.float64``
* ``f16`` -> ``np.uint16`` holding IEEE-754 binary16 bit patterns
* ``bf16`` -> ``np.uint16`` holding bfloat16 bit patterns (upper half of binary32)

The workload recipes follow the shapes and value distributions of the two
onnxruntime pull requests on this subject: "[CUDA] Parallelize ArgMax/ArgMin
over wide last axes" (#32092, results table: vocabulary-wide sampler logits
[1, 32000] ... [1, 262144], batches [8|32, 202048], the medium shapes
[4096, 4096] and [65536, 1024], and the narrow shapes [65536, 64], [4096, 8],
[4096, 128]) and "[CUDA] Parallelize ArgMax/ArgMin over the reduction axis"
(#31694, Testing: random, tied and all-equal rows). No public dataset is
involved: Gaussian logits stand in for a model's vocabulary logits.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Iterator, List, Tuple

import numpy as np

DTYPES = ("f32", "f16", "bf16", "f64")
OPS = ("max", "min")
# Last-index variants (ties resolve to the highest index; ONNX select_last_index = 1).
LAST_OPS = ("max_last", "min_last")
ALL_OPS = OPS + LAST_OPS

ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8, "i32": 4, "i64": 8}


# ----------------------------------------------------------------------------
# Encoding of generated float values into the element types.
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round binary32 values to bfloat16 (round to nearest, ties to even).

    bfloat16 is the upper 16 bits of binary32. Rounding adds 0x7FFF plus the
    lowest kept bit to the 32-bit pattern and truncates; NaNs are mapped to a
    quiet NaN of the same sign so that rounding cannot turn them into inf.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        sign = ((u >> 16) & 0x8000).astype(np.uint16)
        rounded = np.where(nan, sign | np.uint16(0x7FC0), rounded)
    return rounded.astype(np.uint16)


def encode(vals: np.ndarray, dtype: str) -> np.ndarray:
    """Encode float values (f64 or f32 array) as the raw element type."""
    if dtype == "f64":
        return np.ascontiguousarray(vals, dtype=np.float64)
    if dtype == "f32":
        return np.ascontiguousarray(vals, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(vals, dtype=np.float32).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def special_values(dtype: str) -> Dict[str, object]:
    """Raw encodings of the special values used by the edge-case recipes."""
    if dtype in ("f32", "f64"):
        ft = np.float32 if dtype == "f32" else np.float64
        return {
            "nan": ft(np.nan),
            "pinf": ft(np.inf),
            "ninf": ft(-np.inf),
            "pzero": ft(0.0),
            "nzero": ft(-0.0),
            "one": ft(1.0),
            "mone": ft(-1.0),
            "denorm": np.finfo(ft).smallest_subnormal,
            "ndenorm": -np.finfo(ft).smallest_subnormal,
            "half": ft(0.5),
        }
    # 16-bit types: raw bit patterns
    if dtype == "f16":
        return {
            "nan": np.uint16(0x7E00),
            "pinf": np.uint16(0x7C00),
            "ninf": np.uint16(0xFC00),
            "pzero": np.uint16(0x0000),
            "nzero": np.uint16(0x8000),
            "one": np.uint16(0x3C00),
            "mone": np.uint16(0xBC00),
            "denorm": np.uint16(0x0001),
            "ndenorm": np.uint16(0x8001),
            "half": np.uint16(0x3800),
        }
    if dtype == "bf16":
        return {
            "nan": np.uint16(0x7FC0),
            "pinf": np.uint16(0x7F80),
            "ninf": np.uint16(0xFF80),
            "pzero": np.uint16(0x0000),
            "nzero": np.uint16(0x8000),
            "one": np.uint16(0x3F80),
            "mone": np.uint16(0xBF80),
            "denorm": np.uint16(0x0001),
            "ndenorm": np.uint16(0x8001),
            "half": np.uint16(0x3F00),
        }
    raise ValueError(dtype)


# The special-value alphabet of the randomized fuzz in #32092 (Testing:
# "{+/-inf, NaN, +/-0.0, ...}"), plus ordinary finite values and the smallest
# subnormal so that flush-to-zero would be caught.
ALPHABET_KEYS = ("ninf", "mone", "nzero", "pzero", "one", "pinf", "nan", "denorm")


def alphabet(dtype: str) -> np.ndarray:
    sv = special_values(dtype)
    raw_t = np.uint16 if dtype in ("f16", "bf16") else (np.float32 if dtype == "f32" else np.float64)
    return np.array([sv[k] for k in ALPHABET_KEYS], dtype=raw_t)


def exhaustive_rows(dtype: str, length: int) -> np.ndarray:
    """Every row of ``length`` symbols over :func:`alphabet` (8**length rows)."""
    a = alphabet(dtype)
    k = len(a)
    n = k ** length
    digits = np.empty((n, length), dtype=np.int64)
    idx = np.arange(n, dtype=np.int64)
    for j in range(length - 1, -1, -1):
        digits[:, j] = idx % k
        idx //= k
    return np.ascontiguousarray(a[digits])


def fuzz_rows(dtype: str, rows: int, cols: int, seed: int, p_special: float = 0.2) -> np.ndarray:
    """Random rows: small integers (many ties) mixed with alphabet symbols."""
    rng = np.random.Generator(np.random.PCG64(seed))
    base = rng.integers(-3, 4, size=(rows, cols)).astype(np.float64)
    x = encode(base, dtype)
    a = alphabet(dtype)
    mask = rng.random((rows, cols)) < p_special
    pick = rng.integers(0, len(a), size=(rows, cols))
    x = np.where(mask, a[pick], x)
    return np.ascontiguousarray(x)


# ----------------------------------------------------------------------------
# Workload recipes.
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Case:
    """One reduction problem: shape, dtype, op and the recipe that fills it."""

    name: str
    rows: int
    cols: int
    dtype: str
    op: str
    recipe: str
    seed: int
    variant: str = ""
    inner: int = 1  # > 1: reduce the middle axis of [rows (outer), cols (reduce), inner]

    @property
    def nbytes(self) -> int:
        return self.rows * self.cols * self.inner * ELEM_SIZE[self.dtype]


def _gauss(rows: int, cols: int, sigma: float, seed: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(sigma)


def _gauss_per_row(rows: int, cols: int, sigma: float, seed0: int) -> np.ndarray:
    out = np.empty((rows, cols), dtype=np.float32)
    for r in range(rows):
        rng = np.random.Generator(np.random.PCG64(seed0 + r))
        out[r] = rng.standard_normal(cols, dtype=np.float32) * np.float32(sigma)
    return out


def make_logits_1(c: Case) -> np.ndarray:
    """Sampler logits of one row ~ N(0, sigma=2)."""
    return encode(_gauss(c.rows, c.cols, 2.0, c.seed), c.dtype)


def make_planted(c: Case) -> np.ndarray:
    """Logits ~ N(0, sigma=3) with a planted extreme.

    The extreme is +64 for ArgMax and -64 for ArgMin (exact in every element
    type; 21 sigma away, so never reached by the Gaussian). Variant ``unique``
    plants it at one seeded position; variant ``dup`` also plants it at a second,
    later seeded position, which exercises the lowest-index tie rule.
    """
    vals = _gauss(c.rows, c.cols, 3.0, c.seed)
    rng = np.random.Generator(np.random.PCG64(c.seed + 7919))
    extreme = np.float32(64.0 if c.op.startswith("max") else -64.0)
    for r in range(c.rows):
        p1 = int(rng.integers(0, c.cols))
        vals[r, p1] = extreme
        if c.variant == "dup" and c.cols > 1:
            p2 = int(rng.integers(0, c.cols))
            if p2 == p1:
                p2 = (p1 + 1 + int(rng.integers(0, c.cols - 1))) % c.cols
            vals[r, p2] = extreme
    return encode(vals, c.dtype)


def make_batch_logits(c: Case) -> np.ndarray:
    """Batches of sampler logits ~ N(0, sigma=3), row r seeded independently."""
    return encode(_gauss_per_row(c.rows, c.cols, 3.0, c.seed), c.dtype)


N_ROW_CLASSES = 20


def make_uniform_special(c: Case) -> np.ndarray:
    """Rows ~ U(-1, 1) with special row classes selected by ``r mod 20``.

    0: all-equal (0.5); 1: +inf at a random position; 2: -inf at a random
    position; 3: +inf twice and -inf twice; 4: NaN at index 0; 5: NaN mid-row;
    6: all -inf; 7: signed-zero tie (every other element made strictly worse
    than zero for the op, -0.0 at one random position and +0.0 at a later one);
    8..19: plain. Each special class is 5% of the rows.
    """
    rows, cols = c.rows, c.cols
    rng = np.random.Generator(np.random.PCG64(c.seed))
    wide = np.float64 if c.dtype == "f64" else np.float32
    vals = rng.uniform(-1.0, 1.0, size=(rows, cols)).astype(wide)
    cls = np.arange(rows) % N_ROW_CLASSES
    pos = rng.integers(0, cols, size=(rows, 4))
    r_ = np.arange(rows)

    def rows_of(k):
        return r_[cls == k]

    vals[rows_of(0)] = 0.5
    rr = rows_of(1)
    vals[rr, pos[rr, 0]] = np.inf
    rr = rows_of(2)
    vals[rr, pos[rr, 0]] = -np.inf
    rr = rows_of(3)
    for k, v in enumerate((np.inf, np.inf, -np.inf, -np.inf)):
        vals[rr, pos[rr, k]] = v
    rr = rows_of(4)
    vals[rr, 0] = np.nan
    rr = rows_of(5)
    if cols > 2:
        mid = 1 + (pos[rr, 0] % (cols - 1))
        vals[rr, mid] = np.nan
    rr = rows_of(6)
    vals[rr] = -np.inf
    rr = rows_of(7)
    if len(rr):
        sub = np.abs(vals[rr]) + wide(0.25)  # strictly positive, away from zero
        vals[rr] = -sub if c.op.startswith("max") else sub
        if cols >= 2:
            p = pos[rr, 0] % (cols - 1)
            q = p + 1 + (pos[rr, 1] % (cols - 1 - p)) if cols > 2 else p + 1
            vals[rr, p] = wide(-0.0)
            vals[rr, q] = wide(0.0)
    return encode(vals, c.dtype)


def make_small_ints(c: Case) -> np.ndarray:
    """Integers U{0..7} cast to float: heavy ties in narrow rows."""
    rng = np.random.Generator(np.random.PCG64(c.seed))
    return encode(rng.integers(0, 8, size=(c.rows, c.cols)).astype(np.float32), c.dtype)


def make_axis_mixed(c: Case) -> np.ndarray:
    """[outer, R, inner] values ~ U(-1, 1) rounded to 1/64 (many ties along R),
    with 0.1% of the elements replaced by special values (NaN, +-inf, +-0)."""
    rng = np.random.Generator(np.random.PCG64(c.seed))
    shape = (c.rows, c.cols, c.inner)
    vals = np.round(rng.uniform(-1.0, 1.0, size=shape) * 64.0) / 64.0
    x = encode(vals, c.dtype)
    a = alphabet(c.dtype)
    n = x.size
    k = max(1, n // 1000)
    pos = rng.integers(0, n, size=k)
    flat = x.reshape(-1)
    flat[pos] = a[rng.integers(0, len(a), size=k)]
    return x


def make_cum_values(c: Case) -> np.ndarray:
    """Inputs of the cummax / cummin workloads: integers U{-1000..1000} for
    the integer types; N(0, 1) with 0.1% special values for the floats."""
    rng = np.random.Generator(np.random.PCG64(c.seed))
    if c.dtype in ("i32", "i64"):
        return rng.integers(-1000, 1001, size=(c.rows, c.cols)).astype(np.int32 if c.dtype == "i32" else np.int64)
    x = encode(rng.standard_normal((c.rows, c.cols)), c.dtype)
    a = alphabet(c.dtype)
    k = max(1, x.size // 1000)
    flat = x.reshape(-1)
    flat[rng.integers(0, x.size, size=k)] = a[rng.integers(0, len(a), size=k)]
    return x


RECIPES = {
    "logits": make_logits_1,
    "planted": make_planted,
    "batch_logits": make_batch_logits,
    "uniform_special": make_uniform_special,
    "small_ints": make_small_ints,
    "axis_mixed": make_axis_mixed,
    "cum_values": make_cum_values,
}


def make(c: Case) -> np.ndarray:
    x = RECIPES[c.recipe](c)
    shape = (c.rows, c.cols) if c.inner == 1 else (c.rows, c.cols, c.inner)
    assert x.shape == shape and x.flags.c_contiguous
    return x


# The five workload groups. Seeds are fixed constants.
def config_cases(k: int) -> List[Case]:
    """Cases of workload group ``k``: 1..5 the reductions, 6 the non-last
    axis, 7 and 8 the cummax / cummin scans."""
    out: List[Case] = []
    if k == 1:
        out.append(Case("logits_1x32000_f32_max", 1, 32000, "f32", "max", "logits", 1001))
    elif k == 2:
        for si, cols in enumerate((202048, 262144)):
            for dtype in ("f32", "bf16"):
                for op in ("max", "min"):
                    for variant in ("unique", "dup"):
                        out.append(Case(f"planted_1x{cols}_{dtype}_{op}_{variant}", 1, cols, dtype, op,
                                        "planted", 2001 + si, variant))
    elif k == 3:
        for rows in (8, 32):
            for dtype in ("f16", "bf16", "f32"):
                out.append(Case(f"batch_{rows}x202048_{dtype}_max", rows, 202048, dtype, "max",
                                "batch_logits", 3001))
    elif k == 4:
        for rows, cols in ((4096, 4096), (65536, 1024)):
            for dtype in ("f32", "f64"):
                for op in ("min", "max"):
                    out.append(Case(f"uniform_{rows}x{cols}_{dtype}_{op}", rows, cols, dtype, op,
                                    "uniform_special", 4001))
    elif k == 5:
        for rows, cols in ((65536, 64), (4096, 8), (4096, 128)):
            out.append(Case(f"narrow_{rows}x{cols}_f32_max", rows, cols, "f32", "max", "small_ints", 5001))
    elif k == 6:
        # Reduction over a non-last axis [outer, R, inner] (the next widening of the path):
        # column ArgMax/ArgMin of tall and wide matrices, a batched middle axis, a small inner extent.
        out.append(Case("axis_1x100000x1000_f32_max", 1, 100000, "f32", "max", "axis_mixed", 6001, inner=1000))
        out.append(Case("axis_1x1000x100000_f32_min", 1, 1000, "f32", "min", "axis_mixed", 6002, inner=100000))
        out.append(Case("axis_64x512x256_bf16_max", 64, 512, "bf16", "max", "axis_mixed", 6003, inner=256))
        out.append(Case("axis_128x4096x8_f32_max", 128, 4096, "f32", "max", "axis_mixed", 6004, inner=8))
        out.append(Case("axis_16x2048x384_f64_min", 16, 2048, "f64", "min", "axis_mixed", 6005, inner=384))
    elif k == 7:
        # cummax / cummin with indices (the shapes and dtypes of Paddle issue #79670's tables).
        for rows, cols, dtype, op in ((1, 65536, "i64", "max"), (1, 262144, "i64", "max"), (64, 1024, "i64", "max"),
                                      (1024, 64, "i64", "min"), (4, 16384, "i32", "max"), (1, 65536, "f32", "max"),
                                      (1, 65536, "f64", "min"), (256, 256, "bf16", "max")):
            out.append(Case(f"cum_{rows}x{cols}_{dtype}_{op}", rows, cols, dtype, op, "cum_values", 7001 + cols % 97))
    elif k == 8:
        # cummax / cummin at bandwidth scale (hundreds of MB per call)
        for rows, cols, dtype, op in ((1, 1 << 24, "i64", "max"), (16, 1 << 20, "f64", "min"),
                                      (4096, 4096, "f32", "max"), (256, 65536, "f32", "min")):
            out.append(Case(f"cum_{rows}x{cols}_{dtype}_{op}", rows, cols, dtype, op, "cum_values", 8001 + rows % 97))
    else:
        raise ValueError(k)
    return out


def all_cases(groups=range(1, 6)) -> Iterator[Tuple[int, Case]]:
    for k in groups:
        for c in config_cases(k):
            yield k, c


def scaled(c: Case, rows: int = None, cols: int = None) -> Case:
    """The same recipe at a smaller shape (for oracle-sized parity cases)."""
    return dataclasses.replace(c, rows=rows or c.rows, cols=cols or c.cols,
                               name=f"{c.name}@{rows or c.rows}x{cols or c.cols}")
