"""CPU models of the kernels' per-thread vector scans and group merges,
checked against the oracle on fuzz rows (many ties, NaN, +-inf, +-0).

The models restate step for step what the device code in
row_wise_arg_gb300/csrc/device_common.cuh does, so that a flaw in the
decomposition itself would show here without a GPU:
  * VecScan for 16-bit elements: the even- and odd-position elements of a
    thread's vectors are two subsequences, each with its own candidate seeded
    from the thread's candidate; per 32-bit word one packed comparison gives
    both update predicates and a packed max / min (NaN ignored) keeps the
    keys; the two candidates merge by the usual rule at the end.
  * group_merge_redux: keys mapped to order-preserving unsigned integers
    (binary32: bits of key + 0.0; binary64 keys: high word, then low word
    among the lanes holding the best high word), the best key, then the lowest
    (last-occurrence ops: highest) index holding it.
The rule both must reproduce is the sequential scan of the onnxruntime #32092
Semantics section (seed (x[0], 0), replace only on a strictly better element;
the last-occurrence ops replace on "not worse").
"""
import numpy as np
import pytest

import oracle
import workloads as W

OPS = ("max", "min", "max_last", "min_last")


def widen(raw: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of raw 16-bit patterns."""
    if dtype == "f16":
        return raw.view(np.float16).astype(np.float64)
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def takes(x, k, op):
    """The scan's update test: strictly better, or not worse for *_last (false on NaN)."""
    is_min, last = "min" in op, op.endswith("_last")
    if last:
        return x <= k if is_min else x >= k
    return x < k if is_min else x > k


def merge(a, b, op):
    """Better key wins; equal keys keep the lower index (the higher for *_last)."""
    (ka, ia), (kb, ib) = a, b
    is_min, last = "min" in op, op.endswith("_last")
    strictly = kb < ka if is_min else kb > ka
    tie = kb == ka and (ib > ia if last else ib < ia)
    return b if strictly or tie else a


def pair_scan(seed, words, op):
    """VecScan<16-bit>: `words` are (j, x[j], x[j+1]) in the thread's order."""
    k0, i0 = seed
    if k0 != k0:  # a NaN candidate (only x[0]) is never displaced
        return seed
    is_min = "min" in op
    ext = np.fmin if is_min else np.fmax  # NaN-ignoring, like min/max.{f16,bf16}x2
    ke = ko = k0
    ie, io = i0, i0 - 1
    for j, xe, xo in words:
        if takes(xe, ke, op):
            ie = j
        if takes(xo, ko, op):
            io = j
        ke, ko = ext(ke, xe), ext(ko, xo)
    return merge((ke, ie), (ko, io + 1), op)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", OPS)
def test_paired_16bit_scan_matches_oracle(dtype, op):
    rows, cols = 60, 8 * 37  # whole 16-byte vectors of eight 16-bit elements
    for seed, p_special in ((1, 0.2), (2, 0.6), (3, 0.02)):
        raw = W.fuzz_rows(dtype, rows, cols, seed=seed * 17 + OPS.index(op), p_special=p_special)
        raw[::7, 0] = raw[1::7, 3]  # leading specials (a NaN x[0] among them) in some rows
        eidx, _, _ = oracle.argreduce(raw, dtype, op)
        vals = widen(raw, dtype)
        nvec = cols // 8
        for r in range(rows):
            x = vals[r]
            for nthreads in (1, 3, 8):  # thread t visits vectors t, t + T, ... in order
                cands = []
                for t in range(nthreads):
                    words = [(8 * v + 2 * m, x[8 * v + 2 * m], x[8 * v + 2 * m + 1])
                             for v in range(t, nvec, nthreads) for m in range(4)]
                    cands.append(pair_scan((x[0], 0), words, op))
                c = cands[0]
                for o in cands[1:]:
                    c = merge(c, o, op)
                assert c[1] == eidx[r], (dtype, op, r, nthreads, c, eidx[r])


def redux_merge32(cands, op):
    """group_merge_redux for binary32 keys over candidates (key, index)."""
    keys = np.array([k for k, _ in cands], dtype=np.float32)
    b = (keys + np.float32(0.0)).view(np.uint32)  # -0.0 becomes +0.0
    u = b ^ ((b.view(np.int32) >> 31).view(np.uint32) | np.uint32(0x80000000))
    if "min" in op:
        u = ~u
    has = u == u.max()
    idx = [i for (_, i), h in zip(cands, has) if h]
    win = max(idx) if op.endswith("_last") else min(idx)
    return next(c for c in cands if c[1] == win)


def redux_has64(keys):
    """The binary64 reduction: high word, then low word among the best high words."""
    hi, lo = keys >> np.uint64(32), keys & np.uint64(0xFFFFFFFF)
    top = hi == hi.max()
    best_lo = np.where(top, lo, np.uint64(0)).max()
    return top & (lo == best_lo)


@pytest.mark.parametrize("op", OPS)
def test_redux_merge_matches_merge_tree(op):
    rng = np.random.Generator(np.random.PCG64(404 + OPS.index(op)))
    row = W.fuzz_rows("f32", 1, 4000, seed=405, p_special=0.3)[0]
    numbers = np.flatnonzero(row == row)  # candidates are numbers unless x[0] is NaN
    for trial in range(3000):
        n = int(rng.integers(1, 33))
        picks = rng.choice(numbers, size=n)
        picks[rng.random(n) < 0.2] = picks[0]  # lanes holding the same element
        cands = [(np.float32(row[i]), int(i)) for i in picks]
        want = cands[0]
        for o in cands[1:]:
            want = merge(want, o, op)
        got = redux_merge32(cands, op)
        assert got[1] == want[1] and (got[0] == want[0] or (got[0] != got[0] and want[0] != want[0])), (trial, op)
    # x[0] NaN: every candidate is (x[0], 0)
    nan = np.float32(np.nan)
    assert redux_merge32([(nan, 0)] * 32, op)[1] == 0
    # the binary64 two-word reduction selects exactly the lanes with the largest key
    for trial in range(2000):
        n = int(rng.integers(1, 33))
        keys = rng.integers(0, 4, size=n).astype(np.uint64) << np.uint64(32)
        keys |= rng.integers(0, 3, size=n).astype(np.uint64)
        assert (redux_has64(keys) == (keys == keys.max())).all()
