"""CPU-only checks of the C-ABI library: it builds, loads, exports every
symbol include/argreduce.h declares, validates arguments before touching the
device, and its planner (pure host code) produces sound geometry."""
import ctypes
import os
import re

import numpy as np
import pytest

import row_wise_arg_gb300 as A
from row_wise_arg_gb300 import _lib
from row_wise_arg_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "argreduce.h")
INT_MAX = 2**31 - 1


@pytest.fixture(scope="module", autouse=True)
def built():
    build()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*[A-Za-z_][\w \*]*?\b(argreduce\w*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_expected_entry_points():
    names = header_functions()
    assert set(_lib.EXPORTS) <= set(names), names
    assert "argreduce" in names and "argreduce_scratch_bytes" in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib.LIB_PATH)
    for name in header_functions():
        assert hasattr(lib, name), f"{name} declared in argreduce.h but not exported"


def test_version_and_status_strings():
    assert "sm_103a" in A.argreduce_version()
    for s in range(6):
        assert A.argreduce_status_string(s).startswith("ARGR_")
    assert "unknown" in A.argreduce_status_string(99)


def test_validation_before_any_device_work():
    """Bad arguments are rejected before the library asks for a device (this
    machine has none, so anything reaching the device would be ECUDA)."""
    f = _lib.argreduce_raw
    X = 0x10000  # a fake, never dereferenced address
    assert f(X, "f32", 0, 5, "max", X, 0, 0, 0, 0) == _lib.ARGR_OK  # rows == 0: nothing to do
    assert f(0, "f32", 3, 5, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # null x
    assert f(X, "f32", 3, 5, "max", 0, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # null out_idx
    assert f(X, "f32", 3, 0, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # cols == 0
    assert f(X, "f32", 3, INT_MAX + 1, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # cols > INT_MAX
    assert f(X, "f32", -1, 5, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # rows < 0
    assert f(X, 7, 3, 5, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # bad dtype
    assert f(X, "f32", 3, 5, 9, X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # bad op
    assert f(X, "f32", 3, 5, 4, X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # bad op
    assert f(X, "f32", 0, 5, "max_last", X, 0, 0, 0, 0) == _lib.ARGR_OK  # last-index ops are valid
    assert f(X + 2, "f32", 3, 5, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # x not element aligned
    assert f(X, "f32", 3, 5, "max", X + 4, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # out_idx not 8-aligned
    assert f(X, "f64", 3, 5, "max", X, X + 4, 0, 0, 0) == _lib.ARGR_EINVAL  # out_val not aligned
    assert f(X, "f32", 2**62, 2**20, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL  # byte size overflows
    assert A.argreduce_scratch_init(X + 8, 64, 0) == _lib.ARGR_ESCRATCH
    assert A.argreduce_scratch_init(0, 64, 0) == _lib.ARGR_EINVAL
    assert A.argreduce_scratch_init(0, 0, 0) == _lib.ARGR_OK


GB300 = A.make_caps(152)
H200_LIKE = A.make_caps(132)
TINY = A.make_caps(2, 2048)

CONFIG_SHAPES = [(1, 32000), (1, 202048), (1, 262144), (8, 202048), (32, 202048), (4096, 4096),
                 (65536, 1024), (65536, 64), (4096, 8), (4096, 128), (2048, 8192), (8192, 2048)]


@pytest.mark.parametrize("caps", [GB300, H200_LIKE, TINY], ids=["152sm", "132sm", "2sm"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "f64"])
def test_plan_geometry(caps, dtype):
    es = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8}[dtype]
    wave = caps.sm_count * (caps.max_threads_per_sm // 256)
    for rows, cols in CONFIG_SHAPES + [(1, 1), (3, 7), (1, INT_MAX), (70000, 3), (2, 5000)]:
        p = A.argreduce_plan(rows, cols, dtype, "max", caps)
        d = p.as_dict()
        assert d["block"] % 32 == 0 and 32 <= d["block"] <= 1024
        if d["flags"] & _lib.ARGR_PLAN_PIPELINE:  # what check_plan admits for pipelined loads
            assert d["path_name"] == "rows" and d["vec"] == 1 and d["group"] >= 16 and d["block"] <= 256
        if d["path_name"] == "rows":
            assert d["group"] in (1, 2, 4, 8, 16, 32)
            if d["vec"]:
                assert (cols * es) % 16 == 0
            assert d["scratch_bytes"] == 0
        elif d["path_name"] == "cluster":
            assert 2 <= d["cluster"] <= 16 and d["blocks_per_row"] == d["cluster"]
            assert rows * d["cluster"] <= 2 * caps.sm_count and d["scratch_bytes"] == 0
        elif d["path_name"] == "split":
            bpr = d["blocks_per_row"]
            assert 1 <= bpr <= 65535 and 1 <= d["grid_rows"] <= 65535
            if bpr > 1:
                assert d["grid_rows"] >= rows
                # about one wave, and the scratch stays in the kilobytes
                assert rows * bpr <= max(wave, rows)
                assert d["scratch_bytes"] <= 256 + 4 * 2048 + 16 * max(wave, rows)
                assert d["grid_rows"] <= 2048
            else:
                assert d["scratch_bytes"] == 0
        else:
            pytest.fail(f"unexpected path {d}")


def test_plan_paths_for_configs():
    """The planner's choices for the five workload groups on a 152-SM part."""
    def path(rows, cols, dt="f32"):
        return A.argreduce_plan(rows, cols, dt, "max", GB300).as_dict()

    for rows, cols in ((1, 32000), (1, 202048), (1, 262144), (8, 202048), (32, 202048)):
        d = path(rows, cols)
        assert d["path_name"] == "cluster" and d["cluster"] >= 8, d
        assert rows * d["cluster"] <= 2 * 152 and d["scratch_bytes"] == 0
        assert d["flags"] & _lib.ARGR_PLAN_PDL
        if rows == 1:  # one batch of loads covers a CTA's share
            assert d["unroll"] * d["block"] * 16 * d["cluster"] >= cols * 4
    # 16 KB or more per CTA: 512 threads (one row too, with 8 loads each); smaller shares: fewer
    assert path(1, 202048)["block"] == 512 and path(1, 262144)["block"] == 512
    assert path(1, 202048)["unroll"] == 8 and path(1, 32000)["block"] == 256
    assert path(1, 202048, "bf16")["block"] == 512 and path(8, 202048)["block"] == 512
    d = path(1, 10_000_000)  # too wide for one cluster: split over the device
    assert d["path_name"] == "split" and d["blocks_per_row"] > 152
    assert path(4096, 4096)["path_name"] == "rows" and path(4096, 4096)["group"] == 32
    for cols in (8, 64, 128):
        d = path(65536 if cols == 64 else 4096, cols)
        assert d["path_name"] == "rows" and d["vec"] == 1 and d["group"] <= 8
    # narrow vector rows: 128-thread CTAs when 256-thread ones would not reach every SM
    assert path(4096, 8)["block"] == 128 and path(4096, 8)["grid_rows"] == 32
    assert path(4096, 128)["block"] == 128 and path(16384, 32)["block"] == 128
    assert path(65536, 64)["block"] == 256 and path(65536, 64)["grid_rows"] == 608
    assert path(30000, 100)["block"] == 256 and path(4096, 9)["block"] == 256  # many CTAs; scalar rows
    # medium rows: warp per row from 4 KB of binary32; pipelined loads from
    # 16 KB (binary32) / 32 KB (binary64) rows, 8 deep while the rows fit
    # 16 warps per SM, else 4 deep
    pipe = _lib.ARGR_PLAN_PIPELINE
    d = path(65536, 1024)
    assert d["group"] == 32 and not d["flags"] & pipe and d["unroll"] == 8
    d = path(65536, 1024, "f64")
    assert d["group"] == 16 and not d["flags"] & pipe
    d = path(4096, 4096)
    assert d["group"] == 32 and d["flags"] & pipe and d["unroll"] == 4 and d["block"] == 128
    d = path(2048, 8192)
    assert d["group"] == 32 and d["flags"] & pipe and d["unroll"] == 8
    d = path(4096, 4096, "f64")
    assert d["group"] == 32 and d["flags"] & pipe and d["unroll"] == 4 and d["block"] == 256
    d = path(8192, 2048, "f64")
    assert d["group"] == 32 and not d["flags"] & pipe
    assert not path(4096, 4095)["flags"] & pipe  # rows not 16-byte aligned: no vector loads
    # 16-bit rows: a warp from 4 KB, 256-thread CTAs from 16 KB, no pipelining
    d = path(8192, 4096, "f16")
    assert d["group"] == 32 and d["block"] == 128 and not d["flags"] & pipe
    d = path(4096, 8192, "bf16")
    assert d["group"] == 32 and d["block"] == 256 and not d["flags"] & pipe
    # rows below one wave: a row is shared by CTAs only in pieces of 32 KB or more
    for rows, cols, dt in ((256, 8192, "f32"), (512, 4096, "f64")):
        d = path(rows, cols, dt)
        assert d["path_name"] == "split" and d["blocks_per_row"] == 1 and d["block"] == 256, d
    d = path(1024, 8192)
    assert d["path_name"] == "split" and d["blocks_per_row"] == 1 and d["block"] == 128
    d = path(1024, 4096, "f64")  # 32 KB rows of 4096 elements: pipelined warp per row
    assert d["path_name"] == "rows" and d["group"] == 32 and d["flags"] & pipe and d["unroll"] == 8
    assert path(1024, 4095, "f64")["path_name"] == "split"  # not aligned
    d = path(256, 202048)
    assert d["path_name"] == "split" and d["blocks_per_row"] == 4


def test_split_rows_capped():
    """A multi-CTA split never uses more row slots than the scratch has
    counters (2048), even on a device whose wave holds more rows."""
    big = A.make_caps(2000)
    for rows in (2047, 2048, 2049, 5000):
        d = A.argreduce_plan(rows, 100000, "f32", "max", big).as_dict()
        if d["blocks_per_row"] > 1:
            assert d["grid_rows"] == rows <= 2048


def test_plan_rejects_bad_input():
    with pytest.raises(A.ArgreduceError):
        A.argreduce_plan(1, 0, "f32", "max", GB300)
    with pytest.raises(A.ArgreduceError):
        A.argreduce_plan(1, 10, "f32", "max", A.make_caps(0))
    assert A.argreduce_plan(0, 10, "f32", "max", GB300).as_dict()["path_name"] == "none"


# ---------------------------------------------------------------------------
# Host simulation of the kernels' index arithmetic.
# ---------------------------------------------------------------------------
class Overflow(Exception):
    pass


def i32(v):
    if not (-2**31 <= v < 2**31):
        raise Overflow(v)
    return v


def sim_split_thread(cols, es, misalign, b, nb, t, nt, U, count_only=False):
    """Positions one thread of scan_share() visits, computed with the same
    int operations (each checked for int32 overflow)."""
    E = 16 // es
    head = ((16 - misalign) & 15) // es
    head = min(head, cols)
    nvec = i32(i32(cols - head) // E)
    tail0 = i32(head + i32(nvec * E))
    chunk = i32(nvec // nb + (1 if nvec % nb else 0))
    bc = i32(b * chunk)
    vb = bc if bc < nvec else nvec
    ve = i32(vb + chunk) if i32(nvec - vb) > chunk else nvec
    out = []
    n = 0
    if b == 0 and t < head:
        out.append(t)
    v0 = i32(vb + t)
    if v0 < ve:
        while True:
            rem = i32(ve - v0)
            for u in range(U):
                if i32(u * nt) < rem:
                    j0 = i32(head + i32(i32(v0 + u * nt) * E))
                    n += E
                    if not count_only:
                        out.extend(range(j0, j0 + E))
                    else:
                        assert 0 <= j0 and j0 + E <= cols
            if rem <= i32(U * nt):
                break
            if count_only:
                # jump to the last iteration without changing the arithmetic
                steps = (rem - 1) // (U * nt)
                v0 = i32(v0 + steps * U * nt)
                n += (steps - 1) * U * E if steps > 1 else 0
                continue
            v0 = i32(v0 + U * nt)
    if b == nb - 1 and t < cols - tail0:
        out.append(i32(tail0 + t))
    return out, n


@pytest.mark.parametrize("es", [2, 4, 8])
def test_split_partition_exact_small(es):
    """Every element of the row is visited exactly once, in increasing order
    per thread, for many widths, misalignments and CTA counts."""
    for cols in list(range(1, 70)) + [127, 128, 129, 255, 256, 257, 1000, 4099]:
        for misalign in range(0, 16, es):
            for nb in (1, 2, 3, 7):
                for nt, U in ((32, 1), (64, 2), (32, 4)):
                    seen = []
                    for b in range(nb):
                        for t in range(nt):
                            pos, _ = sim_split_thread(cols, es, misalign, b, nb, t, nt, U)
                            assert pos == sorted(pos)
                            seen.extend(pos)
                    assert sorted(seen) == list(range(cols)), (cols, misalign, nb, nt, U)


@pytest.mark.parametrize("cols", [INT_MAX, INT_MAX - 1, INT_MAX - 262143, 2**30 + 5])
@pytest.mark.parametrize("es", [2, 4, 8])
def test_split_index_arithmetic_at_int_max(cols, es):
    """The widest rows: no int32 intermediate overflows and every position
    stays inside [0, cols), for the first, last and boundary threads."""
    for nb in (1, 197, 1184):
        for nt, U in ((256, 4), (1024, 8)):
            for b in (0, 1, nb // 2, nb - 1):
                for t in (0, 1, nt - 1):
                    for misalign in (0, es, 16 - es):
                        sim_split_thread(cols, es, misalign, b, nb, t, nt, U, count_only=True)


def sim_rows_lane(cols, es, vec, G, U, lg):
    E = 16 // es if vec else 1
    n = i32(cols // E) if vec else cols
    v0 = lg
    rem = i32(n - v0)
    out = []
    while True:
        for u in range(U):
            if i32(u * G) < rem:
                idx = i32(v0 + u * G)
                out.extend(range(i32(idx * E), i32(idx * E) + E))
        if not rem > i32(G * U):
            break
        v0 = i32(v0 + G * U)
        rem = i32(n - v0)
    return out


def sim_rows_pipe_lane(nvec, G, U, lg):
    """Vectors one lane of the pipelined rows loop loads and visits (same
    arithmetic as rows_kernel with PIPE): returns (loaded, visited) in order."""
    v0 = lg
    rem = i32(nvec - v0)
    loaded = [i32(v0 + u * G) for u in range(U) if i32(u * G) < rem]
    visited = []
    while True:
        more = rem > i32(G * U)
        if more:
            v1 = i32(v0 + G * U)
            rem1 = i32(nvec - v1)
            loaded.extend(i32(v1 + u * G) for u in range(U) if i32(u * G) < rem1)
        visited.extend(i32(v0 + u * G) for u in range(U) if i32(u * G) < rem)
        if not more:
            break
        v0, rem = v1, rem1
    return loaded, visited


def test_rows_pipeline_partition_exact():
    for G in (16, 32):
        for U in (4, 8):
            for nvec in range(1, 600):
                seen = []
                for lg in range(G):
                    loaded, visited = sim_rows_pipe_lane(nvec, G, U, lg)
                    assert loaded == visited and visited == sorted(visited)
                    assert all(0 <= v < nvec for v in loaded)
                    seen.extend(visited)
                assert sorted(seen) == list(range(nvec))
    # v1 = v0 + G*U is formed only while it stays below nvec = cols / E, and a
    # 16-byte vector holds E >= 2 elements, so nvec <= INT32_MAX / 2: no overflow.
    assert (2**31 - 1) // 2 + 32 * 8 < 2**31


def test_rows_partition_exact():
    for es in (2, 4, 8):
        for G in (1, 2, 4, 8, 16, 32):
            for cols in range(1, 300):
                for vec in (False, True):
                    if vec and (cols * es) % 16:
                        continue
                    seen = []
                    for lg in range(G):
                        pos = sim_rows_lane(cols, es, vec, G, 4, lg)
                        assert pos == sorted(pos)
                        seen.extend(pos)
                    assert sorted(seen) == list(range(cols))


def sim_stream_pieces(rows, row_bytes, stage_bytes, n_warps):
    """Byte ranges the stream kernel's warps copy (same arithmetic as
    stream_piece()): every 16-byte unit of the matrix exactly once, every copy
    16-byte aligned, a multiple of 16 bytes, at most one stage, in bounds."""
    covered = bytearray(rows * row_bytes // 16)
    for gw in range(n_warps):
        r0, r1 = rows * gw // n_warps, rows * (gw + 1) // n_warps
        rpp = stage_bytes // row_bytes if row_bytes <= stage_bytes else 0
        ppr = 1 if rpp else -(-row_bytes // stage_bytes)
        total = -(-(r1 - r0) // rpp) if rpp else (r1 - r0) * ppr
        for q in range(total):
            if rpp:
                row = r0 + q * rpp
                off, nbytes = 0, min(rpp, r1 - row) * row_bytes
            else:
                row, j = r0 + q // ppr, q % ppr
                off = j * stage_bytes
                nbytes = min(stage_bytes, row_bytes - off)
            start = row * row_bytes + off
            assert 0 < nbytes <= stage_bytes and nbytes % 16 == 0 and start % 16 == 0
            assert start + nbytes <= rows * row_bytes
            for u in range(start // 16, (start + nbytes) // 16):
                assert covered[u] == 0
                covered[u] = 1
    assert all(covered)


def test_stream_piece_mapping():
    for rows in (1, 2, 7, 33, 300):
        for row_bytes in (16, 32, 64, 256, 1008, 4000, 8192, 16384, 80000):
            for stage_bytes in (1024, 4096, 8192):
                for n_warps in (1, 3, 40, 64):
                    sim_stream_pieces(rows, row_bytes, stage_bytes, n_warps)


# ---------------------------------------------------------------------------
# Host simulation of the binary64 integer keys and their high-word pre-test.
# ---------------------------------------------------------------------------
M64 = (1 << 64) - 1
SIGN = 1 << 63
INF_BITS = 0x7FF0000000000000


def f64_bits(v):
    import struct
    return struct.unpack("<Q", struct.pack("<d", v))[0]


def key64(b, is_min):
    """TagF64::order_key(): negative values to -b (two's complement), positive
    ones to b with the sign bit set; ArgMin takes the key of the negated value."""
    if is_min:
        b ^= SIGN
    s = M64 if b & SIGN else 0
    return (((b ^ s) - s) & M64) ^ (~s & SIGN)


def limit64(is_min):
    return 0xFFF0000000000000


def elem_key(b, is_min):
    return 0 if (b & ~SIGN & M64) > INF_BITS else key64(b, is_min)


def seed_key(b, is_min):
    return M64 if (b & ~SIGN & M64) > INF_BITS else key64(b, is_min)


def row_scan_takes(b, cand_key, is_min, last):
    """The row scans' f64 update test (no NaN test, one limit comparison)."""
    k = key64(b, is_min)
    return k <= limit64(is_min) and (k > cand_key or (last and k == cand_key))


def test_f64_keys_and_row_scan_test():
    import math
    import random
    specials = [0.0, -0.0, 5e-324, -5e-324, 2.2250738585072014e-308, -2.2250738585072014e-308, 1.0, -1.0,
                1.0000000000000002, 0.9999999999999999, -1.0000000000000002, 1.7976931348623157e308,
                -1.7976931348623157e308, math.inf, -math.inf, 2.0 ** -1022, 3.0, -3.0]
    rnd = random.Random(7)
    vals = [f64_bits(v) for v in specials] + [rnd.getrandbits(64) for _ in range(300)]
    vals += [0x7FF8000000000000, 0xFFF8000000000000, 0x7FF0000000000001, 0x8000000000000001, 0x8000000100000000,
             0x0000000100000000, 0x7FFFFFFFFFFFFFFF]
    import struct
    dv = {b: struct.unpack("<d", struct.pack("<Q", b))[0] for b in vals}
    for is_min in (False, True):
        for a in vals:
            for b in vals:
                xa, xb = dv[a], dv[b]
                better = (xa < xb) if is_min else (xa > xb)      # element a strictly better than candidate b
                equal = xa == xb                                  # IEEE equality (false on NaN)
                ka, kb = elem_key(a, is_min), seed_key(b, is_min)
                assert (ka > kb) == better, (hex(a), hex(b), is_min)
                assert (ka == kb) == equal, (hex(a), hex(b), is_min)
                assert row_scan_takes(a, kb, is_min, False) == better, (hex(a), hex(b), is_min)
                assert row_scan_takes(a, kb, is_min, True) == (better or equal), (hex(a), hex(b), is_min)
    # the key range of the numbers and where the NaNs fall
    for is_min in (False, True):
        lo_key, hi_key = key64(f64_bits(-math.inf), is_min), key64(f64_bits(math.inf), is_min)
        if is_min:
            lo_key, hi_key = hi_key, lo_key
        assert hi_key == limit64(is_min) and lo_key >= 1
        for nan in (0x7FF0000000000001, 0x7FF8000000000000, 0x7FFFFFFFFFFFFFFF, 0xFFF0000000000001,
                    0xFFF8000000000000, 0xFFFFFFFFFFFFFFFF):
            k = key64(nan, is_min)
            assert k > hi_key or k < lo_key, (hex(nan), is_min)
    # the binary64 vector scan rebuilds a value from its key (VecScan<TagF64>::finish):
    # exact for every nonzero number; both zeros share a key and come back as one
    # of them, which is why cand_value() reads zeros back from the row
    for is_min in (False, True):
        for b in vals:
            if dv[b] != dv[b]:
                continue  # NaNs never become a scan's candidate through a key
            got = key_value64(key64(b, is_min), is_min)
            if b & ~SIGN & M64:
                assert got == b, (hex(b), is_min)
            else:
                assert got in (0, SIGN), (hex(b), is_min)


def key_value64(k, is_min):
    """Inverse of key64 on the numbers (VecScan<TagF64>::finish)."""
    b = (k ^ SIGN) if k & SIGN else ((0 - k) & M64)
    return b ^ SIGN if is_min else b


def test_axis_plans():
    caps = GB300
    p = A.argreduce_axis_plan(7, 1000, 1, "f32", "max", caps).as_dict()
    assert p["path_name"] != "axis"  # inner == 1: the last-axis planner
    for outer, R, inner, dt in [(1, 100000, 1000, "f32"), (1, 1000, 100000, "f32"), (64, 512, 256, "bf16"),
                                (128, 4096, 8, "f32"), (16, 2048, 384, "f64"), (3, 5, 7, "f16")]:
        d = A.argreduce_axis_plan(outer, R, inner, dt, "min", caps).as_dict()
        assert d["path_name"] == "axis" and d["scratch_bytes"] == 0
        assert 1 <= d["cluster"] <= 16 and d["block"] % 32 == 0 and d["block"] <= 1024
        if d["cluster"] > 1:
            assert d["grid_rows"] == outer
        v = (2 if dt == "f64" else 4) if d["vec"] else 1
        assert d["group"] in (1, 2, 4, 8, 16, 32)
        tiles = -(-inner // (d["group"] * v))
        assert (d["grid_rows"] * tiles * d["cluster"]) >= min(2 * 152, d["grid_rows"] * tiles)
    # warps along R: ~32 a SM for column segments below a line on a grid of a CTA per SM or more, else ~16
    blocks = {shape: A.argreduce_axis_plan(*shape, "max", caps).as_dict()["block"]
              for shape in [(64, 512, 256, "bf16"), (16, 2048, 384, "f64"), (1, 1000, 100000, "f32"),
                            (1, 100000, 1000, "f32"), (128, 4096, 8, "f32")]}
    assert list(blocks.values()) == [128, 224, 128, 640, 512], blocks
    with pytest.raises(A.ArgreduceError):
        A.argreduce_axis_plan(1, 0, 5, "f32", "max", caps)
    assert _lib.argreduce_axis_raw(0x10000, "f32", 0, 10, 5, "max", 0x10000, 0, 0, 0, 0) == _lib.ARGR_OK
    assert _lib.argreduce_axis_raw(0x10000, "f32", 2, 10, 0, "max", 0x10000, 0, 0, 0, 0) == _lib.ARGR_EINVAL


def test_cum_plans_and_validation():
    seen = set()
    for rows, cols, dt in [(1, 65536, "i64"), (1, 262144, "i64"), (64, 1024, "i64"), (1024, 64, "i64"),
                           (4, 16384, "i32"), (1, 65536, "f32"), (256, 256, "bf16"), (1, 3, "f64"),
                           (1, 16777216, "i64"), (64, 65536, "f32"), (600, 100000, "f16"), (1, 16384, "i64"),
                           (200, 30000, "f32"), (4096, 4096, "f32"), (65536, 256, "f32"), (256, 65536, "f32"),
                           (16, 1 << 20, "f64"), (128, 131072, "f64"), (100, 131072, "f32")]:
        d = A.argreduce_cum_plan(rows, cols, dt, "max", GB300).as_dict()
        seen.add((d["path_name"], d["cluster"] > 1))
        es = {"f32": 4, "f16": 2, "bf16": 2, "f64": 8, "i32": 4, "i64": 8}[dt]
        if d["path_name"] == "cum_split" and d["flags"] & 8:
            # ARGR_PLAN_STASH: inputs of 32 MiB and more, chunks that fit 80 KiB of shared memory
            chunks = d["blocks_per_row"]
            assert rows * cols * es >= 32 << 20 and -(-cols // chunks) * es <= 80 * 1024 and d["block"] == 512
            assert chunks >= -(-76 // rows) and rows * chunks <= 65536
            total = rows * chunks
            assert d["scratch_bytes"] == (256 if total <= 1024 else 1 << 20) + 8 * total
        elif d["path_name"] == "cum_split":
            # long rows, fewer than the SMs: 76..304 CTAs (38 for one row of <= 64K
            # elements, 608 of 256 threads for one row of 64 MiB or more), records of
            # one launch <= 1024
            chunks = d["blocks_per_row"]
            many = rows > 1 and rows * cols >= 1 << 24  # several long rows: up to 8 x 152 chunks
            assert rows < 152 and chunks >= 2 and rows * chunks <= (8 * 152 if many else 1024) and cols > 32768
            big = rows == 1 and cols * es >= 64 << 20
            assert rows * chunks <= (4 * 152 if big else 2 * 152 + 1 if rows == 1 else 8 * 152 if many else 1024)
            if big:
                assert d["block"] == 256
            floor = 38 if rows == 1 and cols <= 65536 else 76
            assert rows * chunks >= floor or cols // chunks < 1024 or chunks == 1024 // rows
            assert cols // chunks >= 512
            cap = 256 if big else 512 if rows == 1 else 128
            assert d["block"] in (64, 128, 256, 512) and d["block"] <= cap
            assert d["block"] * 7 >= -(-cols // chunks) or d["block"] == cap
            total = rows * chunks
            assert d["scratch_bytes"] == (256 if total <= 1024 else 1 << 20) + 8 * total and d["cluster"] == 1
            assert d["grid_rows"] == rows and cols > 32768 and (es == 8 or cols > 65536 or rows * 16 > 304)
        elif d["cluster"] > 1:
            # short rows, fewer than the SMs: one cluster per row
            assert d["path_name"] == "cum" and rows < 152 and d["cluster"] <= 16
            assert cols <= 32768 or (es <= 4 and cols <= 65536 and rows * 16 <= 304)
            assert d["block"] == (256 if cols <= 32768 else 1024)
            assert d["grid_rows"] == rows and d["scratch_bytes"] == 0
            assert d["blocks_per_row"] == d["cluster"]
        else:
            # one CTA per row: as many rows as SMs, or rows too short to split; 512
            # threads with fewer than two CTAs a SM and rows of two such tiles, 1024
            # from three quarters of a row per SM and rows of two such tiles
            assert d["path_name"] == "cum" and d["scratch_bytes"] == 0 and 32 <= d["block"] <= 1024
            assert rows >= 152 or cols < 4 * 7 * d["block"] or (d["block"] == 1024 and rows >= 114)
            assert (d["block"] == 512) == (152 <= rows < 304 and cols >= 2 * 512 * 7), (rows, cols)
            assert (d["block"] == 1024) == (114 <= rows < 152 and cols >= 2 * 1024 * 7), (rows, cols)
            if rows >= 4 * 152:
                assert d["block"] <= 128 and (d["block"] == 32 or d["block"] * 7 <= cols)
    assert seen == {("cum_split", False), ("cum", True), ("cum", False)}
    big = A.argreduce_cum_plan(1, 16777216, "i64", "max", GB300).as_dict()
    assert big["blocks_per_row"] == 608 and big["flags"] & 8 == 0  # the stash is a forced-plan option
    d = A.argreduce_cum_plan(1, 65536, "i64", "max", GB300).as_dict()  # the pages' 65536-element int64 row
    assert d["blocks_per_row"] == 38 and d["block"] == 256
    assert A.argreduce_cum_plan(1, 131072, "i64", "max", GB300).as_dict()["blocks_per_row"] == 76
    assert A.argreduce_cum_plan(4, 16384, "i32", "max", GB300).as_dict()["cluster"] == 16
    assert A.argreduce_cum_plan(4096, 4096, "f32", "max", GB300).as_dict()["block"] == 128
    assert A.argreduce_cum_plan(65536, 256, "f32", "max", GB300).as_dict()["block"] == 32
    with pytest.raises(A.ArgreduceError):
        A.argreduce_cum_plan(1, 10, "f32", "max_last", GB300)
    X = 0x10000
    assert _lib.argreduce_cum_raw(X, "i64", 0, 10, "max", X, 0, 0, 0, 0) == _lib.ARGR_OK
    assert _lib.argreduce_cum_raw(X, "i64", 2, 0, "max", X, 0, 0, 0, 0) == _lib.ARGR_EINVAL
    assert _lib.argreduce_cum_raw(X, "i64", 2, 10, "min_last", X, 0, 0, 0, 0) == _lib.ARGR_EUNSUPPORTED
    assert _lib.argreduce_raw(X, "i64", 2, 10, "max", X, 0, 0, 0, 0) == _lib.ARGR_EUNSUPPORTED


def test_cum_split_index_arithmetic():
    """Host simulation of the split scan's ticket, chunk and record arithmetic
    (the kernel's integer formulas, restated): tickets 0..total-1 map to
    distinct (row, chunk) pairs, every row's chunks partition [0, cols) in
    order (empty chunks allowed), every 8-byte record lies in the 8 KiB
    region after the 256-byte header and inside the plan's scratch, and a
    record's index + 1 never collides with 0 (unpublished) or 0xffffffff
    (empty chunk)."""
    for rows, cols, chunks in [(1, 65536, 18), (1, 5, 7), (3, 7, 5), (1024, 1, 1), (1, 2**31 - 1, 1024),
                               (2, 2**31 - 1, 512), (16, 65536, 64), (5, 4099, 204), (1, 2**31 - 1, 65536),
                               (16, 2**20, 4096), (1, 1025, 1025)]:
        total = rows * chunks
        assert total <= 65536
        region = 256 if total <= 1024 else 1 << 20
        if region == 256:
            assert region + 8 * total <= 8448  # inside the split counters' region
        else:
            # beyond every argreduce partial: 8448 + 16 * (grid_rows * blocks_per_row) <= 1 MiB
            assert 8448 + 16 * ((1 << 20) - 8448) // 16 <= region
        seen = set()
        for ticket in range(total):
            r, c = divmod(ticket, chunks)
            seen.add((r, c))
            word = region + 8 * (r * chunks + c)
            assert region <= word and word + 8 <= region + 8 * total
        assert len(seen) == total
        for c_ in range(chunks):
            cb = cols * c_ // chunks
            ce = cols * (c_ + 1) // chunks
            assert 0 <= cb <= ce <= cols and cb < 2**31 and ce < 2**31
            if c_ + 1 < chunks:
                assert ce == cols * (c_ + 1) // chunks  # the next chunk starts where this one ends
            if ce > cb:
                assert 1 <= (ce - 1) + 1 < 0xffffffff
        assert cols * chunks // chunks == cols
    # the wrapping counters: atom.inc with bound total-1 hands out 0..total-1 and ends at 0
    for total in (1, 2, 18, 1024, 65536):
        ctr, got = 0, []
        for _ in range(total):
            got.append(ctr)
            ctr = 0 if ctr >= total - 1 else ctr + 1
        assert got == list(range(total)) and ctr == 0




def test_cub_compare_library_exports():
    """The benchmark's comparison library (cub::DeviceReduce called as a
    library) is built beside libargreduce.so and exports its two entry points;
    libargreduce.so itself has no CUB symbol of ours."""
    import ctypes
    from row_wise_arg_gb300 import cub_compare
    lib = ctypes.CDLL(cub_compare.LIB_PATH)
    for name in ("cubcmp_temp_bytes", "cubcmp_argreduce"):
        assert hasattr(lib, name)
    assert not hasattr(_lib.load(), "cubcmp_argreduce")


def _stash_fill_plan(g0, n, es, stash_bytes=80 * 1024, piece=16384):
    """The split scan's stash arithmetic (stash_fill), restated: the chunk
    [g0, g0 + n*es) goes to shared offset (g0 % 16) onward; its 16-byte
    aligned middle by bulk copies of at most `piece` bytes, the head and the
    tail element by element."""
    g1 = g0 + n * es
    a0 = (g0 + 15) & ~15
    a1 = g1 & ~15
    bulk = a1 > a0
    head = (a0 - g0) // es if bulk else n
    tail = (a1 - g0) // es if bulk else n
    stash = g0 & 15  # shared offset of element 0 of the chunk
    copies = []
    if bulk:
        dst = stash + (a0 - g0)
        off = 0
        while off < a1 - a0:
            ln = min(piece, a1 - a0 - off)
            copies.append((dst + off, a0 + off, ln))
            off += ln
    return head, tail, stash, copies


def test_cum_stash_fill_arithmetic():
    """Every element of a stashed chunk is written exactly once (head and tail
    by threads, the middle by bulk copies whose global and shared addresses
    and sizes are multiples of 16, at most 16 KiB each), and the stash stays
    within its 80 KiB + 16 bytes of shared memory, before the tile indices."""
    stash_bytes = 80 * 1024
    for es in (2, 4, 8):
        cap = stash_bytes // es
        for phase in range(0, 16, es):
            for n in (1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 100, 4095, cap - 1, cap):
                g0 = 0x7f0000000000 + 4096 * 3 + phase
                head, tail, stash, copies = _stash_fill_plan(g0, n, es)
                covered = np.zeros(n, dtype=np.int64)
                covered[:head] += 1
                covered[tail:] += 1
                for dst, src, ln in copies:
                    assert dst % 16 == 0 and src % 16 == 0 and ln % 16 == 0 and 0 < ln <= 16384
                    first = (src - g0) // es
                    assert (src - g0) % es == 0 and dst - stash == src - g0
                    covered[first:first + ln // es] += 1
                assert (covered == 1).all(), (es, phase, n)
                assert 0 <= head <= tail <= n and (head == n) == (not copies)
                assert stash + n * es <= stash_bytes + 16  # the tile indices start at stash_bytes + 16
                assert len(copies) <= 5


def test_cum_lookback_scratch_size():
    """A look-back split scan keeps two record words per chunk ([aggregate,
    inclusive prefix]); past 1024 words they move 1 MiB into the buffer."""
    for rows, chunks, want in ((1, 76, 256 + 16 * 76), (1, 512, 256 + 16 * 512), (1, 513, (1 << 20) + 16 * 513),
                               (4, 4681, (1 << 20) + 16 * 4 * 4681)):
        p = _lib.argr_plan()
        p.path, p.block, p.cluster, p.blocks_per_row, p.grid_rows = _lib.ARGR_PATH_CUM_SPLIT, 512, 1, chunks, rows
        p.flags = _lib.ARGR_PLAN_PDL | _lib.ARGR_PLAN_LOOKBACK
        assert _lib.argreduce_plan_scratch_bytes(p, rows) == want
        p.flags = _lib.ARGR_PLAN_PDL
        assert _lib.argreduce_plan_scratch_bytes(p, rows) == (256 if rows * chunks <= 1024 else 1 << 20) + 8 * rows * chunks


def test_cum_stream_scratch_size():
    """The streaming scan keeps [aggregate, inclusive prefix] per tile."""
    for rows, cols, block, want in ((1, 65536, 512, 256 + 16 * 19), (1, 1 << 24, 512, (1 << 20) + 16 * 4682),
                                    (3, 1 << 20, 1024, 256 + 16 * 3 * 147)):
        p = _lib.argr_plan()
        p.path, p.block, p.cluster, p.grid_rows = _lib.ARGR_PATH_CUM_STREAM, block, 1, 304
        p.blocks_per_row = -(-cols // (block * 7))
        assert _lib.argreduce_plan_scratch_bytes(p, rows) == want


def test_warp_collectives_not_short_circuited():
    """Every lane named in a warp collective's mask must execute it, or the
    others wait for it forever. A collective written after `&&`, `||` or `?`
    in the same expression is skipped by the lanes that short-circuit, so
    device code computes collectives into variables first."""
    import glob
    pat = re.compile(r"(&&|\|\||\?)[^;{}]*\b__\w+_sync\(")
    bad = []
    for path in sorted(glob.glob(os.path.join(ROOT, "row_wise_arg_gb300", "csrc", "*.cu*"))):
        for n, line in enumerate(open(path), 1):
            code = line.split("//")[0]
            if pat.search(code):
                bad.append(f"{os.path.basename(path)}:{n}: {line.strip()}")
    assert not bad, bad


def test_plan_check_without_a_gpu():
    """argreduce_plan_check() applies argreduce_with_plan()'s checks against
    simulated device properties: the planner's own plans always pass, and each
    rule of a forced plan is enforced (ARGR_PLAN_PIPELINE only on vector rows
    plans with 16 or 32 lanes and at most 256 threads)."""
    from row_wise_arg_gb300 import _lib as L
    rng = np.random.Generator(np.random.PCG64(77))
    shapes = CONFIG_SHAPES + [(1, 1), (3, 7), (2, 5000), (70000, 3), (1024, 4096), (256, 8192), (512, 8192)]
    shapes += [(int(rng.integers(1, 5000)), int(rng.integers(1, 300000))) for _ in range(40)]
    for caps in (GB300, H200_LIKE, TINY):
        for dt in ("f32", "f16", "bf16", "f64"):
            for rows, cols in shapes:
                p = A.argreduce_plan(rows, cols, dt, "max", caps)
                assert A.argreduce_plan_check(p, rows, cols, dt, caps) == L.ARGR_OK, (rows, cols, dt, p)

    def rows_plan(group=32, vec=1, block=128, unroll=4, pipe=True):
        p = L.argr_plan()
        p.path, p.group, p.vec, p.block, p.unroll = L.ARGR_PATH_ROWS, group, vec, block, unroll
        p.flags = L.ARGR_PLAN_PDL | (L.ARGR_PLAN_PIPELINE if pipe else 0)
        p.grid_rows, p.blocks_per_row = 64, 1
        return p

    chk = lambda p, aligned=True, rows=4096, cols=4096: A.argreduce_plan_check(p, rows, cols, "f32", GB300, aligned)
    assert chk(rows_plan()) == L.ARGR_OK
    assert chk(rows_plan(group=16, block=256, unroll=8)) == L.ARGR_OK
    assert chk(rows_plan(group=8)) == L.ARGR_EINVAL          # pipelined: 16 or 32 lanes per row
    assert chk(rows_plan(vec=0)) == L.ARGR_EINVAL            # pipelined: vector loads only
    assert chk(rows_plan(block=512)) == L.ARGR_EINVAL        # pipelined: at most 256 threads
    assert chk(rows_plan(pipe=False, block=512)) == L.ARGR_OK
    assert chk(rows_plan(pipe=False), aligned=False) == L.ARGR_EINVAL  # vector loads need aligned rows
    assert chk(rows_plan(pipe=False, vec=0), aligned=False) == L.ARGR_OK
    assert chk(rows_plan(pipe=False, unroll=5)) == L.ARGR_EINVAL
    assert chk(rows_plan(pipe=False, group=3)) == L.ARGR_EINVAL
    assert chk(rows_plan(), rows=0) == L.ARGR_OK             # nothing to launch
    sp = L.argr_plan()
    sp.path, sp.block, sp.unroll, sp.blocks_per_row, sp.grid_rows = L.ARGR_PATH_SPLIT, 256, 4, 4, 4
    sp.flags = L.ARGR_PLAN_PDL
    assert chk(sp, rows=4, cols=1 << 20) == L.ARGR_OK
    sp.flags |= L.ARGR_PLAN_PIPELINE
    assert chk(sp, rows=4, cols=1 << 20) == L.ARGR_EINVAL    # pipelining is a rows-path flag
    sp.flags = L.ARGR_PLAN_PDL
    sp.grid_rows = 2
    assert chk(sp, rows=4, cols=1 << 20) == L.ARGR_EINVAL    # a split row may not loop
    cp = L.argr_plan()
    cp.path, cp.block, cp.unroll, cp.cluster, cp.blocks_per_row, cp.grid_rows = L.ARGR_PATH_CLUSTER, 512, 8, 16, 16, 1
    assert chk(cp, rows=1, cols=202048) == L.ARGR_OK
    assert A.argreduce_plan_check(cp, 1, 202048, "f32", A.make_caps(152, max_cluster=8)) == L.ARGR_EUNSUPPORTED
    cp.cluster = cp.blocks_per_row = 17
    assert chk(cp, rows=1, cols=202048) == L.ARGR_EINVAL
    # the test hook of the push merge's bounded wait: a row slot per row, no bulk copies
    cp.cluster = cp.blocks_per_row = 16
    cp.flags = L.ARGR_PLAN_PDL | L.ARGR_PLAN_TEST_EXPIRE
    assert chk(cp, rows=1, cols=202048) == L.ARGR_OK
    assert chk(cp, rows=2, cols=202048) == L.ARGR_EINVAL     # rows loop: barrier merge, no such wait
    cp.flags |= L.ARGR_PLAN_BULK
    assert chk(cp, rows=1, cols=202048) == L.ARGR_EINVAL


def test_prefetch_flag_rules():
    """ARGR_PLAN_PREFETCH: set by the planner for inputs of at most 32 MiB,
    and with ARGR_PLAN_PREFETCH_HEAD (16 KiB a CTA) for larger inputs on the
    rows path; admitted on the rows, split, cluster and streaming paths only
    (not with the cluster's bulk copies, not on the non-last-axis path), the
    head variant on the rows path only."""
    from row_wise_arg_gb300 import _lib as L
    PF, HEAD = L.ARGR_PLAN_PREFETCH, L.ARGR_PLAN_PREFETCH_HEAD
    for dt, es in (("f32", 4), ("bf16", 2), ("f64", 8)):
        for rows, cols in CONFIG_SHAPES + [(1, 1), (5, 7), (2048, 4096), (2049, 4096), (8, 1 << 20), (9, 1 << 20),
                                           (1024, 16384), (1 << 20, 64)]:
            p = A.argreduce_plan(rows, cols, dt, "max", GB300)
            small = rows * cols * es <= 32 << 20
            head = not small and p.path == L.ARGR_PATH_ROWS and cols * es > 1024
            assert bool(p.flags & PF) == (small or head), (rows, cols, dt)
            assert bool(p.flags & HEAD) == head, (rows, cols, dt)
            assert A.argreduce_plan_check(p, rows, cols, dt, GB300) == L.ARGR_OK
    for rows, cols, dt in ((4096, 4096, "f32"), (4096, 4096, "f64"), (65536, 1024, "f32"), (65536, 1024, "f64")):
        assert A.argreduce_plan(rows, cols, dt, "max", GB300).flags & HEAD, (rows, cols, dt)
    chk = lambda p, rows=4, cols=1 << 16: A.argreduce_plan_check(p, rows, cols, "f32", GB300, True)
    cp = L.argr_plan()
    cp.path, cp.block, cp.unroll, cp.cluster, cp.blocks_per_row, cp.grid_rows = L.ARGR_PATH_CLUSTER, 256, 4, 4, 4, 4
    cp.flags = L.ARGR_PLAN_PDL | PF
    assert chk(cp) == L.ARGR_OK
    cp.flags |= L.ARGR_PLAN_BULK
    assert chk(cp) == L.ARGR_EINVAL                      # bulk copies already fetch the share
    st = L.argr_plan()
    st.path, st.block, st.group, st.stages, st.stage_bytes, st.grid_rows = L.ARGR_PATH_STREAM, 128, 32, 2, 8192, 8
    st.vec, st.flags = 1, L.ARGR_PLAN_PDL
    assert chk(st) == L.ARGR_OK
    st.flags |= PF
    assert chk(st) == L.ARGR_OK                          # its CTA's rows, before the wait
    st.flags |= L.ARGR_PLAN_BULK
    assert chk(st) == L.ARGR_EINVAL                      # bulk flag: cluster plans only
    rp = A.argreduce_plan(4096, 4096, "f32", "max", GB300)
    assert chk(rp, rows=4096, cols=4096) == L.ARGR_OK
    rp.flags &= ~PF
    assert chk(rp, rows=4096, cols=4096) == L.ARGR_EINVAL  # the head variant of a prefetch
    cp.grid_rows, cp.flags = 4, L.ARGR_PLAN_PDL | PF | HEAD
    assert chk(cp) == L.ARGR_EINVAL                      # rows path only
    ax = A.argreduce_axis_plan(64, 512, 256, "bf16", "max", GB300)
    assert not ax.flags & PF


def test_bench_thread_per_row_plans_are_valid():
    """The thread-per-row plans bench.py times beside the narrow configs pass the
    library's own plan checks (scalar loads always, vector loads on aligned rows)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    from row_wise_arg_gb300 import _lib as L
    for c in W.config_cases(5):
        aligned = c.cols * W.ELEM_SIZE[c.dtype] % 16 == 0
        for vec in (False, True):
            p = bench.ThreadPerRowCalls(A, [c], vec).plans[0]
            assert p.group == 1 and p.path == L.ARGR_PATH_ROWS
            want = L.ARGR_OK if (aligned or not vec) else L.ARGR_EINVAL
            assert A.argreduce_plan_check(p, c.rows, c.cols, c.dtype, GB300, aligned) == want, (c.name, vec)
