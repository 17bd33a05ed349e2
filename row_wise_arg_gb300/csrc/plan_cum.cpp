// Launch-geometry planner for cummax / cummin with indices (argreduce_cum):
// a pure function of the problem and the device's properties, testable on a
// machine without a GPU. Paddle issue #79670 (launch-geometry analysis: a
// fixed block shape leaves a long innermost scan on one CTA; "Possible
// fixes": derive the block shape from (rows, row length) and route shapes
// that cannot fill the GPU to a two-pass tiled scan).
#include <algorithm>
#include <climits>

#include "internal.h"

namespace argr {

namespace {

constexpr int64_t kMaxGridY = 65535;                 // hardware limit of gridDim.y
constexpr int64_t kMaxDynamicSmem = 227 * 1024;      // dynamic shared memory one CTA may use

int64_t ceil_div(int64_t a, int64_t b) { return a / b + (a % b != 0); }

bool caps_ok(const argr_caps& c) { return c.sm_count > 0 && c.max_threads_per_sm >= 32; }

}  // namespace

// A CTA scans tiles of block * 7 elements (7 per thread); a row is one CTA's,
// a cluster's (up to 16 CTAs exchanging aggregates in distributed shared
// memory) or a split scan's (chunks exchanging aggregates through scratch).
static constexpr int kCumItems = 7;
// Measured on GB300 (sweeps of one-CTA, cluster and split geometries over
// rows of 256 to 16M elements): one CTA per row once there are as many rows as
// SMs (128 threads or fewer when rows are plentiful), clusters up to 32K
// elements per row, the split scan beyond, best at about one CTA per 3.5K
// elements: 76..304 CTAs of up to 512 threads for one row, up to 1024 CTAs of
// up to 128 threads for several.
static constexpr int64_t kCumManyRowsWaves = 4;     // rows per SM from which CTAs shrink
static constexpr int64_t kCumMinChunkTiles = 2;     // rows shorter than 2 x 2 tiles are not split
static constexpr int64_t kCumMinChunk = 512;        // elements per split-scan or cluster CTA at least
static constexpr int64_t kCumSplitElems = 3584;     // elements per split-scan CTA the planner aims for
static constexpr int64_t kCumClusterMaxCols = 32768;

argr_status make_cum_plan(int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps, argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    *out = argr_plan{};
    if (elem_size(dtype) == 0 || rows < 0 || cols < 1 || cols > INT_MAX) return ARGR_EINVAL;
    if (op != ARGR_MAX && op != ARGR_MIN) return (op == ARGR_MAX_LAST || op == ARGR_MIN_LAST) ? ARGR_EUNSUPPORTED
                                                                                                : ARGR_EINVAL;
    if (!caps_ok(caps)) return ARGR_EINVAL;
    if (rows == 0) {
        out->path = ARGR_PATH_NONE;
        return ARGR_OK;
    }
    const int64_t sms = caps.sm_count;
    out->flags = ARGR_PLAN_PDL;
    out->cluster = 1;
    out->blocks_per_row = 1;
    out->grid_rows = std::min(rows, kMaxGridY);
    out->path = ARGR_PATH_CUM;
    int block = 32;
    if (rows >= kCumManyRowsWaves * sms) {
        // Many rows: one CTA per row, small CTAs (more of them resident per
        // SM, fewer threads held by each barrier), at least two tiles a row.
        while (block < 128 && 2 * block * kCumItems <= cols) block <<= 1;
        out->block = block;
        return ARGR_OK;
    }
    while (block < 256 && block * kCumItems < cols) block <<= 1;
    out->block = block;
    const int64_t tile = static_cast<int64_t>(block) * kCumItems;
    if (rows >= sms && rows < 2 * sms && cols >= 2 * 512 * kCumItems) {
        // One CTA per row, fewer than two a SM: 512 threads, twice the loads
        // in flight on each SM ([256,65536] f32 51.0 -> 45.6 us, [160,100000]
        // i32 62.0 -> 54.6 us, [256,65536] f64 76.7 -> 75.6 us; with 512 rows
        // 256 threads stay faster, [512,32768] f32 46.1 against 48.7 us).
        out->block = 512;
        return ARGR_OK;
    }
    if (rows >= 3 * sms / 4 && rows < sms && cols >= 2 * 1024 * kCumItems) {
        // Almost a row per SM: one 1024-thread CTA per row instead of the
        // split scan ([128,131072] f32 56.6 -> 49.0 us, f64 91.7 -> 83.0,
        // [140,65536] i32 32.1 -> 27.5; with 64 rows the split stays much
        // faster, [64,131072] f32 29.2 against 45.8 us).
        out->block = 1024;
        return ARGR_OK;
    }
    if (cols < kCumMinChunkTiles * 2 * tile || rows >= sms) return ARGR_OK;  // one CTA per row
    const int64_t es = elem_size(dtype);
    const bool wide_cluster = es <= 4 && cols <= 2 * kCumClusterMaxCols && rows * 16 <= 2 * sms && caps.max_cluster >= 16;
    if ((cols <= kCumClusterMaxCols || wide_cluster) && caps.max_cluster >= 2) {
        // Short rows: a cluster per row exchanges aggregates through
        // distributed shared memory, a round trip cheaper than scratch. Up to
        // 64K elements of 4 bytes or less, while clusters of 16 fit, 1024-thread
        // CTAs keep each CTA's chunk in one tile ([1,65536] f32 7.9 -> 6.9 us);
        // the 64-bit scan kernels spill at that size and stay with the split
        // scan, and so do more rows ([64,65536] f32: clusters of 5 x 1024
        // 39 us, the split 26 us).
        const int64_t c = std::min<int64_t>({16, caps.max_cluster, ceil_div(2 * sms, rows),
                                             std::max<int64_t>(2, cols / kCumMinChunk)});
        out->block = cols <= kCumClusterMaxCols ? 256 : 1024;
        out->cluster = static_cast<int32_t>(c);
        out->blocks_per_row = c;
        out->grid_rows = rows;
        return ARGR_OK;
    }
    // Long rows, fewer than the SMs: a split scan with one CTA per
    // kCumSplitElems elements in total, from half an SM's worth up to two
    // 512-thread CTAs per SM for one row, or as many 128-thread CTAs as the
    // records allow for several rows.
    // One row of 64 MiB or more: four 256-thread chunks per SM, two waves, so
    // that the chunks in flight fit L2 and phase B's second read of a chunk
    // mostly hits it ([1,2^24] int64 107.4 -> 102.5 us, [1,2^25] f32 142.1 ->
    // 137.9 us against two 512-thread chunks per SM).
    const bool big_row = rows == 1 && cols * static_cast<int64_t>(elem_size(dtype)) >= (int64_t(64) << 20);
    // Several long rows of 2^24 elements or more in total: up to 8·SMs chunks
    // of 128 threads (above kCumMaxChunks the records move to the scratch's
    // 1 MiB region): [16,2^20] f64 108.5 -> 102.2 us with 76 chunks a row
    // instead of 64. Smaller inputs keep at most kCumMaxChunks.
    const int64_t many_max = rows * cols >= (int64_t(1) << 24) ? std::max<int64_t>(kCumMaxChunks, 8 * sms) : kCumMaxChunks;
    const int64_t max_ctas = big_row ? 4 * sms : rows == 1 ? 2 * sms : many_max;
    const int max_block = big_row ? 256 : rows == 1 ? 512 : 128;
    // One row of at most 64K elements: a quarter of the SMs, in 256-thread
    // CTAs instead of half of them in 128-thread CTAs ([1,65536] int64
    // 8.68 -> 8.63 us, f64 9.04 -> 8.87 us; one run, median of three).
    const int64_t floor_ctas = (rows == 1 && cols <= 65536) ? sms / 4 : sms / 2;
    const int64_t target = std::min(max_ctas, std::max(floor_ctas, ceil_div(rows * cols, kCumSplitElems)));
    // (ARGR_PLAN_LOOKBACK is not chosen either: one-tile chunks behind a serial
    // ticket / load / look-back / scan chain per CTA measured slower on long
    // rows, [1,2^24] int64 116 vs 110 us.)
    // (ARGR_PLAN_STASH is not chosen: stashing 80 KiB chunks reads the input
    // once but leaves two CTAs per SM alternating a load burst and a compute
    // burst, measured slower than re-reading from L2 or memory: [1,2^24]
    // int64 128 vs 111 us, [16,2^20] f64 131 vs 110 us.)
    const int64_t chunks = std::min<int64_t>({max_ctas / rows, ceil_div(target, rows), cols / kCumMinChunk});
    if (chunks < 2) return ARGR_OK;
    const int64_t per_chunk = ceil_div(cols, chunks);
    int b = 64;
    while (b < max_block && b * kCumItems < per_chunk) b <<= 1;
    out->path = ARGR_PATH_CUM_SPLIT;
    out->block = b;
    out->blocks_per_row = chunks;
    out->grid_rows = rows;
    out->scratch_bytes = plan_scratch(*out, rows);
    return ARGR_OK;
}

size_t cum_plan_scratch(const argr_plan& p, int64_t rows) {
    if (p.path != ARGR_PATH_CUM_SPLIT && p.path != ARGR_PATH_CUM_STREAM) return 0;
    const int64_t words =
        rows * p.blocks_per_row * ((p.path == ARGR_PATH_CUM_STREAM || (p.flags & ARGR_PLAN_LOOKBACK)) ? 2 : 1);
    return cum_records_offset(words) + 8 * static_cast<size_t>(words);
}

argr_status check_cum_plan(const argr_plan& p, int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps) {
    if (elem_size(dtype) == 0 || rows < 0 || cols < 1 || cols > INT_MAX) return ARGR_EINVAL;
    if (op != ARGR_MAX && op != ARGR_MIN) return ARGR_EUNSUPPORTED;
    if (rows == 0) return ARGR_OK;
    if (p.block < 32 || p.block > 1024 || p.block % 32 != 0) return ARGR_EINVAL;
    const int64_t smem = static_cast<int64_t>(p.block) * kCumItems * (elem_size(dtype) + 4);
    if (smem > kMaxDynamicSmem) return ARGR_EINVAL;
    if (p.path == ARGR_PATH_CUM_SPLIT) {
        if (p.flags & ~(ARGR_PLAN_PDL | ARGR_PLAN_TEST_EXPIRE | ARGR_PLAN_STASH | ARGR_PLAN_LOOKBACK))
            return ARGR_EINVAL;
        if ((p.flags & ARGR_PLAN_STASH) && (p.flags & ARGR_PLAN_LOOKBACK)) return ARGR_EINVAL;
        const int64_t words = (p.flags & ARGR_PLAN_LOOKBACK) ? 2 : 1;  // record words per chunk
        if (p.cluster != 1 || p.blocks_per_row < 1 || p.blocks_per_row > kCumMaxChunksBig / words) return ARGR_EINVAL;
        if (rows > kCumMaxChunksBig / words / p.blocks_per_row) return ARGR_EINVAL;  // records of one launch
        if (p.grid_rows != rows) return ARGR_EINVAL;
        if (p.flags & ARGR_PLAN_STASH) {
            // The largest chunk fits the stash; stash and tile indices fit one CTA.
            if (ceil_div(cols, p.blocks_per_row) * elem_size(dtype) > kCumStashBytes) return ARGR_EINVAL;
            if (kCumStashBytes + 16 + static_cast<int64_t>(p.block) * kCumItems * 4 > kMaxDynamicSmem)
                return ARGR_EINVAL;
        }
        return ARGR_OK;
    }
    if (p.path == ARGR_PATH_CUM_STREAM) {
        if (p.flags & ~(ARGR_PLAN_PDL | ARGR_PLAN_TEST_EXPIRE)) return ARGR_EINVAL;
        // exactly the tiles of a row; two record words per tile in one launch
        if (p.cluster != 1 || p.blocks_per_row != ceil_div(cols, static_cast<int64_t>(p.block) * kCumItems))
            return ARGR_EINVAL;
        if (rows > kCumMaxChunksBig / 2 / p.blocks_per_row) return ARGR_EINVAL;
        if (p.grid_rows < 1 || p.grid_rows > kMaxGridY) return ARGR_EINVAL;
        return ARGR_OK;
    }
    if (p.path != ARGR_PATH_CUM) return ARGR_EINVAL;
    if (p.flags & ~ARGR_PLAN_PDL) return ARGR_EINVAL;
    if (p.cluster < 1 || p.cluster > 16 || p.blocks_per_row != p.cluster) return ARGR_EINVAL;
    if (p.cluster > 1 && caps.max_cluster < p.cluster) return ARGR_EUNSUPPORTED;
    if (p.grid_rows < 1 || p.grid_rows > kMaxGridY) return ARGR_EINVAL;
    if (p.cluster > 1 && p.grid_rows < rows) return ARGR_EINVAL;
    return ARGR_OK;
}

}  // namespace argr
