// Launch-geometry planner: a pure function of the problem and the device's
// properties (no CUDA call), so it can be tested on a machine without a GPU.
//
// Geometry rules (onnxruntime #32092 Approach and Kernel profile; #31694
// Description), re-derived for a GB300:
//  * narrow rows (at most kNarrowRowBytes) use G lanes per row, with G the
//    smallest power of two that covers the row in one batch of U loads per
//    lane (G = 1 is one thread per row);
//  * when there are enough rows to fill the device with one warp each, rows of
//    medium width use one warp per row and wider rows one CTA per row;
//  * a few wide rows get one thread-block cluster each (up to 16 CTAs, at most
//    about two CTAs per SM in total), merged through distributed shared memory
//    with no global round trip (each warp pushes its candidate into CTA 0),
//    as long as a CTA's share stays small enough (kClusterMaxCtaBytes) for the
//    cluster's SMs to stream it quickly;
//  * otherwise (very wide rows) a row is split over several CTAs of the whole
//    device, about one wave in total (more CTAs than one wave was measured
//    slower on the pages' H200, and the merge cost grows with the CTA count),
//    while every CTA keeps at least kMinSplitShare of the row; rows too short
//    for that get one CTA (or, 16-32 KB rows of many elements, one warp).
// Every default plan launches as a programmatic dependent of the previous grid
// in the stream, which hides launch latency between back-to-back calls.
#include <algorithm>
#include <climits>

#include "internal.h"

namespace argr {

namespace {

constexpr int64_t kNarrowRowBytes = 1024;  // rows up to this width: G lanes per row
constexpr int64_t kWarpRowBytes = 32768;   // many rows up to this width: a warp (or half) per row
constexpr int kManyRowsBlock = 128;        // CTA size on the many-rows path
constexpr int kManyRowsUnroll = 8;         // 16-byte loads in flight per lane on the many-rows path
constexpr int kBlock = 256;                // threads per CTA on every path
constexpr int kNarrowVecBlock = 128;       // narrow rows with vector loads
constexpr int64_t kAxisWarpsPerSmNarrow = 32;  // non-last axis, narrow column segments: warps per SM
constexpr int kRowsUnroll = 4;             // loads in flight per lane on the rows path
constexpr int kSplitUnroll = 4;            // vector loads in flight per thread on the split path
constexpr int64_t kRowsWaves = 8;          // rows path: grid of at most this many waves (grid-stride beyond)
constexpr int64_t kMaxGridY = 65535;       // hardware limit of gridDim.y
constexpr int64_t kMaxBlocksPerRow = 65535;
constexpr int64_t kClusterMaxCtaBytes = 128 * 1024;  // largest share of a row per cluster CTA
constexpr int64_t kMaxDynamicSmem = 227 * 1024;        // dynamic shared memory one CTA may use
constexpr int64_t kPipeDeepWarpsPerSm = 16;  // resident warps of the 8-deep pipelined rows kernel (registers)
constexpr int64_t kMinSplitShare = 32768;    // a row is shared by several CTAs only in pieces of this size
// Inputs up to this size get ARGR_PLAN_PREFETCH: two calls' inputs then fit
// L2 together, so what one call prefetches while the previous one runs is
// still there when it reads it. Measured on GB300 (graphs of 16 calls, L2-cold
// inputs): [32,202048] bf16 5.22 -> 4.72 us, [8,202048] f32 4.14 -> 3.80 us,
// [1,202048] f32 3.31 -> 3.11 us, [4096,128] f32 2.08 -> 1.93 us; above it,
// [4096,4096] f32 (67 MB) 11.6 -> 14.2 us, so larger inputs on the rows path
// prefetch only the head of each CTA's rows (ARGR_PLAN_PREFETCH_HEAD).
constexpr int64_t kPrefetchMaxInput = 32 * 1024 * 1024;

int64_t ceil_div(int64_t a, int64_t b) { return a / b + (a % b != 0); }

int pow2_ceil(int64_t v) {
    int p = 1;
    while (p < v && p < 32) p <<= 1;
    return p;
}

bool valid_dtype(int d) { return d == ARGR_F32 || d == ARGR_F16 || d == ARGR_BF16 || d == ARGR_F64; }
bool valid_op(int o) { return o == ARGR_MAX || o == ARGR_MIN || o == ARGR_MAX_LAST || o == ARGR_MIN_LAST; }

int64_t ctas_per_wave(const argr_caps& caps, int block) {
    const int64_t per_sm = std::max<int64_t>(1, caps.max_threads_per_sm / block);
    return std::max<int64_t>(1, caps.sm_count) * per_sm;
}

}  // namespace

static bool caps_ok(const argr_caps& c) { return c.sm_count > 0 && c.max_threads_per_sm >= 32; }

int elem_size(int dtype) {
    switch (dtype) {
        case ARGR_F32: return 4;
        case ARGR_F16: return 2;
        case ARGR_BF16: return 2;
        case ARGR_F64: return 8;
        case ARGR_I32: return 4;
        case ARGR_I64: return 8;
        default: return 0;
    }
}

size_t plan_scratch(const argr_plan& p, int64_t rows) {
    if (p.path == ARGR_PATH_CUM || p.path == ARGR_PATH_CUM_SPLIT || p.path == ARGR_PATH_CUM_STREAM)
        return cum_plan_scratch(p, rows);
    if (p.path == ARGR_PATH_SPLIT && p.blocks_per_row > 1)
        return kPartialsOffset +
               static_cast<size_t>(p.grid_rows) * static_cast<size_t>(p.blocks_per_row) * kPartialBytes;
    return 0;
}


argr_status make_plan(int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps, bool base_aligned,
                      argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    *out = argr_plan{};
    if (!valid_dtype(dtype) || !valid_op(op) || rows < 0 || cols < 1 || cols > INT_MAX) return ARGR_EINVAL;
    if (!caps_ok(caps)) return ARGR_EINVAL;
    if (rows == 0) {
        out->path = ARGR_PATH_NONE;
        return ARGR_OK;
    }
    const int64_t es = elem_size(dtype);
    const int64_t E = 16 / es;
    const int64_t row_bytes = cols * es;
    const bool aligned = base_aligned && row_bytes % 16 == 0;  // every row starts 16-byte aligned

    out->block = kBlock;
    out->cluster = 0;
    out->flags = ARGR_PLAN_PDL;
    const bool big = rows > kPrefetchMaxInput / row_bytes;
    if (!big) out->flags |= ARGR_PLAN_PREFETCH;

    if (row_bytes <= kNarrowRowBytes) {
        // One batch of kRowsUnroll loads per lane covers the row.
        const int64_t units = aligned ? cols / E : cols;
        const int g = pow2_ceil(ceil_div(units, kRowsUnroll));
        out->path = ARGR_PATH_ROWS;
        out->group = g;
        out->vec = aligned ? 1 : 0;
        out->unroll = kRowsUnroll;
        // Vector rows that would give fewer 256-thread CTAs than SMs:
        // 128-thread CTAs, so that the rows spread over twice the SMs
        // ([4096,8] f32 1.61 -> 1.40 us, [16384,32] 2.07 -> 2.02, [1000,64]
        // 1.67 -> 1.63). With more rows 256 stays ([30000,100] f32 3.84
        // against 4.03 us with 128; [65536,64] and [131072,16] the same).
        out->block = (aligned && ceil_div(rows, kBlock / g) < caps.sm_count) ? kNarrowVecBlock : kBlock;
        const int64_t rows_per_cta = out->block / g;
        // With the prefetch, at most half the device's threads: the next
        // call's CTAs then find room while this one runs and fetch their rows
        // meanwhile ([65536,64] f32 4.67 -> 3.97 us with 608 CTAs of 256
        // instead of 1024); without it, up to kRowsWaves waves.
        const int64_t wave_ctas = ctas_per_wave(caps, out->block);
        const int64_t max_grid = (out->flags & ARGR_PLAN_PREFETCH) ? std::max<int64_t>(1, wave_ctas / 2)
                                                                    : kRowsWaves * wave_ctas;
        out->grid_rows = std::min(ceil_div(rows, rows_per_cta), max_grid);
        out->blocks_per_row = 1;
        out->scratch_bytes = 0;
        return ARGR_OK;
    }

    const int64_t wave = ctas_per_wave(caps, kBlock);
    if (rows >= wave || rows > kMaxSplitRows) {
        // Enough rows: no row is split.
        if (row_bytes <= kWarpRowBytes) {
            // Measured on GB300: 128-thread CTAs with 8 loads in flight per
            // lane, a whole warp for rows of 16 KB and more (4 KB for
            // 2- and 4-byte elements: [65536,1024] f32 38.4 -> 37.9 us,
            // [8192,4096] f16 13.2 -> 12.2 us), half a warp below.
            const int g = (row_bytes >= 16384 || (es <= 4 && row_bytes >= 4096)) ? 32 : 16;
            out->path = ARGR_PATH_ROWS;
            out->group = g;
            // 256-thread CTAs for 32 KB binary64 rows ([4096,4096] f64 30.4 ->
            // 27.6 us) and 16-bit rows of 16 KB and more ([4096,8192] bf16
            // 13.7 -> 13.0 us).
            const bool wide_ctas = (es == 8 && row_bytes >= kWarpRowBytes) || (es == 2 && row_bytes >= 16384);
            out->block = wide_ctas ? 2 * kManyRowsBlock : kManyRowsBlock;
            out->vec = aligned ? 1 : 0;
            out->unroll = kManyRowsUnroll;
            // Long rows (16 KB of binary32, 32 KB of binary64): software-
            // pipelined loads, 8 deep while the rows fit the warps that kernel
            // keeps resident, else 4 deep ([4096,4096] f32 11.9 -> 11.5 us,
            // f64 24.3 -> 23.9 us; [2048,8192] f32 13.2 -> 12.7 us).
            const bool pipe_rows = (es == 4 && row_bytes >= 16384) || (es == 8 && row_bytes >= kWarpRowBytes);
            if (aligned && pipe_rows) {
                out->flags |= ARGR_PLAN_PIPELINE;
                out->unroll = rows <= kPipeDeepWarpsPerSm * caps.sm_count ? 8 : 4;
            }
            out->grid_rows = std::min(ceil_div(rows, out->block / g), kRowsWaves * ctas_per_wave(caps, out->block));
            out->blocks_per_row = 1;
            // Inputs above 32 MiB: only the head of each CTA's rows (16 KiB)
            // before the dependency wait ([4096,4096] f64 23.4 -> 22.0 us, f32
            // 11.6 -> 11.3 us, [65536,1024] f32 38.1 -> 37.5 us; the full 128 KiB
            // evicts lines the previous call still reads: f32 11.6 -> 14.2 us).
            if (big) out->flags |= ARGR_PLAN_PREFETCH | ARGR_PLAN_PREFETCH_HEAD;
        } else {
            // One CTA per row: small CTAs with 8 loads in flight per thread,
            // more rows in flight per SM ([1024,16384] f32 14.1 -> 12.6 us).
            out->path = ARGR_PATH_SPLIT;
            out->block = kManyRowsBlock;
            out->unroll = kManyRowsUnroll;
            out->blocks_per_row = 1;
            out->grid_rows = std::min(rows, kMaxGridY);
        }
        out->scratch_bytes = plan_scratch(*out, rows);
        return ARGR_OK;
    }

    // Few rows: one cluster per row while a CTA's share stays small.
    if (caps.max_cluster >= 2 && rows <= caps.sm_count) {
        int c = 16;
        while (c > 2 && (c > caps.max_cluster || rows * c > 2 * static_cast<int64_t>(caps.sm_count))) c /= 2;
        const int64_t per_cta = row_bytes / c;
        if (c <= caps.max_cluster && rows * c <= 2 * static_cast<int64_t>(caps.sm_count) &&
            per_cta <= kClusterMaxCtaBytes) {
            // 512 threads from 16 KB per CTA (with the push merge a single row
            // too: [1,202048] f32 2.78 us with 1024 threads and 4 loads each,
            // 2.65 us with 512 threads and 8), 256 from 4 KB, else 128.
            const int block = per_cta >= 16384 ? 512 : per_cta >= 4096 ? 256 : 128;
            int unroll = 1;
            while (unroll < 8 && static_cast<int64_t>(unroll) * block * 16 < per_cta) unroll <<= 1;
            out->path = ARGR_PATH_CLUSTER;
            out->cluster = c;
            out->block = block;
            out->unroll = unroll;
            out->blocks_per_row = c;
            out->grid_rows = std::min(rows, kMaxGridY);
            out->scratch_bytes = 0;
            return ARGR_OK;
        }
    }

    // Very wide rows: split each row over CTAs, about one wave in total, each
    // CTA with at least kMinSplitShare of the row: below that the merge of
    // the partials costs more than the extra CTAs gain ([256,8192] f32 over
    // 4 CTAs 6.6 us, one CTA per row 4.0 us).
    const int64_t by_wave = std::max<int64_t>(1, wave / rows);
    const int64_t by_work = std::max<int64_t>(1, row_bytes / kMinSplitShare);
    const int64_t bpr = std::min({by_wave, by_work, kMaxBlocksPerRow});
    out->path = ARGR_PATH_SPLIT;
    out->unroll = kSplitUnroll;
    out->blocks_per_row = bpr;
    out->grid_rows = rows;  // rows < one wave <= kMaxGridY here
    if (bpr == 1) {
        const int64_t sms = caps.sm_count;
        if (aligned && rows > 4 * sms && cols <= 4096 && es >= 4 && row_bytes >= 16384) {
            // Rows of 16-32 KB with at most 4096 elements: a warp per row with
            // 8-deep pipelined loads ([1024,4096] f64 10.0 -> 8.9 us,
            // [1200,4096] f32 5.5 -> 5.2 us).
            out->path = ARGR_PATH_ROWS;
            out->group = 32;
            out->vec = 1;
            out->block = kManyRowsBlock;
            out->unroll = 8;
            out->flags |= ARGR_PLAN_PIPELINE;
            out->grid_rows = ceil_div(rows, kManyRowsBlock / 32);
            out->blocks_per_row = 1;
            out->scratch_bytes = 0;
            return ARGR_OK;
        }
        // One CTA per row with 8 loads in flight per thread: 256 threads while
        // there are few rows per SM ([512,8192] f32 5.8 -> 5.4 us), else 128
        // as on the many-rows path.
        out->block = rows <= 4 * sms ? kBlock : kManyRowsBlock;
        out->unroll = kManyRowsUnroll;
        out->grid_rows = std::min(rows, kMaxGridY);
    }
    out->scratch_bytes = plan_scratch(*out, rows);
    (void)E;
    return ARGR_OK;
}

// ---------------------------------------------------------------------------
// Non-last axis. A warp is CG column lanes (V inner positions each) by 32/CG
// lanes along R; Y warps of a CTA split R; when the grid still has too few
// warps, a cluster of C CTAs also splits R (AcceleratedKernels.jl #138:
// threads along the reduction and a split with a combine step when the
// outputs do not fill the device; the combine here is distributed shared
// memory). The rules below reproduce the best of a sweep of CG, Y and C on
// GB300 for tall, wide, batched, narrow-inner and binary64 shapes.
// ---------------------------------------------------------------------------
static int axis_vec(int dtype) { return elem_size(dtype) == 8 ? 2 : 4; }

static bool axis_vec_ok(int dtype, int64_t inner, uintptr_t x_addr) {
    const int v = axis_vec(dtype);
    const int vb = v * elem_size(dtype);  // 16 bytes, or 8 for 16-bit elements
    return inner % v == 0 && x_addr % vb == 0;
}

argr_status make_axis_plan(int64_t outer, int64_t reduce, int64_t inner, int dtype, int op, const argr_caps& caps,
                           bool base_aligned, argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    *out = argr_plan{};
    if (inner < 1 || outer < 0 || !valid_dtype(dtype) || !valid_op(op) || reduce < 1 || reduce > INT_MAX)
        return ARGR_EINVAL;
    if (inner == 1) return make_plan(outer, reduce, dtype, op, caps, base_aligned, out);
    if (!caps_ok(caps)) return ARGR_EINVAL;
    if (outer == 0) {
        out->path = ARGR_PATH_NONE;
        return ARGR_OK;
    }
    const bool vec = base_aligned && inner % axis_vec(dtype) == 0;
    const int64_t v = vec ? axis_vec(dtype) : 1;
    const int64_t es = elem_size(dtype);
    const int64_t sms = caps.sm_count;
    // Column lanes: from a full warp of columns (or as many as the columns
    // need) down to 32-byte segments per step along R, halving while the
    // grid would have fewer than 4 CTAs per SM; the other lanes go along R.
    int64_t cg = 32;
    while (cg > 1 && (cg / 2) * v >= inner) cg >>= 1;
    const int64_t cg_min = std::max<int64_t>(1, 32 / (v * es));
    while (cg > cg_min && std::min(outer, kMaxGridY) * ceil_div(inner, cg * v) < 4 * sms) cg >>= 1;
    const int64_t tiles = ceil_div(inner, cg * v);
    if (tiles > kMaxGridY) return ARGR_EUNSUPPORTED;
    const int64_t slots = std::min(outer, kMaxGridY);
    const int64_t rg = 32 / cg;
    const int64_t ctas = slots * tiles;
    // Warps along R: enough for ~16 warps per SM over the grid, each R lane
    // keeping at least 16 steps. Column segments narrower than a 128-byte
    // line on a grid of at least a CTA per SM wait on their loads: there ~32
    // ([64,512,256] bf16 8.35 -> 8.02 us, [16,2048,384] f64 27.8 -> 25.9 us;
    // 512-byte segments were slower with 32, [1,1000,100000] f32 65.8 -> 77.0,
    // and so was a grid below one CTA per SM, [1,100000,1000] f32 71.0 -> 72.5).
    const bool narrow_segments = cg * v * es < 128 && ctas >= sms;
    int64_t y = ceil_div((narrow_segments ? kAxisWarpsPerSmNarrow : 16) * sms, ctas);
    y = std::max<int64_t>(1, std::min<int64_t>({y, 32, reduce / (rg * 16)}));
    int64_t c = 1;
    if (ctas * y < 4 * sms && outer <= kMaxGridY && caps.max_cluster >= 2) {
        // Still too few warps: a cluster of CTAs splits R further.
        c = std::min<int64_t>(std::min<int64_t>(16, caps.max_cluster), ceil_div(16 * sms, ctas * y));
        while (c > 1 && reduce / (c * y * rg) < 16) --c;
    }
    out->path = ARGR_PATH_AXIS;
    out->block = static_cast<int32_t>(32 * y);
    out->group = static_cast<int32_t>(cg);
    out->vec = vec ? 1 : 0;
    out->unroll = 8;
    out->cluster = static_cast<int32_t>(c);
    out->blocks_per_row = c;
    out->grid_rows = c > 1 ? outer : slots;
    out->flags = ARGR_PLAN_PDL;
    out->scratch_bytes = 0;
    return ARGR_OK;
}

argr_status check_axis_plan(const argr_plan& p, int64_t outer, int64_t reduce, int64_t inner, int dtype,
                            const argr_caps& caps, uintptr_t x_addr) {
    if (!valid_dtype(dtype) || outer < 0 || inner < 1 || reduce < 1 || reduce > INT_MAX) return ARGR_EINVAL;
    if (outer == 0) return ARGR_OK;
    if (p.path != ARGR_PATH_AXIS) return ARGR_EINVAL;
    if (p.block < 32 || p.block > 1024 || p.block % 32 != 0) return ARGR_EINVAL;
    if (p.flags & ~ARGR_PLAN_PDL) return ARGR_EINVAL;
    if (p.unroll != 4 && p.unroll != 8) return ARGR_EINVAL;
    if (p.vec != 0 && p.vec != 1) return ARGR_EINVAL;
    if (p.vec && !axis_vec_ok(dtype, inner, x_addr)) return ARGR_EINVAL;
    const int g = p.group;
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32) return ARGR_EINVAL;
    const int64_t v = p.vec ? axis_vec(dtype) : 1;
    if (ceil_div(inner, g * v) > kMaxGridY) return ARGR_EUNSUPPORTED;
    if (p.cluster < 1 || p.cluster > 16 || p.blocks_per_row != p.cluster) return ARGR_EINVAL;
    if (p.cluster > 1 && caps.max_cluster < p.cluster) return ARGR_EUNSUPPORTED;
    if (p.grid_rows < 1 || p.grid_rows > kMaxGridY) return ARGR_EINVAL;
    if (p.cluster > 1 && p.grid_rows < outer) return ARGR_EINVAL;  // cluster slots are not reused across outer
    const int64_t smem = (p.block / 32 + (p.cluster > 1 ? p.cluster : 0)) * g * v * 16;
    if (smem > kMaxDynamicSmem) return ARGR_EINVAL;
    return ARGR_OK;
}

argr_status check_plan(const argr_plan& p, int64_t rows, int64_t cols, int dtype, const argr_caps& caps,
                       bool row_aligned) {
    if (!valid_dtype(dtype) || rows < 0 || cols < 1 || cols > INT_MAX) return ARGR_EINVAL;
    if (rows == 0) return ARGR_OK;
    if (p.block < 32 || p.block > 1024 || p.block % 32 != 0) return ARGR_EINVAL;
    if (p.flags & ~(ARGR_PLAN_PDL | ARGR_PLAN_BULK | ARGR_PLAN_TEST_EXPIRE | ARGR_PLAN_PIPELINE | ARGR_PLAN_PREFETCH |
                    ARGR_PLAN_PREFETCH_HEAD))
        return ARGR_EINVAL;
    if ((p.flags & ARGR_PLAN_PREFETCH_HEAD) && (p.path != ARGR_PATH_ROWS || !(p.flags & ARGR_PLAN_PREFETCH)))
        return ARGR_EINVAL;
    if ((p.flags & ARGR_PLAN_BULK) && p.path != ARGR_PATH_CLUSTER) return ARGR_EINVAL;
    if ((p.flags & ARGR_PLAN_PREFETCH) &&
        ((p.path != ARGR_PATH_ROWS && p.path != ARGR_PATH_SPLIT && p.path != ARGR_PATH_CLUSTER &&
          p.path != ARGR_PATH_STREAM) ||
         (p.flags & ARGR_PLAN_BULK)))
        return ARGR_EINVAL;
    if ((p.flags & ARGR_PLAN_PIPELINE) &&
        (p.path != ARGR_PATH_ROWS || p.vec != 1 || p.group < 16 || p.block > kPipeMaxBlock))
        return ARGR_EINVAL;
    // the test hook exists on the waits of the streaming kernel and of the
    // push merge (cluster plans with a row slot per row, no bulk copies)
    if ((p.flags & ARGR_PLAN_TEST_EXPIRE) && p.path != ARGR_PATH_STREAM &&
        (p.path != ARGR_PATH_CLUSTER || (p.flags & ARGR_PLAN_BULK) || p.grid_rows != rows || p.block > 512))
        return ARGR_EINVAL;
    switch (p.path) {
        case ARGR_PATH_ROWS: {
            const int g = p.group;
            if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32) return ARGR_EINVAL;
            if (p.unroll != 4 && p.unroll != 8) return ARGR_EINVAL;
            if (p.vec && !row_aligned) return ARGR_EINVAL;
            if (p.vec != 0 && p.vec != 1) return ARGR_EINVAL;
            if (p.grid_rows < 1 || p.grid_rows > INT_MAX) return ARGR_EINVAL;
            return ARGR_OK;
        }
        case ARGR_PATH_SPLIT: {
            if (p.unroll != 1 && p.unroll != 2 && p.unroll != 4 && p.unroll != 8) return ARGR_EINVAL;
            if (p.blocks_per_row < 1 || p.blocks_per_row > kMaxBlocksPerRow) return ARGR_EINVAL;
            if (p.grid_rows < 1 || p.grid_rows > kMaxGridY) return ARGR_EINVAL;
            // A split row owns its partial slots and counter: no row loop, and
            // at most kMaxSplitRows counters exist.
            if (p.blocks_per_row > 1 && (p.grid_rows < rows || p.grid_rows > kMaxSplitRows)) return ARGR_EINVAL;
            // The partials stay below the split scan's large record region.
            if (p.blocks_per_row > 1 && p.grid_rows * p.blocks_per_row > kMaxPartials) return ARGR_EINVAL;
            return ARGR_OK;
        }
        case ARGR_PATH_STREAM: {
            const int g = p.group;
            if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32) return ARGR_EINVAL;
            if (!row_aligned) return ARGR_EINVAL;  // bulk copies need 16-byte aligned rows
            if (p.stages < 1 || p.stages > 4) return ARGR_EINVAL;
            if (p.stage_bytes < 1024 || p.stage_bytes > 65536 || p.stage_bytes % 16 != 0) return ARGR_EINVAL;
            if (p.block > 1024) return ARGR_EINVAL;
            if (static_cast<int64_t>(p.block / 32) * p.stages * p.stage_bytes > kMaxDynamicSmem) return ARGR_EINVAL;
            const int64_t row_bytes = cols * elem_size(dtype);
            if (row_bytes > p.stage_bytes && g != 32) return ARGR_EINVAL;  // pieces of a row need the whole warp
            if (p.grid_rows < 1 || p.grid_rows > INT_MAX) return ARGR_EINVAL;
            return ARGR_OK;
        }
        case ARGR_PATH_CLUSTER: {
            if (p.unroll != 1 && p.unroll != 2 && p.unroll != 4 && p.unroll != 8) return ARGR_EINVAL;
            if (p.cluster < 2 || p.cluster > 16 || p.blocks_per_row != p.cluster) return ARGR_EINVAL;
            if (p.grid_rows < 1 || p.grid_rows > kMaxGridY) return ARGR_EINVAL;
            if (caps.max_cluster < p.cluster) return ARGR_EUNSUPPORTED;
            if (p.flags & ARGR_PLAN_BULK) {
                // one CTA's share of the aligned body must fit the bulk buffer
                const int64_t nvec = cols * elem_size(dtype) / 16;
                if ((nvec + p.cluster - 1) / p.cluster * 16 > kClusterMaxCtaBytes) return ARGR_EINVAL;
            }
            return ARGR_OK;
        }
        default: return ARGR_EINVAL;
    }
}

}  // namespace argr
