/*
 * argreduce.h - row-wise ArgMax / ArgMin over the last axis on a GB300 GPU.
 *
 * C ABI of libargreduce.so. Every argument is a plain pointer or integer; no
 * C++ or framework type crosses this boundary. Device pointers are CUDA
 * device addresses in the caller's current context. The library never
 * allocates, frees or synchronises memory inside argreduce(); all work is
 * queued on the caller's stream.
 *
 * The operation is defined by two onnxruntime pull requests:
 *   - "[CUDA] Parallelize ArgMax/ArgMin over wide last axes" (#32092),
 *     sections Approach and Semantics: a [rows, cols] row-major tensor is
 *     reduced over its last axis to one int64 index per row; ties resolve to
 *     the lowest index; a leading NaN yields index 0; rows that are entirely
 *     -inf, +inf or NaN yield index 0; the result equals the sequential
 *     one-thread-per-row scan bit for bit for every input.
 *   - "[CUDA] Parallelize ArgMax/ArgMin over the reduction axis" (#31694),
 *     section Semantics: the sequential scan seeds with element 0 and a later
 *     element replaces the candidate only when strictly better.
 *
 * "Strictly better" is an IEEE comparison: greater (ArgMax) or less (ArgMin),
 * false when either operand is NaN. So a NaN after element 0 never wins, +0.0
 * and -0.0 tie (lowest index wins), and subnormals are compared exactly
 * (no flush to zero). binary16 and bfloat16 values are compared after an
 * exact widening to binary32.
 */
#ifndef ARGREDUCE_H
#define ARGREDUCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t. NULL is the legacy default stream. */
typedef struct CUstream_st* argr_stream;

/* Element type of x (and of out_val). argreduce() and argreduce_axis() take
 * the floating types; the integer types are for argreduce_cum(). */
typedef enum {
    ARGR_F32 = 0,  /* IEEE binary32 */
    ARGR_F16 = 1,  /* IEEE binary16 */
    ARGR_BF16 = 2, /* bfloat16 (upper half of binary32) */
    ARGR_F64 = 3,  /* IEEE binary64 */
    ARGR_I32 = 4,  /* int32: argreduce_cum() only */
    ARGR_I64 = 5   /* int64: argreduce_cum() only */
} argr_dtype;

/* ArgMax / ArgMin; ties resolve to the first index, or to the last index for
 * the *_LAST ops (ONNX select_last_index = 1: the same scan with a non-strict
 * comparison, still false on NaN, so NaN handling is unchanged). */
typedef enum { ARGR_MAX = 0, ARGR_MIN = 1, ARGR_MAX_LAST = 2, ARGR_MIN_LAST = 3 } argr_op;

typedef enum {
    ARGR_OK = 0,
    ARGR_EINVAL = 1,      /* bad pointer, size, enum or plan; nothing was launched */
    ARGR_ESCRATCH = 2,    /* scratch missing, too small or not 16-byte aligned; nothing launched */
    ARGR_EUNSUPPORTED = 3,/* valid request this build or device cannot run; nothing launched */
    ARGR_ECUDA = 4,       /* a CUDA runtime call failed (launch or device query) */
    ARGR_ETIMEOUT = 5     /* a bounded device-side wait expired (reported by argreduce_read_error) */
} argr_status;

/* Kernel paths the planner chooses between (#32092 Approach: thread per row
 * for narrow rows; a row spread over warps and blocks otherwise). */
typedef enum {
    ARGR_PATH_NONE = 0,    /* rows == 0: nothing to launch */
    ARGR_PATH_ROWS = 1,    /* `group` lanes per row (1 = thread per row, 32 = warp per row) */
    ARGR_PATH_SPLIT = 2,   /* `blocks_per_row` CTAs per row; >1 merges through scratch,
                              the last CTA to arrive for a row reduces the partials */
    ARGR_PATH_CLUSTER = 3, /* one thread-block cluster of `cluster` CTAs per row, merged
                              through distributed shared memory; no scratch. With a row
                              slot per row (grid_rows == rows) and at most 512 threads
                              per CTA every warp pushes its
                              candidate into CTA 0 (st.async on an mbarrier, a bounded
                              wait in CTA 0); with fewer slots CTAs loop over rows and
                              merge through a cluster barrier */
    ARGR_PATH_AXIS = 5,    /* non-last axis (argreduce_axis): a warp is `group` column lanes (each
                              V consecutive inner positions, `vec`: V-element vectors) by 32/group
                              lanes along R; the CTA's block/32 warps split R, and a cluster of
                              `cluster` CTAs (1 = none) splits it further. unroll 4 or 8 */
    ARGR_PATH_CUM = 6,     /* cummax / cummin (argreduce_cum): a row in `cluster` chunks, one CTA
                              each (1 = none), scanned in tiles of block * 7 elements */
    ARGR_PATH_CUM_SPLIT = 7, /* cummax / cummin: a row in `blocks_per_row` chunks, one CTA each,
                              any number of CTAs; chunk aggregates are exchanged through
                              scratch (rows * blocks_per_row <= 65536; above 1024 record
                              words the records need a scratch buffer of more than 1 MiB) */
    ARGR_PATH_CUM_STREAM = 8, /* cummax / cummin: tiles of block * 7 elements (`blocks_per_row` =
                              tiles per row) taken in ticket order by `grid_rows` CTAs, each
                              tile read once; carries by decoupled look-back through scratch
                              (rows * blocks_per_row <= 32768). Not chosen by the planner */
    ARGR_PATH_STREAM = 4   /* every warp streams a contiguous range of rows through its own
                              `stages` shared-memory buffers of `stage_bytes`, filled by bulk
                              (TMA) copies; `group` lanes per row for rows that fit a buffer,
                              the whole warp otherwise. Needs 16-byte aligned rows. */
} argr_path;

/* Device properties the planner uses. */
typedef struct {
    int32_t sm_count;           /* streaming multiprocessors */
    int32_t max_threads_per_sm; /* resident threads per SM */
    int32_t max_cluster;        /* largest cluster size this device launches (1 = none) */
    int32_t cc_major, cc_minor; /* compute capability */
} argr_caps;

/* Plan flag: launch as a programmatic dependent of the previous grid in the
 * stream. The kernel still waits for that grid to complete before it touches
 * memory, so results are the same; only the launch latency overlaps. */
#define ARGR_PLAN_PDL 1
/* Plan flag (CLUSTER path): each CTA's share of the row is fetched into shared
 * memory by bulk (TMA) copies issued all at once, instead of by loads from
 * every thread. The share must be at most 128 KiB. */
#define ARGR_PLAN_BULK 2
/* Plan flag for tests of failure handling (STREAM, CLUSTER with a row slot
 * per row, CUM_SPLIT and CUM_STREAM paths only). STREAM: one bulk copy's
 * barrier is made to expect more bytes than arrive, so the kernel's bounded
 * wait (2 ms under this flag) expires; the kernel records the expiry, skips
 * its work and returns. CLUSTER (push merge only: grid_rows == rows, at
 * most 512 threads): CTA 0's barrier expects 16 bytes more than
 * the cluster's candidates, so its wait expires and it returns without
 * writing the row. CUM_SPLIT and
 * CUM_STREAM: the first chunk (tile) of each row never publishes its record,
 * so every wait for it expires after 2 ms. Either way argreduce_read_error()
 * then reports ARGR_ETIMEOUT and outputs are undefined. Never set in the
 * planner's plans. */
#define ARGR_PLAN_TEST_EXPIRE 4
/* Plan flag (CUM_SPLIT path): each CTA copies its whole chunk (at most 80 KiB)
 * into shared memory with bulk (TMA) copies and scans it there, so the input
 * is read from memory once; without it, phase B reads the chunk again (from
 * L2 while the chunks in flight fit it). Measured slower on GB300 at every
 * size (two CTAs per SM alternate loading and scanning), so the planner does
 * not set it. */
#define ARGR_PLAN_STASH 8
/* Plan flag (CUM_SPLIT path, not with ARGR_PLAN_STASH): decoupled look-back.
 * Every chunk also publishes its inclusive prefix once known, and a CTA reads
 * back only to the nearest one, so chunks can be one tile each (read once,
 * from registers) at any chunk count; two record words per chunk. */
#define ARGR_PLAN_LOOKBACK 16
/* Plan flag (ROWS path with vec = 1 and group 16 or 32): software-pipelined
 * loads. Every lane issues the next batch of `unroll` 16-byte loads before it
 * compares the current batch, so its loads stay in flight while it compares;
 * twice the registers for loaded data, so at most 256 threads per CTA. */
#define ARGR_PLAN_PIPELINE 32
/* Plan flag (ROWS, SPLIT, CLUSTER and STREAM paths): before its dependency
 * wait, each CTA asks the L2 cache to fetch the part of x it reads first (bulk L2
 * prefetches of 16-byte aligned pieces). A prefetch changes no value (L2 is
 * where the GPU keeps memory coherent, so a line written by the previous
 * grid is read as written), so results are the same; when the CTA starts
 * while the previous grid in the stream is still running (ARGR_PLAN_PDL),
 * the read of x from HBM overlaps that grid instead of following it. */
#define ARGR_PLAN_PREFETCH 64
/* Plan flag (ROWS path, with ARGR_PLAN_PREFETCH): each CTA prefetches at most
 * 16 KiB (the head of its rows) instead of 128 KiB. For inputs above 32 MiB,
 * where two calls' inputs no longer share L2: only the first bytes each CTA
 * reads come early, covering the gap between the previous grid's last loads
 * and this grid's first, without evicting what the previous grid still needs. */
#define ARGR_PLAN_PREFETCH_HEAD 128

/* A launch plan. Produced by argreduce_plan(); tests may edit it to force a
 * path and pass it to argreduce_with_plan(), which re-validates it. */
typedef struct {
    int32_t path;           /* argr_path */
    int32_t block;          /* threads per CTA: multiple of 32, 32..1024 */
    int32_t group;          /* ROWS / STREAM: lanes per row; AXIS: column lanes per warp; power of two 1..32 */
    int32_t vec;            /* 1: 16-byte vector loads (ROWS needs every row 16-byte aligned) */
    int32_t unroll;         /* loads in flight per thread per step: ROWS 4 or 8; SPLIT/CLUSTER 1,2,4,8 */
    int32_t cluster;        /* CLUSTER: CTAs per cluster, 2..16 */
    int32_t flags;          /* ARGR_PLAN_* bits */
    int32_t stages;         /* STREAM: buffers per warp, 1..4 */
    int32_t stage_bytes;    /* STREAM: bytes per buffer, multiple of 16, 1 KiB..64 KiB */
    int32_t reserved;       /* 0 */
    int64_t blocks_per_row; /* SPLIT / CLUSTER / CUM: CTAs that share one row; CUM_SPLIT: chunks
                               per row; CUM_STREAM: tiles per row */
    int64_t grid_rows;      /* SPLIT / CLUSTER / CUM: row slots in the grid (rows loop over them;
                               CUM_SPLIT: the rows); ROWS / STREAM / CUM_STREAM: number of CTAs */
    uint64_t scratch_bytes; /* bytes of scratch this plan needs (0 = none) */
} argr_plan;

/*
 * Scratch bytes argreduce() needs for this problem on the current device
 * (0 when the chosen path needs none). The bound is small: a multi-CTA row
 * needs one 16-byte partial per CTA plus a 4-byte counter per row, and such
 * plans are only chosen while the whole grid fits one wave of the device
 * (#32092 Approach: scratch bounded by the device's thread capacity).
 * Returns 0 also when the device cannot be queried; argreduce() then reports
 * the error.
 */
size_t argreduce_scratch_bytes(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op);

/*
 * Prepare a scratch buffer once after allocating it: zeroes the per-row
 * arrival counters and the error word (an asynchronous memset on `stream`).
 * After that the counters reset themselves at the end of every call, so no
 * per-call memset is needed and argreduce() can be captured in a CUDA graph
 * and replayed. The partial-result region may hold any bytes between calls.
 * `scratch` must be a device pointer, 16-byte aligned.
 */
argr_status argreduce_scratch_init(void* scratch, size_t scratch_bytes, argr_stream stream);

/*
 * Row-wise ArgMax (op = ARGR_MAX) or ArgMin (ARGR_MIN) of x[rows, cols]
 * (onnxruntime #32092, Approach: one int64 index per row of the last axis,
 * chosen by a planner among thread-per-row, block-per-row and multi-block
 * kernels; Semantics: the sequential first-occurrence scan, bit for bit).
 *
 *   x         device pointer to rows*cols elements of `dtype`, row-major and
 *             contiguous (row r starts at element r*cols). Any address that is
 *             a multiple of the element size; unaligned row starts are handled.
 *   rows      >= 0. rows == 0 returns ARGR_OK and launches nothing.
 *   cols      1 .. INT32_MAX (the index is computed in 32 bits within a row).
 *   out_idx   device pointer to rows int64 values (written).
 *   out_val   NULL, or a device pointer to rows elements of `dtype`, aligned to
 *             the element size; receives the raw bits of x[r, out_idx[r]]
 *             (NaN payloads and the sign of zero preserved).
 *   scratch   device pointer prepared by argreduce_scratch_init(), 16-byte
 *             aligned, at least argreduce_scratch_bytes() bytes; may be NULL
 *             when that is 0. Owned by the caller. Two calls that may run at
 *             the same time on the GPU must not share a scratch buffer.
 *   stream    CUDA stream the kernel is queued on.
 *
 * All validation happens before any launch: on an error status nothing was
 * queued. The call does not synchronise; kernel faults surface on the stream.
 * No per-call allocation, memset or host synchronisation, so the call can be
 * captured into a CUDA graph (as long as the same scratch stays alive).
 */
argr_status argreduce(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op,
                      int64_t* out_idx, void* out_val, void* scratch, size_t scratch_bytes,
                      argr_stream stream);

/*
 * Query the planner. caps == NULL uses the current device (one query per
 * device, cached); a non-NULL caps plans for those properties instead, which
 * lets tests force geometries of other device sizes (#32092 Testing: fuzz
 * repeated with several simulated device capacities). Pure host code when
 * caps is given: needs no GPU.
 */
argr_status argreduce_plan(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op,
                           const argr_caps* caps, argr_plan* out);

/*
 * argreduce() with an explicit plan (tests and benchmarks force each path
 * with it). The plan is checked against the problem and the device: an
 * impossible plan returns ARGR_EINVAL (or ARGR_EUNSUPPORTED for a cluster the
 * device cannot launch) before anything is queued. Scratch must be at least
 * plan->scratch_bytes as recomputed for the problem.
 */
argr_status argreduce_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t rows,
                                int64_t cols, argr_op op, int64_t* out_idx, void* out_val, void* scratch,
                                size_t scratch_bytes, argr_stream stream);

/*
 * The checks argreduce_with_plan() applies to a plan, against the given device
 * properties instead of the current device's: path, CTA size, lanes per row,
 * loads in flight, flags (each only on the paths it applies to), grid limits
 * and the cluster size (ARGR_EUNSUPPORTED above caps->max_cluster). Covers the
 * last-axis paths (NONE, ROWS, SPLIT, CLUSTER, STREAM). rows_aligned != 0 says
 * every row of the input starts on a 16-byte boundary (vector loads allowed).
 * Returns ARGR_OK, ARGR_EINVAL or ARGR_EUNSUPPORTED as argreduce_with_plan()
 * would; pure host code (#32092 Testing: every dispatch path, simulated device
 * capacities), so forced plans can be checked without a GPU.
 */
argr_status argreduce_plan_check(const argr_plan* plan, int64_t rows, int64_t cols, argr_dtype dtype,
                                 const argr_caps* caps, int rows_aligned);

/*
 * ArgMax / ArgMin over a non-last axis: x is row-major [outer, reduce, inner]
 * and the result is out_idx[outer, inner] (int64, the position along the
 * reduced axis), out_val[outer, inner] optional. Element (o, r, i) is at
 * x[(o * reduce + r) * inner + i]; each output applies exactly the rules of
 * argreduce() to the `reduce` elements x[o, 0..reduce-1, i], which lie
 * `inner` elements apart. With inner == 1 this is argreduce() on
 * [outer, reduce]. Needs no scratch unless inner == 1 and the last-axis plan
 * does (pass scratch as for argreduce(); argreduce_scratch_bytes(outer,
 * reduce, ...) sizes it). Errors as for argreduce(); ARGR_EUNSUPPORTED if
 * inner needs more than 65535 column tiles of 32 lanes.
 */
argr_status argreduce_axis(const void* x, argr_dtype dtype, int64_t outer, int64_t reduce, int64_t inner,
                           argr_op op, int64_t* out_idx, void* out_val, void* scratch, size_t scratch_bytes,
                           argr_stream stream);

/* The planner for argreduce_axis() (a last-axis plan when inner == 1). */
argr_status argreduce_axis_plan(int64_t outer, int64_t reduce, int64_t inner, argr_dtype dtype, argr_op op,
                                const argr_caps* caps, argr_plan* out);

/* argreduce_axis() with an explicit plan (re-validated; an ARGR_PATH_AXIS
 * plan for any inner, a last-axis plan only for inner == 1). */
argr_status argreduce_axis_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t outer,
                                     int64_t reduce, int64_t inner, argr_op op, int64_t* out_idx, void* out_val,
                                     void* scratch, size_t scratch_bytes, argr_stream stream);

/*
 * cummax / cummin with indices along the last axis of x[rows, cols]
 * (op = ARGR_MAX or ARGR_MIN; the *_LAST ops return ARGR_EUNSUPPORTED).
 * For every position j of every row: out_idx[r * cols + j] is the row's
 * ArgMax (ArgMin) over x[r, 0..j] by the rules of argreduce() (ties keep the
 * earlier index; a NaN after x[r, 0] is never chosen; a leading NaN gives 0
 * everywhere), and out_val[r * cols + j] (optional) the raw bits of that
 * element. So out_idx[r * cols + cols - 1] equals argreduce()'s result.
 * Element types: the four floating types and ARGR_I32 / ARGR_I64 (compared
 * as integers). Paddle issue #79670 ("Possible fixes": a scan with argmax
 * semantics where ties take the earlier index, and a two-pass tiled scan when
 * the rows alone do not fill the GPU). out_idx holds rows * cols int64.
 * Scratch: argreduce_cum_scratch_bytes() bytes (0 when the plan needs none;
 * then scratch may be NULL), prepared once by argreduce_scratch_init(); the
 * same buffer may serve argreduce() calls that do not run at the same time.
 * Errors as for argreduce().
 */
argr_status argreduce_cum(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op, int64_t* out_idx,
                          void* out_val, void* scratch, size_t scratch_bytes, argr_stream stream);

/* Scratch bytes argreduce_cum() needs for this problem on the current device
 * (0 = none). */
size_t argreduce_cum_scratch_bytes(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op);

/* The planner for argreduce_cum(). */
argr_status argreduce_cum_plan(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op, const argr_caps* caps,
                               argr_plan* out);

/* argreduce_cum() with an explicit ARGR_PATH_CUM, ARGR_PATH_CUM_SPLIT or
 * ARGR_PATH_CUM_STREAM plan (re-validated). */
argr_status argreduce_cum_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t rows,
                                    int64_t cols, argr_op op, int64_t* out_idx, void* out_val, void* scratch,
                                    size_t scratch_bytes, argr_stream stream);

/* Scratch bytes a given plan needs for `rows` rows. */
size_t argreduce_plan_scratch_bytes(const argr_plan* plan, int64_t rows);

/*
 * Failure reporting for the bounded device-side waits (onnxruntime #32092,
 * Testing: forced dispatch paths must neither hang nor silently corrupt; the
 * scan's waits follow Paddle issue #79670, "Possible fixes", whose two-pass
 * scan hands chunk totals from one CTA to the next).
 * Synchronise `stream` and read the library's device error words (set by a
 * kernel whose bounded wait expired: for a bulk copy, after which the kernel
 * skips the rest of its work, or for another CTA's chunk record in the split
 * or streaming scan) and the one in `scratch` (may be NULL). Returns
 * ARGR_ESCRATCH if a split or streaming scan found counters or records its
 * launch did not write (a scratch buffer that argreduce_scratch_init() never
 * prepared), else ARGR_ETIMEOUT if
 * any word was set, ARGR_OK otherwise (the words are cleared), and ARGR_ECUDA
 * if the stream reports a fault. For tests and benchmarks; it blocks the host.
 */
argr_status argreduce_read_error(void* scratch, argr_stream stream);

/*
 * argreduce() for callers that cannot allocate device memory. The paper has
 * no counterpart to this entry point: it exists for code that runs where
 * cudaMalloc is not available to it, for example a plugin inside an inference
 * engine that owns every device allocation and hands it no allocator, a
 * real-time path that may not make a call that can synchronise the device or
 * block for an unbounded time, or code that must not grow its memory use
 * after start-up.
 *
 * It runs the split-row kernel (a row spread over CTAs of the whole device,
 * merged by the CTA that arrives last) with its scratch in a 32 KiB array
 * inside this library instead of caller memory. That array exists once per
 * GPU, on every GPU that loads the library, until the process exits. The
 * caller still passes x, out_idx and out_val exactly as for argreduce();
 * there is no scratch argument. The call allocates and frees nothing.
 *
 *   - The first call on each device (with that device current) finds the
 *     array's device address and zeroes it, synchronously. Make that first
 *     call before capturing any stream on the device. The address is kept
 *     for the device's primary context: after cudaDeviceReset(), or with a
 *     context other than the primary one current, it is stale, so do not
 *     call this entry point there.
 *   - Every call reuses the same array, which keeps what the last call left:
 *     two calls that can overlap on the GPU (other streams, other host
 *     threads) race on it and give wrong results; serialise them. No call
 *     clears it: each row's arrival counter is bumped with a wrapping
 *     increment that leaves it at zero when the row's last CTA arrives, and
 *     every partial is written before it is read.
 *   - A problem whose plan needs more than the array holds returns
 *     ARGR_ESCRATCH before anything is queued (on a GB300 every shape fits).
 *   - Other errors as for argreduce(), checked before anything is queued:
 *     ARGR_EUNSUPPORTED for the integer types, ARGR_EINVAL for the rest.
 */
argr_status argreduce_noalloc(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op,
                              int64_t* out_idx, void* out_val, argr_stream stream);

/* Properties of `device` as the planner sees them (queried once, cached). */
argr_status argreduce_device_caps(int device, argr_caps* out);

/* Static, human-readable name of a status code. */
const char* argreduce_status_string(argr_status status);

/* Build identification: "argreduce <version> sm_103a". */
const char* argreduce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ARGREDUCE_H */
