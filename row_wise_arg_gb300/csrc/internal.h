// Host-side declarations shared by the planner, the API layer and the kernel
// launchers. Not part of the public interface (include/argreduce.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "argreduce.h"

#ifdef __CUDACC__
#define ARGR_HD __host__ __device__
#else
#define ARGR_HD
#endif

namespace argr {

// Scratch layout (the buffer is 16-byte aligned). The layout does not depend
// on the plan, so calls with different plans can share one buffer: no call's
// partials ever overlap another call's counters.
//   [0, 4)                     device error word (set by an expired bounded wait)
//   [kCounterOffset, +4*kMaxSplitRows)
//                              one uint32 arrival counter per row slot
//   [kPartialsOffset, ...)     row_slots * blocks_per_row partials of 16 bytes
//                              (raw value bits in the low 8 bytes, index in 4)
//   argreduce_cum's split scan (ARGR_PATH_CUM_SPLIT) uses, in the same buffer:
//   [kCumTicketOffset, +4)     ticket counter (wraps to 0 after each launch)
//   [kCumDoneOffset, +4)       done counter (wraps to 0 after each launch)
//   [kCounterOffset, +8*kCumMaxChunks)
//                              one 64-bit record per chunk for launches of up to
//                              kCumMaxChunks chunks, zeroed again by the
//                              launch's last CTA, so the split counters stay 0
//   [kCumBigRecordsOffset, +8*chunks)
//                              the records of larger launches (up to
//                              kCumMaxChunksBig chunks), zeroed the same way;
//                              argreduce's partials never reach this offset
constexpr size_t kCounterOffset = 256;
constexpr int64_t kMaxSplitRows = 2048;  // row slots a multi-CTA split may use
constexpr size_t kPartialsOffset = kCounterOffset + 4 * kMaxSplitRows;
constexpr size_t kPartialBytes = 16;
constexpr size_t kCumTicketOffset = 4;
constexpr size_t kCumDoneOffset = 8;
constexpr size_t kCumRecordsOffset = kCounterOffset;
constexpr int64_t kCumMaxChunks = kMaxSplitRows / 2;  // rows * chunks of a split scan, small region
constexpr size_t kCumBigRecordsOffset = size_t(1) << 20;
constexpr int64_t kCumMaxChunksBig = 65536;           // rows * chunks of a split scan, large region
constexpr int64_t kMaxPartials = (kCumBigRecordsOffset - kPartialsOffset) / kPartialBytes;
constexpr int64_t kCumStashBytes = 80 * 1024;         // a stashed split-scan chunk, at most
constexpr int kPipeMaxBlock = 256;  // threads per CTA of the pipelined rows kernel (its registers)
ARGR_HD inline size_t cum_records_offset(int64_t total_chunks) {
    return total_chunks <= kCumMaxChunks ? kCounterOffset : kCumBigRecordsOffset;
}

ARGR_HD inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Problem {
    const void* x;
    int dtype;     // argr_dtype
    int op;        // argr_op
    int64_t rows;  // last axis: rows. Non-last axis: outer
    int cols;      // 1 .. INT32_MAX. Last axis: columns. Non-last axis: the reduced extent R
    int64_t inner; // non-last axis: elements after the reduced axis (1 for the last axis)
    int64_t* out_idx;
    void* out_val;
    void* scratch;
    cudaStream_t stream;
};

int elem_size(int dtype);

// Planner (plan.cpp): pure host code. `base_aligned`: x is 16-byte aligned.
argr_status make_plan(int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps, bool base_aligned,
                      argr_plan* out);
// Validates a (possibly hand-edited) plan for this problem and device.
// `row_aligned`: every row start is 16-byte aligned (base aligned and
// cols * elem_size a multiple of 16).
argr_status check_plan(const argr_plan& p, int64_t rows, int64_t cols, int dtype, const argr_caps& caps,
                       bool row_aligned);
size_t plan_scratch(const argr_plan& p, int64_t rows);
// Non-last axis x[outer][reduce][inner]: a last-axis plan when inner == 1,
// else an ARGR_PATH_AXIS plan. `base_aligned`: x is 16-byte aligned.
argr_status make_axis_plan(int64_t outer, int64_t reduce, int64_t inner, int dtype, int op, const argr_caps& caps,
                           bool base_aligned, argr_plan* out);
argr_status check_axis_plan(const argr_plan& p, int64_t outer, int64_t reduce, int64_t inner, int dtype,
                            const argr_caps& caps, uintptr_t x_addr);

// Kernel launchers (one translation unit per element type). They assume a
// checked plan and return the launch's CUDA error.
#define ARGR_DECLARE_LAUNCHERS(sfx)                                              \
    cudaError_t launch_rows_##sfx(const argr_plan& p, const Problem& pr);    \
    cudaError_t launch_split_##sfx(const argr_plan& p, const Problem& pr);   \
    cudaError_t launch_cluster_##sfx(const argr_plan& p, const Problem& pr); \
    cudaError_t launch_stream_##sfx(const argr_plan& p, const Problem& pr);  \
    cudaError_t launch_axis_##sfx(const argr_plan& p, const Problem& pr);    \
    cudaError_t read_and_clear_error_##sfx(unsigned* out);
ARGR_DECLARE_LAUNCHERS(f32)
ARGR_DECLARE_LAUNCHERS(f16)
ARGR_DECLARE_LAUNCHERS(bf16)
ARGR_DECLARE_LAUNCHERS(f64)
#undef ARGR_DECLARE_LAUNCHERS

// cummax / cummin (argreduce_cum), one translation unit per element type.
cudaError_t launch_cum_f32(const argr_plan& p, const Problem& pr);
cudaError_t launch_cum_f16(const argr_plan& p, const Problem& pr);
cudaError_t launch_cum_bf16(const argr_plan& p, const Problem& pr);
cudaError_t launch_cum_f64(const argr_plan& p, const Problem& pr);
cudaError_t launch_cum_i32(const argr_plan& p, const Problem& pr);
cudaError_t launch_cum_i64(const argr_plan& p, const Problem& pr);
argr_status make_cum_plan(int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps, argr_plan* out);
argr_status check_cum_plan(const argr_plan& p, int64_t rows, int64_t cols, int dtype, int op, const argr_caps& caps);
// Scratch bytes of a cummax / cummin plan (records of the split and streaming scans).
size_t cum_plan_scratch(const argr_plan& p, int64_t rows);

}  // namespace argr
