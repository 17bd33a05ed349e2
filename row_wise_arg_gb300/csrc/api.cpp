// C ABI of libargreduce.so: argument validation, device queries, dispatch to
// the kernel launchers. Every check happens before anything is queued; the
// library never allocates, frees or synchronises inside argreduce().
#include <climits>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace argr {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_caps_mu;
argr_caps g_caps[kMaxDevices];
bool g_caps_valid[kMaxDevices];

argr_status query_caps(int dev, argr_caps* out) {
    if (dev < 0 || dev >= kMaxDevices) return ARGR_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_caps_mu);
    if (!g_caps_valid[dev]) {
        argr_caps c{};
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ARGR_ECUDA;
        c.sm_count = v;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess)
            return ARGR_ECUDA;
        c.max_threads_per_sm = v;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return ARGR_ECUDA;
        c.cc_major = v;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return ARGR_ECUDA;
        c.cc_minor = v;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrClusterLaunch, dev) != cudaSuccess) v = 0;
        // Cluster launch is available from compute capability 9.0; 16 CTAs is
        // the non-portable maximum (enabled per kernel at launch).
        c.max_cluster = v ? 16 : 1;
        g_caps[dev] = c;
        g_caps_valid[dev] = true;
    }
    *out = g_caps[dev];
    return ARGR_OK;
}

argr_status current_caps(argr_caps* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    return query_caps(dev, out);
}

bool valid_dtype(int d) { return d == ARGR_F32 || d == ARGR_F16 || d == ARGR_BF16 || d == ARGR_F64; }
bool valid_op(int o) { return o == ARGR_MAX || o == ARGR_MIN || o == ARGR_MAX_LAST || o == ARGR_MIN_LAST; }

// Checks shared by argreduce() and argreduce_with_plan().
argr_status check_args(const void* x, int dtype, int64_t rows, int64_t cols, int op, const int64_t* out_idx,
                       const void* out_val) {
    if (dtype == ARGR_I32 || dtype == ARGR_I64) return ARGR_EUNSUPPORTED;  // integer types: argreduce_cum only
    if (!valid_dtype(dtype) || !valid_op(op)) return ARGR_EINVAL;
    if (rows < 0 || cols < 1 || cols > INT_MAX) return ARGR_EINVAL;
    const int64_t es = elem_size(dtype);
    if (rows > INT64_MAX / cols / es) return ARGR_EINVAL;  // rows * cols * es must fit
    if (rows == 0) return ARGR_OK;
    if (!x || !out_idx) return ARGR_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % es != 0) return ARGR_EINVAL;
    if (reinterpret_cast<uintptr_t>(out_idx) % 8 != 0) return ARGR_EINVAL;
    if (out_val && reinterpret_cast<uintptr_t>(out_val) % es != 0) return ARGR_EINVAL;
    return ARGR_OK;
}

bool rows_aligned(const void* x, int dtype, int64_t cols) {
    return reinterpret_cast<uintptr_t>(x) % 16 == 0 && (cols * elem_size(dtype)) % 16 == 0;
}

argr_status run(const argr_plan& p, const Problem& pr, size_t scratch_bytes) {
    const size_t need = plan_scratch(p, pr.rows);
    if (need > 0) {
        if (!pr.scratch || scratch_bytes < need) return ARGR_ESCRATCH;
        if (reinterpret_cast<uintptr_t>(pr.scratch) % 16 != 0) return ARGR_ESCRATCH;
    }
    cudaError_t e = cudaErrorInvalidValue;
#define ARGR_DISPATCH(sfx)                                                 \
    switch (p.path) {                                                      \
        case ARGR_PATH_ROWS: e = launch_rows_##sfx(p, pr); break;          \
        case ARGR_PATH_SPLIT: e = launch_split_##sfx(p, pr); break;        \
        case ARGR_PATH_CLUSTER: e = launch_cluster_##sfx(p, pr); break;    \
        case ARGR_PATH_STREAM: e = launch_stream_##sfx(p, pr); break;      \
        case ARGR_PATH_AXIS: e = launch_axis_##sfx(p, pr); break;          \
        default: return ARGR_EINVAL;                                       \
    }
    switch (pr.dtype) {
        case ARGR_F32: ARGR_DISPATCH(f32) break;
        case ARGR_F16: ARGR_DISPATCH(f16) break;
        case ARGR_BF16: ARGR_DISPATCH(bf16) break;
        case ARGR_F64: ARGR_DISPATCH(f64) break;
        default: return ARGR_EINVAL;
    }
#undef ARGR_DISPATCH
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear a non-sticky launch error
        return e == cudaErrorInvalidClusterSize ? ARGR_EUNSUPPORTED : ARGR_ECUDA;
    }
    return ARGR_OK;
}

Problem make_problem(const void* x, int dtype, int64_t rows, int64_t cols, int op, int64_t* out_idx,
                     void* out_val, void* scratch, argr_stream stream) {
    Problem pr;
    pr.x = x;
    pr.dtype = dtype;
    pr.op = op;
    pr.rows = rows;
    pr.cols = static_cast<int>(cols);
    pr.inner = 1;
    pr.out_idx = out_idx;
    pr.out_val = out_val;
    pr.scratch = scratch;
    pr.stream = reinterpret_cast<cudaStream_t>(stream);
    return pr;
}

}  // namespace
}  // namespace argr

using namespace argr;

extern "C" {

size_t argreduce_scratch_bytes(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op) {
    argr_caps caps;
    if (current_caps(&caps) != ARGR_OK) return 0;
    argr_plan p;
    if (make_plan(rows, cols, dtype, op, caps, true, &p) != ARGR_OK) return 0;
    // The plan for an unaligned base never needs more scratch than this one:
    // alignment only changes the rows path, which needs none.
    return p.scratch_bytes;
}

argr_status argreduce_scratch_init(void* scratch, size_t scratch_bytes, argr_stream stream) {
    if (scratch_bytes == 0) return ARGR_OK;
    if (!scratch) return ARGR_EINVAL;
    if (reinterpret_cast<uintptr_t>(scratch) % 16 != 0) return ARGR_ESCRATCH;
    if (cudaMemsetAsync(scratch, 0, scratch_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    return ARGR_OK;
}

argr_status argreduce(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op, int64_t* out_idx,
                      void* out_val, void* scratch, size_t scratch_bytes, argr_stream stream) {
    argr_status s = check_args(x, dtype, rows, cols, op, out_idx, out_val);
    if (s != ARGR_OK || rows == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    argr_plan p;
    const bool base_aligned = reinterpret_cast<uintptr_t>(x) % 16 == 0;
    if ((s = make_plan(rows, cols, dtype, op, caps, base_aligned, &p)) != ARGR_OK) return s;
    return run(p, make_problem(x, dtype, rows, cols, op, out_idx, out_val, scratch, stream), scratch_bytes);
}

argr_status argreduce_plan(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op, const argr_caps* caps,
                           argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    argr_caps c;
    if (caps) {
        c = *caps;
    } else {
        argr_status s = current_caps(&c);
        if (s != ARGR_OK) return s;
    }
    return make_plan(rows, cols, dtype, op, c, true, out);
}

argr_status argreduce_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t rows, int64_t cols,
                                argr_op op, int64_t* out_idx, void* out_val, void* scratch, size_t scratch_bytes,
                                argr_stream stream) {
    if (!plan) return ARGR_EINVAL;
    argr_status s = check_args(x, dtype, rows, cols, op, out_idx, out_val);
    if (s != ARGR_OK || rows == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    if ((s = check_plan(*plan, rows, cols, dtype, caps, rows_aligned(x, dtype, cols))) != ARGR_OK) return s;
    return run(*plan, make_problem(x, dtype, rows, cols, op, out_idx, out_val, scratch, stream), scratch_bytes);
}

argr_status argreduce_plan_check(const argr_plan* plan, int64_t rows, int64_t cols, argr_dtype dtype,
                                 const argr_caps* caps, int rows_aligned) {
    if (!plan || !caps) return ARGR_EINVAL;
    return check_plan(*plan, rows, cols, dtype, *caps, rows_aligned != 0);
}

// ---------------------------------------------------------------------------
// Reduction over a non-last axis.
// ---------------------------------------------------------------------------
static argr_status check_axis_args(const void* x, int dtype, int64_t outer, int64_t reduce, int64_t inner, int op,
                                   const int64_t* out_idx, const void* out_val) {
    if (inner < 1 || outer < 0) return ARGR_EINVAL;
    if (outer > 0 && inner > INT64_MAX / outer) return ARGR_EINVAL;
    // the same checks as a [outer * inner, reduce] problem (sizes, alignment)
    return check_args(x, dtype, outer * inner, reduce, op, out_idx, out_val);
}

argr_status argreduce_axis_plan(int64_t outer, int64_t reduce, int64_t inner, argr_dtype dtype, argr_op op,
                                const argr_caps* caps, argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    argr_caps c;
    if (caps) {
        c = *caps;
    } else {
        argr_status s = current_caps(&c);
        if (s != ARGR_OK) return s;
    }
    return make_axis_plan(outer, reduce, inner, dtype, op, c, true, out);
}

static argr_status run_axis(const argr_plan& p, const void* x, int dtype, int64_t outer, int64_t reduce,
                            int64_t inner, int op, int64_t* out_idx, void* out_val, void* scratch,
                            size_t scratch_bytes, argr_stream stream) {
    if (p.path != ARGR_PATH_AXIS) {
        // inner == 1: the last-axis problem [outer, reduce]
        return run(p, make_problem(x, dtype, outer, reduce, op, out_idx, out_val, scratch, stream), scratch_bytes);
    }
    Problem pr = make_problem(x, dtype, outer, reduce, op, out_idx, out_val, scratch, stream);
    pr.inner = inner;
    return run(p, pr, scratch_bytes);
}

argr_status argreduce_axis(const void* x, argr_dtype dtype, int64_t outer, int64_t reduce, int64_t inner,
                           argr_op op, int64_t* out_idx, void* out_val, void* scratch, size_t scratch_bytes,
                           argr_stream stream) {
    argr_status s = check_axis_args(x, dtype, outer, reduce, inner, op, out_idx, out_val);
    if (s != ARGR_OK || outer == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    argr_plan p;
    if ((s = make_axis_plan(outer, reduce, inner, dtype, op, caps, reinterpret_cast<uintptr_t>(x) % 16 == 0, &p)) !=
        ARGR_OK)
        return s;
    return run_axis(p, x, dtype, outer, reduce, inner, op, out_idx, out_val, scratch, scratch_bytes, stream);
}

argr_status argreduce_axis_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t outer,
                                     int64_t reduce, int64_t inner, argr_op op, int64_t* out_idx, void* out_val,
                                     void* scratch, size_t scratch_bytes, argr_stream stream) {
    if (!plan) return ARGR_EINVAL;
    argr_status s = check_axis_args(x, dtype, outer, reduce, inner, op, out_idx, out_val);
    if (s != ARGR_OK || outer == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    if (plan->path == ARGR_PATH_AXIS) {
        if ((s = check_axis_plan(*plan, outer, reduce, inner, dtype, caps, reinterpret_cast<uintptr_t>(x))) != ARGR_OK)
            return s;
    } else {
        if (inner != 1) return ARGR_EINVAL;  // a last-axis plan needs inner == 1
        if ((s = check_plan(*plan, outer, reduce, dtype, caps, rows_aligned(x, dtype, reduce))) != ARGR_OK) return s;
    }
    return run_axis(*plan, x, dtype, outer, reduce, inner, op, out_idx, out_val, scratch, scratch_bytes, stream);
}

// ---------------------------------------------------------------------------
// cummax / cummin.
// ---------------------------------------------------------------------------
static argr_status check_cum_args(const void* x, int dtype, int64_t rows, int64_t cols, int op,
                                  const int64_t* out_idx, const void* out_val) {
    const int64_t es = elem_size(dtype);
    if (es == 0 || op < ARGR_MAX || op > ARGR_MIN_LAST) return ARGR_EINVAL;
    if (op != ARGR_MAX && op != ARGR_MIN) return ARGR_EUNSUPPORTED;
    if (rows < 0 || cols < 1 || cols > INT_MAX || rows > INT64_MAX / cols / 8) return ARGR_EINVAL;
    if (rows == 0) return ARGR_OK;
    if (!x || !out_idx) return ARGR_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % es || reinterpret_cast<uintptr_t>(out_idx) % 8) return ARGR_EINVAL;
    if (out_val && reinterpret_cast<uintptr_t>(out_val) % es) return ARGR_EINVAL;
    return ARGR_OK;
}

static argr_status run_cum(const argr_plan& p, const void* x, int dtype, int64_t rows, int64_t cols, int op,
                           int64_t* out_idx, void* out_val, void* scratch, size_t scratch_bytes,
                           argr_stream stream) {
    const size_t need = plan_scratch(p, rows);
    if (need > 0) {
        if (!scratch || scratch_bytes < need) return ARGR_ESCRATCH;
        if (reinterpret_cast<uintptr_t>(scratch) % 16 != 0) return ARGR_ESCRATCH;
    }
    Problem pr = make_problem(x, dtype, rows, cols, op, out_idx, out_val, scratch, stream);
    cudaError_t e = cudaErrorInvalidValue;
    switch (dtype) {
        case ARGR_F32: e = launch_cum_f32(p, pr); break;
        case ARGR_F16: e = launch_cum_f16(p, pr); break;
        case ARGR_BF16: e = launch_cum_bf16(p, pr); break;
        case ARGR_F64: e = launch_cum_f64(p, pr); break;
        case ARGR_I32: e = launch_cum_i32(p, pr); break;
        case ARGR_I64: e = launch_cum_i64(p, pr); break;
        default: return ARGR_EINVAL;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorInvalidClusterSize ? ARGR_EUNSUPPORTED : ARGR_ECUDA;
    }
    return ARGR_OK;
}

argr_status argreduce_cum(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op, int64_t* out_idx,
                          void* out_val, void* scratch, size_t scratch_bytes, argr_stream stream) {
    argr_status s = check_cum_args(x, dtype, rows, cols, op, out_idx, out_val);
    if (s != ARGR_OK || rows == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    argr_plan p;
    if ((s = make_cum_plan(rows, cols, dtype, op, caps, &p)) != ARGR_OK) return s;
    return run_cum(p, x, dtype, rows, cols, op, out_idx, out_val, scratch, scratch_bytes, stream);
}

size_t argreduce_cum_scratch_bytes(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op) {
    argr_caps caps;
    if (current_caps(&caps) != ARGR_OK) return 0;
    argr_plan p;
    if (make_cum_plan(rows, cols, dtype, op, caps, &p) != ARGR_OK) return 0;
    return p.scratch_bytes;
}

argr_status argreduce_cum_plan(int64_t rows, int64_t cols, argr_dtype dtype, argr_op op, const argr_caps* caps,
                               argr_plan* out) {
    if (!out) return ARGR_EINVAL;
    argr_caps c;
    if (caps) {
        c = *caps;
    } else {
        argr_status s = current_caps(&c);
        if (s != ARGR_OK) return s;
    }
    return make_cum_plan(rows, cols, dtype, op, c, out);
}

argr_status argreduce_cum_with_plan(const argr_plan* plan, const void* x, argr_dtype dtype, int64_t rows,
                                    int64_t cols, argr_op op, int64_t* out_idx, void* out_val, void* scratch,
                                    size_t scratch_bytes, argr_stream stream) {
    if (!plan) return ARGR_EINVAL;
    argr_status s = check_cum_args(x, dtype, rows, cols, op, out_idx, out_val);
    if (s != ARGR_OK || rows == 0) return s;
    argr_caps caps;
    if ((s = current_caps(&caps)) != ARGR_OK) return s;
    if ((s = check_cum_plan(*plan, rows, cols, dtype, op, caps)) != ARGR_OK) return s;
    return run_cum(*plan, x, dtype, rows, cols, op, out_idx, out_val, scratch, scratch_bytes, stream);
}

size_t argreduce_plan_scratch_bytes(const argr_plan* plan, int64_t rows) {
    return plan ? plan_scratch(*plan, rows) : 0;
}

argr_status argreduce_read_error(void* scratch, argr_stream stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    if (scratch && reinterpret_cast<uintptr_t>(scratch) % 16 != 0) return ARGR_ESCRATCH;
    // Error words of the kernels of every element type (bounded waits that
    // expired), and the one in the caller's scratch.
    unsigned any = 0;
    cudaError_t (*readers[])(unsigned*) = {read_and_clear_error_f32, read_and_clear_error_f16,
                                           read_and_clear_error_bf16, read_and_clear_error_f64};
    for (auto rd : readers) {
        unsigned v = 0;
        if (rd(&v) != cudaSuccess) {
            cudaGetLastError();
            return ARGR_ECUDA;
        }
        any |= v;
    }
    if (scratch) {
        unsigned int word = 0;
        if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return ARGR_ECUDA;
        }
        if (word) {
            const unsigned int zero = 0;
            if (cudaMemcpy(scratch, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
                cudaGetLastError();
                return ARGR_ECUDA;
            }
        }
        any |= word;
    }
    if (any & 2u) return ARGR_ESCRATCH;  // a split scan met a ticket or record its launch did not write
    return any ? ARGR_ETIMEOUT : ARGR_OK;
}

argr_status argreduce_device_caps(int device, argr_caps* out) {
    if (!out) return ARGR_EINVAL;
    return query_caps(device, out);
}

const char* argreduce_status_string(argr_status status) {
    switch (status) {
        case ARGR_OK: return "ARGR_OK: success";
        case ARGR_EINVAL: return "ARGR_EINVAL: invalid argument or plan";
        case ARGR_ESCRATCH: return "ARGR_ESCRATCH: scratch missing, too small or misaligned";
        case ARGR_EUNSUPPORTED: return "ARGR_EUNSUPPORTED: not supported on this device";
        case ARGR_ECUDA: return "ARGR_ECUDA: CUDA runtime error";
        case ARGR_ETIMEOUT: return "ARGR_ETIMEOUT: a bounded device wait expired";
        default: return "unknown argr_status";
    }
}

const char* argreduce_version(void) { return "argreduce 0.1.0 sm_103a"; }

}  // extern "C"
