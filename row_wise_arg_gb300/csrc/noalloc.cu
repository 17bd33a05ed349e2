// argreduce_noalloc(): the split-row ArgMax/ArgMin with its scratch in a
// fixed device array owned by this library, for callers that cannot allocate
// device memory (see include/argreduce.h).
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it. Host code cannot use the array's name as a device address (on the
// host the name refers to a host-side shadow), so the first call on each
// device looks up the real device address with cudaGetSymbolAddress() and
// zeroes the array once; later calls reuse the cached address. The address
// belongs to the device's primary context: after cudaDeviceReset(), or with
// another context current, it is no longer valid (documented limit).
//
// No call clears anything: the split kernel bumps each row's arrival counter
// with a wrapping increment, so the last CTA of a row leaves it at zero, and
// the partials are written before they are read in every launch.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace argr {
namespace {

// Room for the fixed header and counters plus 1520 partials: every split plan
// on a device of up to 190 SMs (one wave of 256-thread CTAs) fits.
constexpr size_t kNoAllocScratchBytes = 32768;
static_assert(kNoAllocScratchBytes > kPartialsOffset, "no room for partials");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices];

// Device address of the array on the current device; set up on first use.
argr_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return ARGR_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return ARGR_ECUDA;
        }
        if (cudaMemset(p, 0, kNoAllocScratchBytes) != cudaSuccess) {
            cudaGetLastError();
            return ARGR_ECUDA;
        }
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return ARGR_OK;
}

// The same checks as argreduce(): the integer types are argreduce_cum()'s
// only (ARGR_EUNSUPPORTED), anything else malformed is ARGR_EINVAL.
argr_status check_noalloc_args(const void* x, int dtype, int64_t rows, int64_t cols, int op, const int64_t* out_idx,
                               const void* out_val) {
    if (dtype == ARGR_I32 || dtype == ARGR_I64) return ARGR_EUNSUPPORTED;
    if (dtype != ARGR_F32 && dtype != ARGR_F16 && dtype != ARGR_BF16 && dtype != ARGR_F64) return ARGR_EINVAL;
    const int es = elem_size(dtype);
    if (op < ARGR_MAX || op > ARGR_MIN_LAST) return ARGR_EINVAL;
    if (rows < 0 || cols < 1 || cols > INT32_MAX || rows > INT64_MAX / cols / es) return ARGR_EINVAL;
    if (rows == 0) return ARGR_OK;
    if (!x || !out_idx) return ARGR_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % es || reinterpret_cast<uintptr_t>(out_idx) % 8) return ARGR_EINVAL;
    if (out_val && reinterpret_cast<uintptr_t>(out_val) % es) return ARGR_EINVAL;
    return ARGR_OK;
}

}  // namespace
}  // namespace argr

using namespace argr;

extern "C" argr_status argreduce_noalloc(const void* x, argr_dtype dtype, int64_t rows, int64_t cols, argr_op op,
                                         int64_t* out_idx, void* out_val, argr_stream stream) {
    const argr_status bad = check_noalloc_args(x, dtype, rows, cols, op, out_idx, out_val);
    if (bad != ARGR_OK || rows == 0) return bad;
    argr_caps caps;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    if (argreduce_device_caps(dev, &caps) != ARGR_OK) return ARGR_ECUDA;

    // The split-row plan: each row spread over CTAs of the whole device (about
    // one wave in total), merged through the scratch array by the CTA that
    // arrives last. Many rows (or more than the counters cover) get one CTA
    // per row, which needs no scratch.
    const int64_t es = elem_size(dtype);
    const int64_t row_bytes = cols * es;
    const int64_t wave = static_cast<int64_t>(caps.sm_count) * (caps.max_threads_per_sm / 256);
    argr_plan p{};
    p.path = ARGR_PATH_SPLIT;
    p.block = 256;
    p.unroll = 4;
    p.flags = ARGR_PLAN_PDL;
    if (rows < wave && rows <= kMaxSplitRows) {
        int64_t bpr = wave / rows;
        bpr = std::min<int64_t>(bpr, std::max<int64_t>(1, row_bytes / (256 * 16)));
        bpr = std::min<int64_t>(bpr, 65535);
        p.blocks_per_row = std::max<int64_t>(1, bpr);
        p.grid_rows = rows;
    } else {
        p.blocks_per_row = 1;
        p.grid_rows = std::min<int64_t>(rows, 65535);
    }
    const size_t need = plan_scratch(p, rows);
    if (need > kNoAllocScratchBytes) return ARGR_ESCRATCH;  // larger than the built-in array

    void* scratch = nullptr;
    argr_status s = scratch_for_current_device(&scratch);
    if (s != ARGR_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
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
    pr.stream = st;
    cudaError_t e = cudaErrorInvalidValue;
    switch (dtype) {
        case ARGR_F32: e = launch_split_f32(p, pr); break;
        case ARGR_F16: e = launch_split_f16(p, pr); break;
        case ARGR_BF16: e = launch_split_bf16(p, pr); break;
        case ARGR_F64: e = launch_split_f64(p, pr); break;
        default: return ARGR_EINVAL;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ARGR_ECUDA;
    }
    return ARGR_OK;
}
