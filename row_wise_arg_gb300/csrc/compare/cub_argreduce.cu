// Timing comparison only: cub::DeviceReduce::ArgMax / ArgMin on one row
// [1, n], called as a library (onnxruntime PR #32092, Profile: after the
// profile of [1, 202048] the PR compares its kernel with
// cub::DeviceReduce::ArgMax on the same GPU and shape, the other reference
// point for a single wide row).
// Built into its own libcubcompare.so, which the benchmark and one GPU test
// load; nothing in libargreduce.so uses it.
//
// CUB returns the first maximum (minimum) under `>` (`<`), so on NaN-free
// rows its index equals argreduce()'s; NaN handling differs and is not
// compared.
#include <cstdint>
#include <cstddef>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cub/device/device_reduce.cuh>

namespace {

template <typename T>
cudaError_t run(void* temp, size_t& temp_bytes, const void* x, int op, int64_t n, void* out_val, int64_t* out_idx,
                cudaStream_t stream) {
    const T* in = static_cast<const T*>(x);
    T* val = static_cast<T*>(out_val);
    if (op == 0) return cub::DeviceReduce::ArgMax(temp, temp_bytes, in, val, out_idx, n, stream);
    return cub::DeviceReduce::ArgMin(temp, temp_bytes, in, val, out_idx, n, stream);
}

cudaError_t dispatch(void* temp, size_t& temp_bytes, const void* x, int dtype, int op, int64_t n, void* out_val,
                     int64_t* out_idx, cudaStream_t stream) {
    switch (dtype) {  // argr_dtype codes
        case 0: return run<float>(temp, temp_bytes, x, op, n, out_val, out_idx, stream);
        case 1: return run<__half>(temp, temp_bytes, x, op, n, out_val, out_idx, stream);
        case 2: return run<__nv_bfloat16>(temp, temp_bytes, x, op, n, out_val, out_idx, stream);
        case 3: return run<double>(temp, temp_bytes, x, op, n, out_val, out_idx, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

extern "C" {

// Temporary storage CUB needs for one row of n elements (0 on a bad argument).
size_t cubcmp_temp_bytes(int dtype, int op, int64_t n) {
    size_t bytes = 0;
    if (n < 1 || (op != 0 && op != 1)) return 0;
    if (dispatch(nullptr, bytes, nullptr, dtype, op, n, nullptr, nullptr, nullptr) != cudaSuccess) return 0;
    return bytes;
}

// ArgMax (op 0) / ArgMin (op 1) of x[0..n) with CUB: the extremum into
// out_val (one element of the input type), its index into out_idx. Returns a
// cudaError_t code; launches only, no allocation or synchronisation.
int cubcmp_argreduce(const void* x, int dtype, int op, int64_t n, void* out_val, int64_t* out_idx, void* temp,
                     size_t temp_bytes, void* stream) {
    if (!x || !out_val || !out_idx || !temp || n < 1 || (op != 0 && op != 1)) return cudaErrorInvalidValue;
    size_t bytes = temp_bytes;
    return dispatch(temp, bytes, x, dtype, op, n, out_val, out_idx, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
