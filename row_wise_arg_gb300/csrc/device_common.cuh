// Device building blocks shared by the argreduce kernels: element tags,
// the (value, index) candidate and its merge rule, 16-byte streaming loads,
// and the warp / CTA merge trees.
//
// Semantics (onnxruntime #32092 Semantics, #31694 Semantics): the result of a
// row equals the sequential scan that seeds with (x[0], 0) and replaces the
// candidate only with a strictly better element. The kernels reproduce it in
// parallel as follows:
//  * every thread seeds its candidate with (x[0], 0), whichever elements it
//    owns, and visits its own elements in increasing index order with the
//    strict test, exactly like the sequential scan on a subsequence;
//  * two candidates merge by "better value wins, equal values keep the lower
//    index". If x[0] is NaN no strict test ever succeeds, so every candidate
//    is (x[0], 0) and so is the merge. Otherwise no candidate holds a NaN,
//    and the merge is the maximum of a total order (value, then lower index),
//    so any merge tree gives the sequential result.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace argr {

constexpr int kOpMax = 0;
constexpr int kOpMin = 1;

// ---------------------------------------------------------------------------
// Element tags: raw storage type, comparison type and the exact widening.
// binary16 and bfloat16 widen exactly to binary32; comparisons there decide
// exactly as in the narrow type.
// ---------------------------------------------------------------------------
struct TagF32 {
    using raw = float;
    using cmp = float;
    static __device__ __forceinline__ float to_cmp(float v) { return v; }
};
struct TagF64 {
    using raw = double;
    using cmp = double;
    static __device__ __forceinline__ double to_cmp(double v) { return v; }
};
struct TagF16 {
    using raw = uint16_t;
    using cmp = float;
    static __device__ __forceinline__ float to_cmp(uint16_t v) {
        return __half2float(__ushort_as_half(v));
    }
};
struct TagBF16 {
    using raw = uint16_t;
    using cmp = float;
    static __device__ __forceinline__ float to_cmp(uint16_t v) {
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    }
};

template <int OP, typename C>
__device__ __forceinline__ bool better(C a, C b) {
    // IEEE comparison: false when either side is NaN.
    if constexpr (OP == kOpMax)
        return a > b;
    else
        return a < b;
}

template <class Tag>
struct Cand {
    typename Tag::raw v;
    int i;
};

// Strict update for elements visited in increasing index order.
template <class Tag, int OP>
__device__ __forceinline__ void visit(Cand<Tag>& c, typename Tag::raw x, int j) {
    if (better<OP>(Tag::to_cmp(x), Tag::to_cmp(c.v))) {
        c.v = x;
        c.i = j;
    }
}

// Merge of two candidates: better value wins; equal values keep the lower index.
template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> merge(Cand<Tag> a, Cand<Tag> b) {
    const auto av = Tag::to_cmp(a.v);
    const auto bv = Tag::to_cmp(b.v);
    const bool take_b = better<OP>(bv, av) || (bv == av && b.i < a.i);
    return take_b ? b : a;
}

// ---------------------------------------------------------------------------
// Shuffles of raw values (16-bit values travel in a 32-bit register).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float shfl_xor_raw(unsigned m, float v, int o, int w) {
    return __shfl_xor_sync(m, v, o, w);
}
__device__ __forceinline__ double shfl_xor_raw(unsigned m, double v, int o, int w) {
    return __shfl_xor_sync(m, v, o, w);
}
__device__ __forceinline__ uint16_t shfl_xor_raw(unsigned m, uint16_t v, int o, int w) {
    return static_cast<uint16_t>(__shfl_xor_sync(m, static_cast<unsigned>(v), o, w));
}
__device__ __forceinline__ float shfl_raw(unsigned m, float v, int src, int w) {
    return __shfl_sync(m, v, src, w);
}
__device__ __forceinline__ double shfl_raw(unsigned m, double v, int src, int w) {
    return __shfl_sync(m, v, src, w);
}
__device__ __forceinline__ uint16_t shfl_raw(unsigned m, uint16_t v, int src, int w) {
    return static_cast<uint16_t>(__shfl_sync(m, static_cast<unsigned>(v), src, w));
}

// Butterfly over groups of G lanes (G a power of two <= 32); every lane of
// the group ends with the group's merged candidate.
template <class Tag, int OP, int G>
__device__ __forceinline__ Cand<Tag> group_merge(Cand<Tag> c, unsigned mask) {
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) {
        Cand<Tag> o;
        o.v = shfl_xor_raw(mask, c.v, off, G);
        o.i = __shfl_xor_sync(mask, c.i, off, G);
        c = merge<Tag, OP>(c, o);
    }
    return c;
}

// Whole-CTA merge. Every thread passes its candidate; the merged candidate is
// returned to all threads of warp 0 (other warps get their own warp's result).
// `smem` holds at least 32 candidates. Contains __syncthreads(): all threads of
// the CTA must call it.
template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> block_merge(Cand<Tag> c, Cand<Tag>* smem, Cand<Tag> seed) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    c = group_merge<Tag, OP, 32>(c, 0xffffffffu);
    if (nwarps == 1) return c;
    if (lane == 0) smem[warp] = c;
    __syncthreads();
    if (warp == 0) {
        c = lane < nwarps ? smem[lane] : seed;
        c = group_merge<Tag, OP, 32>(c, 0xffffffffu);
    }
    return c;
}

// ---------------------------------------------------------------------------
// Streaming loads. The input is read exactly once, so lines are not kept in
// L1 (read-only path, no L1 allocation).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <typename R>
__device__ __forceinline__ R ld_scalar(const R* p) {
    return __ldg(p);
}
__device__ __forceinline__ uint16_t ld_scalar(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
}

// Element k of a 16-byte vector, as the raw type.
template <typename R>
__device__ __forceinline__ R vec_elem(const uint4& v, int k);
template <>
__device__ __forceinline__ float vec_elem<float>(const uint4& v, int k) {
    const uint32_t w = k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
    return __uint_as_float(w);
}
template <>
__device__ __forceinline__ double vec_elem<double>(const uint4& v, int k) {
    return k == 0 ? __hiloint2double(static_cast<int>(v.y), static_cast<int>(v.x))
                  : __hiloint2double(static_cast<int>(v.w), static_cast<int>(v.z));
}
template <>
__device__ __forceinline__ uint16_t vec_elem<uint16_t>(const uint4& v, int k) {
    const uint32_t w = (k >> 1) == 0 ? v.x : (k >> 1) == 1 ? v.y : (k >> 1) == 2 ? v.z : v.w;
    return static_cast<uint16_t>((k & 1) ? (w >> 16) : (w & 0xffffu));
}

// Visit the E elements of one vector; `j0` is the index of its first element.
template <class Tag, int OP>
__device__ __forceinline__ void visit_vec(Cand<Tag>& c, const uint4& v, int j0) {
    using R = typename Tag::raw;
    constexpr int E = 16 / sizeof(R);
#pragma unroll
    for (int k = 0; k < E; ++k) visit<Tag, OP>(c, vec_elem<R>(v, k), j0 + k);
}

}  // namespace argr
