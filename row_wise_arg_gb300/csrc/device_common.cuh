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
//  * the last-occurrence ops use the non-strict test ("not worse", still
//    false on NaN) and merge equal values toward the higher index; the same
//    argument applies with the index order reversed.
// Comparisons go through per-type keys (below) that decide exactly as the
// IEEE comparison of the element type.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace argr {

// Ops: ArgMax and ArgMin, first occurrence (0, 1) and last occurrence (2, 3:
// ONNX select_last_index = 1). Bit 0 selects min, bit 1 selects last.
constexpr int kOpMax = 0;
constexpr int kOpMin = 1;
constexpr int kOpMaxLast = 2;
constexpr int kOpMinLast = 3;
template <int OP> constexpr bool kIsMin = (OP & 1) != 0;
template <int OP> constexpr bool kIsLast = (OP & 2) != 0;

// ---------------------------------------------------------------------------
// Element tags: raw storage type and a comparison key.
//
// elem_key(x) is the key of an element the scan visits; seed_key(x) the key
// of a candidate value. better(a, b) says key a is strictly better than key b.
// For binary32, binary16 and bfloat16 the key is the exactly widened binary32
// value and better() is the IEEE comparison, false when either side is NaN.
//
// binary64 is compared through order-preserving 64-bit integer keys instead
// (this GPU's FP64 pipe is far too slow to compare at memory speed): for
// non-NaN values the key is monotone in the value (reversed for ArgMin) and
// +0.0 and -0.0 share one key. A NaN element gets key 0, which nothing is
// worse than, so it never wins; a NaN candidate (only ever x[0]) gets the
// all-ones key, so nothing displaces it. Neither sentinel is the key of a
// number, so "strictly better" decides exactly as the IEEE comparison does.
// The row scans skip the NaN test: order_key() of a NaN lies outside the keys of
// numbers, above kLimit (the key of the best infinity) or below every key of
// a number, so one comparison with kLimit excludes it.
// ---------------------------------------------------------------------------
struct TagF32 {
    using raw = float;
    using key = float;
    template <int OP> static __device__ __forceinline__ float elem_key(float v) { return v; }
    template <int OP> static __device__ __forceinline__ float seed_key(float v) { return v; }
    template <int OP> static __device__ __forceinline__ bool better(float a, float b) {
        if constexpr (kIsMin<OP>) return a < b; else return a > b;
    }
};
struct TagF16 {
    using raw = uint16_t;
    using key = float;
    static __device__ __forceinline__ float widen(uint16_t v) { return __half2float(__ushort_as_half(v)); }
    template <int OP> static __device__ __forceinline__ float elem_key(uint16_t v) { return widen(v); }
    template <int OP> static __device__ __forceinline__ float seed_key(uint16_t v) { return widen(v); }
    template <int OP> static __device__ __forceinline__ bool better(float a, float b) {
        if constexpr (kIsMin<OP>) return a < b; else return a > b;
    }
};
struct TagBF16 {
    using raw = uint16_t;
    using key = float;
    static __device__ __forceinline__ float widen(uint16_t v) {
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    }
    template <int OP> static __device__ __forceinline__ float elem_key(uint16_t v) { return widen(v); }
    template <int OP> static __device__ __forceinline__ float seed_key(uint16_t v) { return widen(v); }
    template <int OP> static __device__ __forceinline__ bool better(float a, float b) {
        if constexpr (kIsMin<OP>) return a < b; else return a > b;
    }
};
struct TagF64 {
    // Raw binary64 elements are carried as their 64-bit patterns: no value
    // of type double exists in the kernels, so nothing runs on the FP64 pipe.
    using raw = unsigned long long;
    using key = unsigned long long;
    static constexpr unsigned long long kSign = 0x8000000000000000ull;
    static constexpr unsigned long long kInfBits = 0x7FF0000000000000ull;
    // Key of a value (larger key = better for OP), monotone on the numbers.
    // ArgMax: a negative value maps to its two's complement negation -b,
    // which gives -0.0 the key kSign of +0.0, a positive one to b with the
    // sign bit set. ArgMin uses the ArgMax key of the negated value (sign bit
    // flipped). The keys of numbers lie in [0x0010000000000000, kLimit];
    // NaNs whose sign bit (after the flip) is clear map above that range,
    // the others below it.
    template <int OP> static __device__ __forceinline__ unsigned long long order_key(unsigned long long b) {
        if constexpr (kIsMin<OP>) b ^= kSign;
        const unsigned long long s = static_cast<unsigned long long>(static_cast<long long>(b) >> 63);
        return ((b ^ s) - s) ^ (~s & kSign);
    }
    // The key of the best infinity (+inf for ArgMax, -inf for ArgMin).
    static constexpr unsigned long long kLimit = 0xFFF0000000000000ull;
    template <int OP> static __device__ __forceinline__ unsigned long long elem_key(unsigned long long b) {
        return (b & ~kSign) > kInfBits ? 0ull : order_key<OP>(b);
    }
    template <int OP> static __device__ __forceinline__ unsigned long long seed_key(unsigned long long b) {
        return (b & ~kSign) > kInfBits ? ~0ull : order_key<OP>(b);
    }
    template <int OP> static __device__ __forceinline__ bool better(unsigned long long a, unsigned long long b) {
        return a > b;
    }
};

// A candidate: raw value (its bits are what out_val receives), its key, and
// its index in the row.
template <class Tag>
struct Cand {
    typename Tag::raw v;
    typename Tag::key k;
    int i;
};

template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> make_cand(typename Tag::raw v, int i) {
    return Cand<Tag>{v, Tag::template seed_key<OP>(v), i};
}

// Update for elements visited in increasing index order: strictly better for
// the first-occurrence ops, not worse for the last-occurrence ops.
template <class Tag, int OP>
__device__ __forceinline__ void visit(Cand<Tag>& c, typename Tag::raw x, int j) {
    if constexpr (sizeof(typename Tag::raw) == 8) {
        // binary64: order_key() without the NaN test. A NaN whose key lies above
        // kLimit is excluded by the first comparison; one whose key lies
        // below every key of a number is never better than the candidate nor
        // equal to it (the candidate is a number or the all-ones NaN seed).
        const typename Tag::key k = Tag::template order_key<OP>(x);
        if (k <= Tag::kLimit && (kIsLast<OP> ? k >= c.k : k > c.k)) {
            c.v = x;
            c.k = k;
            c.i = j;
        }
    } else {
        // "better or equal" is one IEEE comparison (>= / <=, false on NaN).
        const typename Tag::key k = Tag::template elem_key<OP>(x);
        bool take;
        if constexpr (kIsLast<OP>) take = kIsMin<OP> ? k <= c.k : k >= c.k;
        else take = Tag::template better<OP>(k, c.k);
        if (take) {
            c.v = x;
            c.k = k;
            c.i = j;
        }
    }
}

// Programmatic dependent launch. Every kernel waits for the grid before it in
// the stream to complete (and its memory to be visible) before touching global
// memory, and lets the next grid start launching early; when a kernel was not
// launched as a dependent, the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// L2 prefetch (ARGR_PLAN_PREFETCH). A kernel may issue it before its
// dependency wait: a prefetch moves lines of HBM into L2, which is where this
// GPU keeps global memory coherent, so it changes no value a later load sees
// (a line the previous grid writes is read as written). When the CTA is
// resident while the previous grid still runs, its input streams from HBM
// into L2 during that grid instead of after it.
constexpr uintptr_t kPrefetchMinPiece = 4096;         // bytes per bulk prefetch, at least
constexpr uintptr_t kPrefetchMaxBytes = 128 * 1024;   // bytes one CTA prefetches, at most
constexpr uintptr_t kPrefetchHeadBytes = 16 * 1024;   // the same under ARGR_PLAN_PREFETCH_HEAD

// One bulk prefetch of n bytes at p; p 16-byte aligned, n a positive multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(uintptr_t p, unsigned n) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
}

// Prefetch the bytes [lo, hi) of global memory, shrunk to 16-byte boundaries
// and to the first max_bytes: pieces of at least kPrefetchMinPiece bytes, one
// per warp of the CTA, each issued by the warp's lane 0.
__device__ __forceinline__ void prefetch_l2_range(const void* lo, const void* hi,
                                                  uintptr_t max_bytes = kPrefetchMaxBytes) {
    const uintptr_t a = (reinterpret_cast<uintptr_t>(lo) + 15) & ~static_cast<uintptr_t>(15);
    uintptr_t b = reinterpret_cast<uintptr_t>(hi) & ~static_cast<uintptr_t>(15);
    if ((threadIdx.x & 31) != 0 || b <= a) return;
    if (b - a > max_bytes) b = a + max_bytes;
    const uintptr_t nw = (blockDim.x + 31) >> 5;
    uintptr_t piece = ((b - a + nw - 1) / nw + 15) & ~static_cast<uintptr_t>(15);
    if (piece < kPrefetchMinPiece) piece = kPrefetchMinPiece;
    const uintptr_t s = a + (threadIdx.x >> 5) * piece;  // one piece per warp covers [a, b)
    if (s < b) prefetch_l2_bulk(s, static_cast<unsigned>(b - s < piece ? b - s : piece));
}

// Merge of two candidates: better key wins; equal keys keep the lower index
// (the higher index for the last-occurrence ops).
template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> merge(Cand<Tag> a, Cand<Tag> b) {
    const bool tie_to_b = kIsLast<OP> ? b.i > a.i : b.i < a.i;
    const bool take_b = Tag::template better<OP>(b.k, a.k) || (b.k == a.k && tie_to_b);
    return take_b ? b : a;
}

// ---------------------------------------------------------------------------
// Shuffles of raw values (16-bit values travel in a 32-bit register).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float shfl_xor_raw(unsigned m, float v, int o, int w) {
    return __shfl_xor_sync(m, v, o, w);
}
__device__ __forceinline__ unsigned long long shfl_xor_raw(unsigned m, unsigned long long v, int o, int w) {
    return __shfl_xor_sync(m, v, o, w);
}
__device__ __forceinline__ uint16_t shfl_xor_raw(unsigned m, uint16_t v, int o, int w) {
    return static_cast<uint16_t>(__shfl_xor_sync(m, static_cast<unsigned>(v), o, w));
}
__device__ __forceinline__ float shfl_raw(unsigned m, float v, int src, int w) {
    return __shfl_sync(m, v, src, w);
}
__device__ __forceinline__ unsigned long long shfl_raw(unsigned m, unsigned long long v, int src, int w) {
    return __shfl_sync(m, v, src, w);
}
__device__ __forceinline__ uint16_t shfl_raw(unsigned m, uint16_t v, int src, int w) {
    return static_cast<uint16_t>(__shfl_sync(m, static_cast<unsigned>(v), src, w));
}

// Butterfly over groups of G lanes (G a power of two <= 32); every lane of
// the group ends with the group's merged candidate.
// Merge of the candidates of a group of lanes (`mask`) through the warp
// reduction unit. Keys map to unsigned integers with the same order: a
// binary32 key through its bits (-0.0 first becomes +0.0 by adding +0.0, so
// both zeros map alike), a binary64 key is one already and is reduced high
// word first, then low word among the lanes that hold the best high word.
// Then the lowest index holding the best key is found (the highest, for the
// last-occurrence ops), and the value comes from a lane with that index (lanes
// with the same index hold the same element). When x[0] is NaN every
// candidate is (x[0], 0), so all keys map alike there too. Every lane of the
// group gets the result; all of them must take part.
template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> group_merge_redux(const Cand<Tag>& c, unsigned mask) {
    bool has;
    if constexpr (sizeof(typename Tag::key) == 4) {
        const unsigned b = __float_as_uint(c.k + 0.0f);
        unsigned u = b ^ (static_cast<unsigned>(static_cast<int>(b) >> 31) | 0x80000000u);
        if constexpr (kIsMin<OP>) u = ~u;
        has = u == __reduce_max_sync(mask, u);
    } else {
        const unsigned hi = static_cast<unsigned>(c.k >> 32), lo = static_cast<unsigned>(c.k);
        const bool top = hi == __reduce_max_sync(mask, hi);
        // every lane of the group must execute each reduction: none may sit
        // behind a short-circuit operator
        const unsigned best_lo = __reduce_max_sync(mask, top ? lo : 0u);
        has = top && lo == best_lo;
    }
    int win;
    if constexpr (kIsLast<OP>)
        win = static_cast<int>(__reduce_max_sync(mask, has ? static_cast<unsigned>(c.i) + 1u : 0u)) - 1;
    else
        win = static_cast<int>(__reduce_min_sync(mask, has ? static_cast<unsigned>(c.i) : 0xffffffffu));
    const int src = __ffs(__ballot_sync(mask, c.i == win) & mask) - 1;
    Cand<Tag> r;
    r.v = shfl_raw(mask, c.v, src, 32);
    r.k = shfl_raw(mask, c.k, src, 32);
    r.i = win;
    return r;
}

template <class Tag, int OP, int G>
__device__ __forceinline__ Cand<Tag> group_merge(Cand<Tag> c, unsigned mask) {
    // Reductions for whole warps and for 16-lane groups of binary64 keys
    // (measured: below that the few shuffle rounds are faster; [4096,128]
    // f32, 8 lanes per row: 2.06 us with shuffles, 2.48 us with reductions).
    if constexpr (G == 32 || (G == 16 && sizeof(typename Tag::key) == 8)) {
        return group_merge_redux<Tag, OP>(c, mask);
    } else {
#pragma unroll
        for (int off = G / 2; off >= 1; off >>= 1) {
            const Cand<Tag> o =
                make_cand<Tag, OP>(shfl_xor_raw(mask, c.v, off, G), __shfl_xor_sync(mask, c.i, off, G));
            c = merge<Tag, OP>(c, o);
        }
        return c;
    }
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
__device__ __forceinline__ unsigned long long vec_elem<unsigned long long>(const uint4& v, int k) {
    return k == 0 ? (static_cast<unsigned long long>(v.y) << 32 | v.x)
                  : (static_cast<unsigned long long>(v.w) << 32 | v.z);
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

// ---------------------------------------------------------------------------
// Vector scanners: visit a thread's 16-byte vectors in increasing index order,
// starting from its candidate so far, then return the updated candidate. The
// generic scanner visits the elements one by one.
// ---------------------------------------------------------------------------
template <class Tag, int OP>
struct VecScanElems {
    Cand<Tag> c;
    __device__ __forceinline__ explicit VecScanElems(const Cand<Tag>& c0) : c(c0) {}
    __device__ __forceinline__ void visit(const uint4& v, int j0) { visit_vec<Tag, OP>(c, v, j0); }
    __device__ __forceinline__ Cand<Tag> finish() const { return c; }
};
template <class Tag, int OP, bool PAIRED = (sizeof(typename Tag::raw) == 2)>
struct VecScan : VecScanElems<Tag, OP> {
    using VecScanElems<Tag, OP>::VecScanElems;
};

// binary32: the key is the value itself, so only (key, index) is carried.
template <int OP>
struct VecScan<TagF32, OP, false> {
    float k;
    int i;
    __device__ __forceinline__ explicit VecScan(const Cand<TagF32>& c) : k(c.k), i(c.i) {}
    __device__ __forceinline__ void el(float x, int j) {
        bool take;  // "better or equal" is one IEEE comparison (false on NaN)
        if constexpr (kIsLast<OP>) take = kIsMin<OP> ? x <= k : x >= k;
        else take = TagF32::better<OP>(x, k);
        if (take) {
            k = x;
            i = j;
        }
    }
    __device__ __forceinline__ void visit(const uint4& v, int j0) {
        el(__uint_as_float(v.x), j0);
        el(__uint_as_float(v.y), j0 + 1);
        el(__uint_as_float(v.z), j0 + 2);
        el(__uint_as_float(v.w), j0 + 3);
    }
    __device__ __forceinline__ Cand<TagF32> finish() const { return Cand<TagF32>{k, k, i}; }
};

// binary64: only (key, index) is carried and the value is rebuilt from the
// key at the end (order_key() is invertible on the numbers, except that both
// zeros share a key: cand_value() reads zeros back). An unchanged candidate is
// returned as it came, which keeps a NaN x[0] exact.
template <int OP>
struct VecScan<TagF64, OP, false> {
    unsigned long long k;
    int i;
    Cand<TagF64> c0;
    __device__ __forceinline__ explicit VecScan(const Cand<TagF64>& c) : k(c.k), i(c.i), c0(c) {}
    __device__ __forceinline__ void el(unsigned long long x, int j) {
        const unsigned long long kx = TagF64::order_key<OP>(x);
        if (kx <= TagF64::kLimit && (kIsLast<OP> ? kx >= k : kx > k)) {
            k = kx;
            i = j;
        }
    }
    __device__ __forceinline__ void visit(const uint4& v, int j0) {
        el(static_cast<unsigned long long>(v.y) << 32 | v.x, j0);
        el(static_cast<unsigned long long>(v.w) << 32 | v.z, j0 + 1);
    }
    __device__ __forceinline__ Cand<TagF64> finish() const {
        if (k == c0.k && i == c0.i) return c0;
        // inverse of order_key: keys with the sign bit set are b | kSign,
        // the others -b; ArgMin flips the sign bit back
        unsigned long long b = (k & TagF64::kSign) ? (k ^ TagF64::kSign) : (0ull - k);
        if constexpr (kIsMin<OP>) b ^= TagF64::kSign;
        return Cand<TagF64>{b, k, i};
    }
};

// One packed step over a 32-bit word w of two 16-bit elements against the
// packed keys kv of two candidates (low half against low half): a packed
// comparison (setp on the pair, false on NaN) decides each candidate's update,
// which sets its index to j (ia: low, ib: high), and a packed max / min
// (which ignores NaNs) updates the keys.
template <class Tag, int OP>
__device__ __forceinline__ void pair_step(uint32_t& kv, int& ia, int& ib, uint32_t w, int j) {
#define ARGR_PAIR_SEL(CMP, TY)                                                                   \
    asm("{\n\t.reg .pred p, q;\n\tsetp." CMP "." TY " p|q, %2, %3;\n\t"                        \
        "selp.b32 %0, %4, %0, p;\n\tselp.b32 %1, %4, %1, q;\n\t}"                              \
        : "+r"(ia), "+r"(ib)                                                                      \
        : "r"(w), "r"(kv), "r"(j))
    if constexpr (std::is_same<Tag, TagBF16>::value) {
        if constexpr (OP == kOpMax) ARGR_PAIR_SEL("gt", "bf16x2");
        else if constexpr (OP == kOpMin) ARGR_PAIR_SEL("lt", "bf16x2");
        else if constexpr (OP == kOpMaxLast) ARGR_PAIR_SEL("ge", "bf16x2");
        else ARGR_PAIR_SEL("le", "bf16x2");
        if constexpr (kIsMin<OP>) asm("min.bf16x2 %0, %0, %1;" : "+r"(kv) : "r"(w));
        else asm("max.bf16x2 %0, %0, %1;" : "+r"(kv) : "r"(w));
    } else {
        if constexpr (OP == kOpMax) ARGR_PAIR_SEL("gt", "f16x2");
        else if constexpr (OP == kOpMin) ARGR_PAIR_SEL("lt", "f16x2");
        else if constexpr (OP == kOpMaxLast) ARGR_PAIR_SEL("ge", "f16x2");
        else ARGR_PAIR_SEL("le", "f16x2");
        if constexpr (kIsMin<OP>) asm("min.f16x2 %0, %0, %1;" : "+r"(kv) : "r"(w));
        else asm("max.f16x2 %0, %0, %1;" : "+r"(kv) : "r"(w));
    }
#undef ARGR_PAIR_SEL
}

// 16-bit elements come two to a 32-bit word: the elements at even and at odd
// positions of the vectors a thread visits form two subsequences, each
// scanned by the exact sequential rule against its own candidate, both
// seeded with the thread's candidate so far. Per word, one packed comparison
// (setp on the 16-bit pair, false on NaN) gives each subsequence's update
// predicate, two selects update the indices, and one packed max / min (which
// ignores NaNs) the keys. The two candidates then merge by the usual rule;
// each is the best of {seed} and its subsequence with ties to the earlier
// (later) index, so the merge is that of the whole sequence. The kept key is
// the winning element itself except that a zero may carry the other sign
// (packed max / min of equal zeros); cand_value() reads zeros back. A NaN
// candidate (only x[0] can be one) is never displaced, so it skips the scan.
template <class Tag, int OP>
struct VecScan<Tag, OP, true> {
    uint32_t kv;    // keys of the two candidates as raw 16-bit patterns (low half: even positions)
    int ie, io;     // index of the even candidate; index - 1 of the odd one
    Cand<Tag> c0;
    bool frozen;
    __device__ __forceinline__ explicit VecScan(const Cand<Tag>& c)
        : kv(static_cast<uint32_t>(c.v) * 0x10001u), ie(c.i), io(c.i - 1), c0(c), frozen(c.k != c.k) {}
    // element j (low half) may take the even candidate, element j + 1 the odd one
    __device__ __forceinline__ void word(uint32_t w, int j) { pair_step<Tag, OP>(kv, ie, io, w, j); }
    __device__ __forceinline__ void visit(const uint4& v, int j0) {
        if (frozen) return;
        word(v.x, j0);
        word(v.y, j0 + 2);
        word(v.z, j0 + 4);
        word(v.w, j0 + 6);
    }
    __device__ __forceinline__ Cand<Tag> finish() const {
        if (frozen) return c0;
        const Cand<Tag> a = make_cand<Tag, OP>(static_cast<uint16_t>(kv & 0xffffu), ie);
        const Cand<Tag> b = make_cand<Tag, OP>(static_cast<uint16_t>(kv >> 16), io + 1);
        return merge<Tag, OP>(a, b);
    }
};

// The raw bits of a candidate's element for out_val. The 16-bit and binary64
// vector scans may hold a zero of the other sign, so a zero is read back from
// the row.
template <class Tag>
__device__ __forceinline__ typename Tag::raw cand_value(const Cand<Tag>& c, const typename Tag::raw* row) {
    if constexpr (sizeof(typename Tag::raw) == 2) {
        if ((c.v & 0x7fffu) == 0) return ld_scalar(row + c.i);
    } else if constexpr (sizeof(typename Tag::raw) == 8) {
        if ((c.v & ~TagF64::kSign) == 0) return ld_scalar(row + c.i);
    }
    return c.v;
}

}  // namespace argr
