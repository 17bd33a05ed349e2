// cummax / cummin with indices along the last axis (argreduce_cum).
//
// For every row and position j the output is the row's ArgMax (ArgMin) over
// x[0..j] under the same rules as argreduce(): seed (x[0], 0), a later element
// replaces the candidate only when strictly better, so ties keep the earlier
// index and a NaN after x[0] is never chosen (Paddle issue #79670, "Possible
// fixes": a scan with argmax semantics whose ties take the earlier index).
//
// The combine of an earlier prefix a and a later part b is "b if b.key >
// a.key, else a" (keys below): associative, so any scan tree reproduces the
// sequential scan.
//
// Decomposition: a row is one CTA's, or is cut into C contiguous chunks, one
// CTA each: a thread-block cluster (C <= 16) or a split scan (any C). Phase A
// (C > 1): every CTA reduces its chunk to an aggregate and hands it to the
// later chunks (distributed shared memory in a cluster, records in scratch
// for the split scan); each CTA folds the aggregates before its chunk into
// its carry-in. Phase B: the CTA scans its chunk tile by tile (NT threads x
// ITEMS elements; tiles loaded and stored through shared memory so that
// global accesses are coalesced, ITEMS odd so that a thread's run of
// consecutive elements spreads over the banks), carrying the running prefix.
// A chunk whose carry-in is at least as good as its aggregate is only filled
// with the carry (no second read), and within a scanned chunk a tile with no
// element better than the carry is filled the same way (elements of up to 4
// bytes). Split-scan chunks of four tiles or more read phase A with 16-byte
// loads; shorter ones keep their first tile in registers for phase B.
#pragma once

#include "device_common.cuh"
#include "internal.h"

namespace argr {

// Comparison keys for the scan: "b replaces a" is b.k > a.k for both ops.
// Floating types of up to 4 bytes compare as binary32 values, negated for
// the min op: an IEEE comparison is false on NaN, so a NaN element never
// replaces anything and a NaN seed (x[0]) is never replaced, and -0.0 equals
// +0.0. The identity (an empty prefix) is the lowest key, -inf: an element
// enters a prefix only when its key is strictly greater, so a prefix whose
// key is -inf is the identity, never an element, while the seed enters
// without that test and is always a real element. binary64 uses ordered
// 64-bit integer keys (GB300's FP64 pipe is too slow to compare at memory
// speed) and the integers their order as unsigned keys; there the identity
// is key 0 and the same argument holds.
struct CumF32 {
    using raw = float;
    using key = float;
    template <int OP> static __device__ __forceinline__ float elem_key(float v) { return kIsMin<OP> ? -v : v; }
    template <int OP> static __device__ __forceinline__ float seed_key(float v) { return elem_key<OP>(v); }
    static __device__ __forceinline__ float identity() { return __int_as_float(0xff800000); }
    static __device__ __forceinline__ unsigned long long to_bits(float k) { return __float_as_uint(k); }
    static __device__ __forceinline__ float from_bits(unsigned long long b) {
        return __uint_as_float(static_cast<unsigned>(b));
    }
};
template <bool BF16>
struct Cum16 {
    using raw = uint16_t;
    using key = float;
    static __device__ __forceinline__ float widen(uint16_t v) {
        if constexpr (BF16) return __uint_as_float(static_cast<unsigned>(v) << 16);
        return __half2float(__ushort_as_half(v));
    }
    template <int OP> static __device__ __forceinline__ float elem_key(uint16_t v) {
        return kIsMin<OP> ? -widen(v) : widen(v);
    }
    template <int OP> static __device__ __forceinline__ float seed_key(uint16_t v) { return elem_key<OP>(v); }
    static __device__ __forceinline__ float identity() { return __int_as_float(0xff800000); }
    static __device__ __forceinline__ unsigned long long to_bits(float k) { return __float_as_uint(k); }
    static __device__ __forceinline__ float from_bits(unsigned long long b) {
        return __uint_as_float(static_cast<unsigned>(b));
    }
};
using CumF16 = Cum16<false>;
using CumBF16 = Cum16<true>;
struct CumF64 {
    using raw = unsigned long long;  // binary64 bit patterns
    using key = unsigned long long;
    template <int OP> static __device__ __forceinline__ unsigned long long elem_key(unsigned long long b) {
        return TagF64::elem_key<OP>(b);
    }
    template <int OP> static __device__ __forceinline__ unsigned long long seed_key(unsigned long long b) {
        return TagF64::seed_key<OP>(b);
    }
    static __device__ __forceinline__ unsigned long long identity() { return 0ull; }
    static __device__ __forceinline__ unsigned long long to_bits(unsigned long long k) { return k; }
    static __device__ __forceinline__ unsigned long long from_bits(unsigned long long b) { return b; }
};
template <typename I, typename U>
struct CumInt {
    using raw = I;
    using key = U;
    // Two's complement to an unsigned order: flip the sign bit (ArgMax),
    // then complement (ArgMin). No NaN: every element has a real key.
    template <int OP> static __device__ __forceinline__ U elem_key(I v) {
        const U u = static_cast<U>(v) ^ (static_cast<U>(1) << (8 * sizeof(U) - 1));
        return kIsMin<OP> ? static_cast<U>(~u) : u;
    }
    template <int OP> static __device__ __forceinline__ U seed_key(I v) { return elem_key<OP>(v); }
    static __device__ __forceinline__ U identity() { return 0; }
    static __device__ __forceinline__ unsigned long long to_bits(U k) { return k; }
    static __device__ __forceinline__ U from_bits(unsigned long long b) { return static_cast<U>(b); }
};
using CumI32 = CumInt<int, unsigned>;
using CumI64 = CumInt<long long, unsigned long long>;

// A prefix result: ordered key and index. Values are not carried through the
// scan: the value of an index inside the current tile is read back from the
// tile in shared memory, and the carry-in keeps its own value.
template <class CT>
struct KI {
    typename CT::key k;
    int i;
};

// The later part b replaces the earlier prefix a only when strictly better.
template <class CT>
__device__ __forceinline__ KI<CT> later(const KI<CT>& a, const KI<CT>& b) {
    return b.k > a.k ? b : a;
}

template <class CT>
__device__ __forceinline__ KI<CT> ki_identity() {
    KI<CT> p;
    p.k = CT::identity();
    p.i = 0;
    return p;
}

template <typename T>
__device__ __forceinline__ T shfl_up_any(T v, int d) {
    if constexpr (sizeof(T) == 8) {
        unsigned long long u;
        memcpy(&u, &v, 8);
        u = __shfl_up_sync(0xffffffffu, u, d);
        memcpy(&v, &u, 8);
        return v;
    } else if constexpr (sizeof(T) == 4) {
        unsigned u;
        memcpy(&u, &v, 4);
        u = __shfl_up_sync(0xffffffffu, u, d);
        memcpy(&v, &u, 4);
        return v;
    } else {
        unsigned u = 0;
        memcpy(&u, &v, sizeof(T));
        u = __shfl_up_sync(0xffffffffu, u, d);
        memcpy(&v, &u, sizeof(T));
        return v;
    }
}

template <typename T>
__device__ __forceinline__ T shfl_xor_any(T v, int d) {
    if constexpr (sizeof(T) == 8) {
        unsigned long long u;
        memcpy(&u, &v, 8);
        u = __shfl_xor_sync(0xffffffffu, u, d);
        memcpy(&v, &u, 8);
        return v;
    } else {
        unsigned u = 0;
        memcpy(&u, &v, sizeof(T));
        u = __shfl_xor_sync(0xffffffffu, u, d);
        memcpy(&v, &u, sizeof(T));
        return v;
    }
}

template <class CT>
__device__ __forceinline__ KI<CT> shfl_up_ki(const KI<CT>& p, int d) {
    KI<CT> q;
    q.k = shfl_up_any(p.k, d);
    q.i = __shfl_up_sync(0xffffffffu, p.i, d);
    return q;
}

template <class CT>
__device__ __forceinline__ KI<CT> shfl_xor_ki(const KI<CT>& p, int d) {
    KI<CT> q;
    q.k = shfl_xor_any(p.k, d);
    q.i = __shfl_xor_sync(0xffffffffu, p.i, d);
    return q;
}

constexpr int kCumMaxCluster = 16;
constexpr int kCumLoadsA = 4;  // independent loads in flight per thread in phase A (stashed chunks)
// 16-byte loads in flight per thread in the 16-byte phase A: 8 for 8-byte
// elements, 4 for smaller ones (their wider per-vector key loop would spill).
template <typename R>
constexpr int kCumLoadsVec = sizeof(R) == 8 ? 8 : 4;
constexpr int kCumVecTiles = 4;  // chunks of at least this many tiles use the 16-byte phase A

// Total order for merging aggregates of disjoint ranges: the higher key, then
// the lower index. Commutative, so the order in which partial aggregates meet
// does not matter. An empty aggregate is key 0 (it never beats a real prefix,
// whose key is at least the seed's and whose index is lower on a tie).
template <class CT>
__device__ __forceinline__ KI<CT> first_best(const KI<CT>& a, const KI<CT>& b) {
    return (b.k > a.k || (b.k == a.k && b.i < a.i)) ? b : a;
}

template <class CT>
__device__ __forceinline__ KI<CT> warp_first_best(KI<CT> a) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = first_best(a, shfl_xor_ki(a, off));
    return a;
}

// first_best over the CTA; the result is valid in every thread of warp 0.
// Ends with warp_tot free for reuse only after the caller's next barrier.
template <class CT>
__device__ __forceinline__ KI<CT> block_first_best(KI<CT> a, KI<CT>* warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    a = warp_first_best(a);
    if (lane == 0) warp_tot[warp] = a;
    __syncthreads();
    if (warp == 0) a = warp_first_best(lane < nwarps ? warp_tot[lane] : ki_identity<CT>());
    return a;
}

// L2 residency for the split scan's second read of its chunk: phase A loads
// the chunk with an evict-last policy, and every scan writes its outputs as
// streaming stores (st.global.cs: evict-first), so that the outputs, twice to
// three times the input's bytes, do not push the chunk out of L2 before
// phase B reads it again.
__device__ __forceinline__ unsigned long long l2_evict_last_policy() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <typename R>
__device__ __forceinline__ R ld_keep(const R* p, unsigned long long pol) {
    R r;
    if constexpr (sizeof(R) == 8) {
        unsigned long long v;
        asm volatile("ld.global.nc.L2::cache_hint.b64 %0, [%1], %2;" : "=l"(v) : "l"(p), "l"(pol));
        __builtin_memcpy(&r, &v, 8);
    } else if constexpr (sizeof(R) == 4) {
        unsigned v;
        asm volatile("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
        __builtin_memcpy(&r, &v, 4);
    } else {
        unsigned short v;
        asm volatile("ld.global.nc.L2::cache_hint.b16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
        __builtin_memcpy(&r, &v, 2);
    }
    return r;
}

// A 16-byte load under the evict-last policy.
__device__ __forceinline__ uint4 ld_keep16(const void* p, unsigned long long pol) {
    uint4 r;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// Element k of a 16-byte vector of raw elements.
template <typename R>
__device__ __forceinline__ R vec_item(const uint4& v, int k) {
    R e;
    __builtin_memcpy(&e, reinterpret_cast<const char*>(&v) + k * sizeof(R), sizeof(R));
    return e;
}

// An element load: with KEEP, under the evict-last policy.
template <bool KEEP, typename R>
__device__ __forceinline__ R ld_elem(const R* p, unsigned long long pol) {
    if constexpr (KEEP) return ld_keep(p, pol);
    else return ld_scalar(p);
}

// The first tile of row[cb, ce) into registers, in the layout the scan uses
// (thread t holds elements cb + t + q * NT); phase A reduces it and phase B
// scans it without loading it again.
template <class CT, int ITEMS, bool KEEP = false>
__device__ __forceinline__ void load_first_tile(const typename CT::raw* row, int cb, int ce,
                                                typename CT::raw (&v)[ITEMS]) {
    const int nt = blockDim.x;
    const int n = ce - cb < nt * ITEMS ? ce - cb : nt * ITEMS;
    const unsigned long long pol = KEEP ? l2_evict_last_policy() : 0ull;
#pragma unroll
    for (int q = 0; q < ITEMS; ++q)
        if (static_cast<int>(threadIdx.x) + q * nt < n) v[q] = ld_elem<KEEP>(row + cb + threadIdx.x + q * nt, pol);
}

// Phase A: the aggregate of row[cb, ce) (its first best element): the first
// tile from v, the rest with kCumLoadsA independent loads in flight per
// thread. Valid in warp 0.
template <class CT, int OP, int ITEMS, bool KEEP = false>
__device__ __forceinline__ KI<CT> chunk_aggregate(const typename CT::raw* row, int cb, int ce,
                                                  const typename CT::raw (&v)[ITEMS], KI<CT>* warp_tot) {
    const unsigned long long pol = KEEP ? l2_evict_last_policy() : 0ull;
    using R = typename CT::raw;
    using K = typename CT::key;
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    const int tile = nt * ITEMS;
    const int n0 = ce - cb < tile ? ce - cb : tile;
    KI<CT> a = ki_identity<CT>();
#pragma unroll
    for (int q = 0; q < ITEMS; ++q) {  // increasing indices within the thread: the first best stays
        if (t + q * nt < n0) {
            const K k = CT::template elem_key<OP>(v[q]);
            if (k > a.k) {
                a.k = k;
                a.i = cb + t + q * nt;
            }
        }
    }
    for (int64_t j0 = static_cast<int64_t>(cb) + n0 + t; j0 < ce; j0 += static_cast<int64_t>(kCumLoadsA) * nt) {
        R w[kCumLoadsA];
#pragma unroll
        for (int u = 0; u < kCumLoadsA; ++u)
            if (j0 + u * nt < ce) w[u] = ld_elem<KEEP>(row + j0 + u * nt, pol);
#pragma unroll
        for (int u = 0; u < kCumLoadsA; ++u) {
            if (j0 + u * nt < ce) {
                const K k = CT::template elem_key<OP>(w[u]);
                if (k > a.k) {
                    a.k = k;
                    a.i = static_cast<int>(j0 + u * nt);
                }
            }
        }
    }
    return block_first_best(a, warp_tot);
}

// One tile of phase B: row[base, base + n) (n == NT * ITEMS when FULL, which
// drops the bounds tests). Unless STASHED (the tile is already in shared
// memory at tin), its elements are in v: they are stored to tin and the next
// tile (nn elements from nbase) is loaded into v while this one is scanned.
// Writes the outputs and moves the carry past the tile.
template <class CT, int OP, int ITEMS, bool FULL, bool STASHED>
__device__ __forceinline__ void scan_tile(const typename CT::raw* row, int base, int n, int nbase, int nn,
                                          KI<CT>& carry, typename CT::raw& carry_v, typename CT::raw (&v)[ITEMS],
                                          int64_t* __restrict__ oi_row, typename CT::raw* __restrict__ ov_row,
                                          typename CT::raw* tin, int* tidx, KI<CT>* warp_tot, KI<CT>* s_total) {
    using K = typename CT::key;
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = nt >> 5;
    if constexpr (!STASHED) {
#pragma unroll
        for (int q = 0; q < ITEMS; ++q)
            if (FULL || t + q * nt < n) tin[t + q * nt] = v[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < ITEMS; ++q)
            if (t + q * nt < nn) v[q] = ld_scalar(row + nbase + t + q * nt);
    }
    // A tile with no element better than the carry (ties keep the carry's
    // earlier index): every output of the tile is the carry and the carry
    // stays; no scan is needed. One barrier decides it for the CTA, before
    // the prefixes below take their registers. Elements of 8 bytes skip the
    // test: the extra branch makes the 64-register kernels spill there.
    bool better = sizeof(typename CT::raw) > 4;
#pragma unroll
    for (int q = 0; q < ITEMS; ++q) {
        const int j = t * ITEMS + q;
        if (sizeof(typename CT::raw) <= 4 && (FULL || j < n)) better |= CT::template elem_key<OP>(tin[j]) > carry.k;
    }
    if (sizeof(typename CT::raw) <= 4 && !__syncthreads_or(better)) {
        const long long ci = carry.i;
        long long* oi = reinterpret_cast<long long*>(oi_row + base);
#pragma unroll
        for (int q = 0; q < ITEMS; ++q)
            if (FULL || t + q * nt < n) __stcs(oi + t + q * nt, ci);
        if (ov_row) {
            typename CT::raw* ov = ov_row + base;
#pragma unroll
            for (int q = 0; q < ITEMS; ++q)
                if (FULL || t + q * nt < n) __stcs(ov + t + q * nt, carry_v);
        }
        __syncthreads();  // the tile buffers are reused by the next tile
        return;
    }
    // thread-local inclusive prefixes of ITEMS consecutive elements
    KI<CT> p[ITEMS];
    KI<CT> run = ki_identity<CT>();
#pragma unroll
    for (int q = 0; q < ITEMS; ++q) {
        const int j = t * ITEMS + q;
        if (FULL || j < n) {
            const K k = CT::template elem_key<OP>(tin[j]);
            if (k > run.k) {
                run.k = k;
                run.i = base + j;
            }
        }
        p[q] = run;
    }
    // warp inclusive scan of the thread totals
    KI<CT> ws = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const KI<CT> o = shfl_up_ki(ws, d);
        if (lane >= d) ws = later(o, ws);
    }
    KI<CT> excl = shfl_up_ki(ws, 1);
    if (lane == 0) excl = ki_identity<CT>();
    if (lane == 31) warp_tot[warp] = ws;
    __syncthreads();
    if (warp == 0) {
        KI<CT> w = lane < nwarps ? warp_tot[lane] : ki_identity<CT>();
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const KI<CT> o = shfl_up_ki(w, d);
            if (lane >= d) w = later(o, w);
        }
        KI<CT> we = shfl_up_ki(w, 1);
        if (lane == 0) we = ki_identity<CT>();
        if (lane < nwarps) warp_tot[lane] = we;  // exclusive prefix of each warp
        if (lane == nwarps - 1) *s_total = w;
    }
    __syncthreads();
    const KI<CT> before = later(later(carry, warp_tot[warp]), excl);
#pragma unroll
    for (int q = 0; q < ITEMS; ++q) {
        const int j = t * ITEMS + q;
        if (FULL || j < n) tidx[j] = later(before, p[q]).i;
    }
    const KI<CT> tot = *s_total;
    __syncthreads();
    // Coalesced stores. An index before this tile can only be the carry's.
    // Streaming (evict-first) stores: the outputs are not read again here.
    int64_t* oi = oi_row + base;
#pragma unroll
    for (int q = 0; q < ITEMS; ++q)
        if (FULL || t + q * nt < n)
            __stcs(reinterpret_cast<long long*>(oi + t + q * nt), static_cast<long long>(tidx[t + q * nt]));
    if (ov_row) {
        typename CT::raw* ov = ov_row + base;
#pragma unroll
        for (int q = 0; q < ITEMS; ++q) {
            if (FULL || t + q * nt < n) {
                const int i = tidx[t + q * nt];
                __stcs(ov + t + q * nt, i >= base ? tin[i - base] : carry_v);
            }
        }
    }
    if (tot.k > carry.k) {  // carry the tile's best past it
        carry = tot;
        carry_v = tin[tot.i - base];
    }
    __syncthreads();  // the tile buffers are reused by the next tile
}

// Phase A with 16-byte loads: the first best element of row[cb, ce) (best
// key, then lowest index), U vector loads in flight per thread under the
// evict-last policy (the chunk stays in L2 for a phase B that needs it); the
// part before the first 16-byte boundary and the part after the last one
// element by element. Every thread visits its elements in increasing index
// order (head, vectors, tail), so the strict comparison keeps its first best;
// the CTA merge breaks ties toward the lower index. Valid in warp 0.
template <class CT, int OP, int U>
__device__ __forceinline__ KI<CT> chunk_aggregate_vec(const typename CT::raw* row, int cb, int ce,
                                                      KI<CT>* warp_tot) {
    using R = typename CT::raw;
    using K = typename CT::key;
    constexpr int E = 16 / sizeof(R);
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    const int n = ce - cb;
    const R* base = row + cb;
    int head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(base) & 15u)) & 15u) / sizeof(R));
    if (head > n) head = n;
    const int nv = (n - head) / E;
    const int tail0 = head + nv * E;
    const uint4* vb = reinterpret_cast<const uint4*>(base + head);
    const unsigned long long pol = l2_evict_last_policy();
    KI<CT> a = ki_identity<CT>();
    if (t < head) {
        const K k = CT::template elem_key<OP>(ld_keep(base + t, pol));
        if (k > a.k) {
            a.k = k;
            a.i = cb + t;
        }
    }
    for (int v0 = t; v0 < nv; v0 += U * nt) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * nt < nv) buf[u] = ld_keep16(vb + v0 + u * nt, pol);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (v0 + u * nt < nv) {
                const int j0 = cb + head + (v0 + u * nt) * E;
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const K key = CT::template elem_key<OP>(vec_item<R>(buf[u], k));
                    if (key > a.k) {
                        a.k = key;
                        a.i = j0 + k;
                    }
                }
            }
        }
    }
    if (t < n - tail0) {
        const K k = CT::template elem_key<OP>(ld_keep(base + tail0 + t, pol));
        if (k > a.k) {
            a.k = k;
            a.i = cb + tail0 + t;
        }
    }
    return block_first_best(a, warp_tot);
}

// p[0, n) = val, as streaming stores: 16-byte stores between the first and
// the last 16-byte boundary, single elements before and after.
template <typename T>
__device__ __forceinline__ void fill_const(T* __restrict__ p, int n, T val) {
    constexpr int E = 16 / sizeof(T);
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    int head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / sizeof(T));
    if (head > n) head = n;
    const int nv = (n - head) / E;
    const int tail0 = head + nv * E;
    if (t < head) __stcs(p + t, val);
    uint4 pat;
#pragma unroll
    for (int k = 0; k < E; ++k) __builtin_memcpy(reinterpret_cast<char*>(&pat) + k * sizeof(T), &val, sizeof(T));
    uint4* pv = reinterpret_cast<uint4*>(p + head);
    for (int v = t; v < nv; v += nt) __stcs(pv + v, pat);
    if (t < n - tail0) __stcs(p + tail0 + t, val);
}

// Phase B of a dominated chunk: when the carry-in is at least as good as the
// chunk's best element (its phase-A aggregate; ties keep the carry, whose
// index is earlier), every prefix of the row that ends in the chunk has the
// carry as its result, so phase B writes (carry_i, carry_v) to every output
// of row[cb, ce) and neither reads nor scans the chunk again. In a long row
// only the chunks that hold a new best of the row so far are not dominated.
template <class CT>
__device__ __forceinline__ void fill_chunk(int cb, int ce, int carry_i, typename CT::raw carry_v,
                                           int64_t* __restrict__ oi_row, typename CT::raw* __restrict__ ov_row) {
    fill_const<long long>(reinterpret_cast<long long*>(oi_row + cb), ce - cb, static_cast<long long>(carry_i));
    if (ov_row) fill_const<typename CT::raw>(ov_row + cb, ce - cb, carry_v);
}

// Phase B: scan row[cb, ce) tile by tile (NT threads x ITEMS consecutive
// elements per thread), starting from the carry-in (carry, carry_v) = the
// prefix result just before cb, with the first tile already in v
// (load_first_tile). Tiles pass through shared memory so that global
// accesses are coalesced (ITEMS odd: a thread's run of consecutive elements
// spreads over the banks), and the next tile's loads are issued into
// registers while the current tile is scanned.
template <class CT, int OP, int ITEMS>
__device__ __forceinline__ void scan_chunk(const typename CT::raw* row, int cb, int ce, KI<CT> carry,
                                           typename CT::raw carry_v, typename CT::raw (&v)[ITEMS],
                                           int64_t* __restrict__ oi_row, typename CT::raw* __restrict__ ov_row,
                                           unsigned char* smem, KI<CT>* warp_tot, KI<CT>* s_total) {
    using R = typename CT::raw;
    const int tile = static_cast<int>(blockDim.x) * ITEMS;
    R* tin = reinterpret_cast<R*>(smem);                                                 // tile input
    int* tidx = reinterpret_cast<int*>(smem + static_cast<size_t>(tile) * sizeof(R));  // tile indices
    int base = cb;
    int n = ce - cb < tile ? ce - cb : tile;
    while (n > 0) {
        const int nbase = base + n;
        const int nn = ce - nbase < tile ? ce - nbase : tile;
        if (n == tile)
            scan_tile<CT, OP, ITEMS, true, false>(row, base, n, nbase, nn, carry, carry_v, v, oi_row, ov_row, tin,
                                                  tidx, warp_tot, s_total);
        else
            scan_tile<CT, OP, ITEMS, false, false>(row, base, n, nbase, nn, carry, carry_v, v, oi_row, ov_row, tin,
                                                   tidx, warp_tot, s_total);
        base = nbase;
        n = nn;
    }
}

// ---------------------------------------------------------------------------
// Stashed chunks (split scan with ARGR_PLAN_STASH): the CTA's whole chunk is
// copied into shared memory once, by 1-D bulk (TMA) copies of its 16-byte
// aligned middle plus plain loads of the ragged head and tail, and both phases
// read it there. The stash starts at the chunk's address modulo 16, so that
// the aligned middle lands on 16-byte aligned shared memory.
// ---------------------------------------------------------------------------
constexpr unsigned kStashPieceBytes = 16384;  // bulk copies in flight at once, up to 5 for 80 KiB

template <class CT>
__device__ __forceinline__ typename CT::raw* stash_fill(const typename CT::raw* row, int cb, int ce,
                                                       unsigned char* smem, unsigned long long* bar,
                                                       unsigned long long limit_ns, unsigned* err) {
    using R = typename CT::raw;
    constexpr int es = sizeof(R);
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(row + cb);
    const uintptr_t g1 = reinterpret_cast<uintptr_t>(row + ce);
    R* stash = reinterpret_cast<R*>(smem + (g0 & 15));
    const uintptr_t a0 = (g0 + 15) & ~static_cast<uintptr_t>(15);
    const uintptr_t a1 = g1 & ~static_cast<uintptr_t>(15);
    const bool bulk = a1 > a0;
    const int n = ce - cb;
    const int head = bulk ? static_cast<int>((a0 - g0) / es) : n;  // elements before the aligned middle
    const int tail = bulk ? static_cast<int>((a1 - g0) / es) : n;  // first element after it
    const unsigned barp = smem_u32(bar);
    if (t == 0 && bulk) {
        mbar_init(barp, 1);
        mbar_init_fence();
        const unsigned bytes = static_cast<unsigned>(a1 - a0);
        mbar_arrive_expect_tx(barp, bytes);
        const unsigned dst = smem_u32(stash) + static_cast<unsigned>(a0 - g0);
        for (unsigned off = 0; off < bytes; off += kStashPieceBytes) {
            const unsigned len = bytes - off < kStashPieceBytes ? bytes - off : kStashPieceBytes;
            bulk_copy_g2s(dst + off, reinterpret_cast<const void*>(a0 + off), len, barp);
        }
    }
    for (int j = t; j < head; j += nt) stash[j] = ld_scalar(row + cb + j);
    for (int j = tail + t; j < n; j += nt) stash[j] = ld_scalar(row + cb + j);
    __syncthreads();  // the barrier is initialised before anyone waits on it
    if (bulk && !mbar_wait_bounded(barp, 0, limit_ns)) {
        atomicOr(err, kErrWaitExpired);
        mbar_wait_bounded(barp, 0, limit_ns);  // let a late copy land before the CTA moves on
    }
    __syncthreads();
    return stash;
}

// Phase A on a stashed chunk: its first best element, valid in warp 0.
template <class CT, int OP>
__device__ __forceinline__ KI<CT> stash_aggregate(const typename CT::raw* stash, int cb, int ce, KI<CT>* warp_tot) {
    using K = typename CT::key;
    KI<CT> a = ki_identity<CT>();
    const int n = ce - cb;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {  // increasing indices within the thread
        const K k = CT::template elem_key<OP>(stash[j]);
        if (k > a.k) {
            a.k = k;
            a.i = cb + j;
        }
    }
    return block_first_best(a, warp_tot);
}

// Phase B on a stashed chunk: the tiles are windows of the stash.
template <class CT, int OP, int ITEMS>
__device__ __forceinline__ void scan_stash(const typename CT::raw* row, typename CT::raw* stash, int cb, int ce,
                                           KI<CT> carry, typename CT::raw carry_v, int64_t* __restrict__ oi_row,
                                           typename CT::raw* __restrict__ ov_row, int* tidx, KI<CT>* warp_tot,
                                           KI<CT>* s_total) {
    using R = typename CT::raw;
    const int tile = static_cast<int>(blockDim.x) * ITEMS;
    R unused[ITEMS];
    for (int base = cb; base < ce;) {
        const int n = ce - base < tile ? ce - base : tile;
        R* tin = stash + (base - cb);
        if (n == tile)
            scan_tile<CT, OP, ITEMS, true, true>(row, base, n, 0, 0, carry, carry_v, unused, oi_row, ov_row, tin,
                                                 tidx, warp_tot, s_total);
        else
            scan_tile<CT, OP, ITEMS, false, true>(row, base, n, 0, 0, carry, carry_v, unused, oi_row, ov_row, tin,
                                                  tidx, warp_tot, s_total);
        base += n;
    }
}

// One CTA per row (CLUSTER false: C = 1, the CTA loops over rows), or a
// cluster of C CTAs per row whose chunk aggregates are exchanged through
// distributed shared memory. Separate instantiations keep the cluster code out
// of the one-CTA kernel's registers.
template <class CT, int OP, int ITEMS, bool CLUSTER>
__global__ void __launch_bounds__(1024)
cum_kernel(const typename CT::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
           typename CT::raw* __restrict__ out_val) {
    using R = typename CT::raw;
    using K = typename CT::key;
    extern __shared__ __align__(16) unsigned char cum_smem[];
    __shared__ KI<CT> warp_tot[32];
    __shared__ KI<CT> s_total;
    __shared__ __align__(16) uint4 agg_slots[2][kCumMaxCluster];  // aggregates pushed by earlier CTAs
    __shared__ bool s_dominated;
    const int t = threadIdx.x;
    const int C = CLUSTER ? static_cast<int>(gridDim.x) : 1;
    const int b = CLUSTER ? static_cast<int>(blockIdx.x) : 0;
    bool started = false;
    if (CLUSTER) cluster_started_arrive();
    grid_dependency_wait();
    allow_dependents();
    int parity = 0;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y, parity ^= 1) {
        const R* row = x + r * static_cast<int64_t>(cols);
        const int cb = static_cast<int>(static_cast<int64_t>(cols) * b / C);
        const int ce = static_cast<int>(static_cast<int64_t>(cols) * (b + 1) / C);
        const R x0 = ld_scalar(row);
        R v[ITEMS];
        load_first_tile<CT, ITEMS>(row, cb, ce, v);
        KI<CT> carry;
        carry.k = CT::template seed_key<OP>(x0);
        carry.i = 0;
        R carry_v = x0;
        if constexpr (CLUSTER) {
            const KI<CT> a = chunk_aggregate<CT, OP, ITEMS>(row, cb, ce, v, warp_tot);
            if (!started) {  // every CTA of the cluster runs before the first remote write
                cluster_started_wait();
                started = true;
            }
            if (t < C - b - 1) {
                // Push this chunk's aggregate (key and index; the winner's raw
                // value is reloaded by whoever needs it) to the later CTA b + 1 + t.
                const uint64_t kk = CT::to_bits(a.k);
                unsigned remote;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                             : "=r"(remote)
                             : "r"(smem_addr(&agg_slots[parity][b])), "r"(b + 1 + t));
                asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote),
                             "r"(static_cast<uint32_t>(kk)), "r"(static_cast<uint32_t>(kk >> 32)),
                             "r"(static_cast<uint32_t>(a.i)), "r"(0u)
                             : "memory");
            }
            cluster_barrier();
            // Fold the aggregates of the earlier chunks, in order, into the carry.
            for (int k = 0; k < b; ++k) {
                const uint4 pk = agg_slots[parity][k];
                const K ek = CT::from_bits(static_cast<uint64_t>(pk.x) | (static_cast<uint64_t>(pk.y) << 32));
                if (ek > carry.k) {
                    carry.k = ek;
                    carry.i = static_cast<int>(pk.z);
                    carry_v = ld_scalar(row + carry.i);  // the winner's raw bits (an L2 hit)
                }
            }
            if (t == 0) s_dominated = !(a.k > carry.k);  // a is valid in warp 0
            __syncthreads();
            if (s_dominated) {
                fill_chunk<CT>(cb, ce, carry.i, carry_v, out_idx + r * static_cast<int64_t>(cols),
                               out_val ? out_val + r * static_cast<int64_t>(cols) : nullptr);
                __syncthreads();  // s_dominated is rewritten for the next row
                continue;
            }
        }
        scan_chunk<CT, OP, ITEMS>(row, cb, ce, carry, carry_v, v, out_idx + r * static_cast<int64_t>(cols),
                                  out_val ? out_val + r * static_cast<int64_t>(cols) : nullptr, cum_smem, warp_tot,
                                  &s_total);
    }
    if (CLUSTER && !started) cluster_started_wait();  // complete the start phase even with no rows
}

// ---------------------------------------------------------------------------
// Split scan: a row in `chunks` chunks, one CTA each, any number of CTAs.
//
// CTAs take tickets in the order they start (an atomic counter that wraps to
// zero after the last ticket); ticket k is chunk k % chunks of row k / chunks.
// After phase A a CTA publishes its chunk's aggregate as one 64-bit record:
// the low word is index + 1 (0 = not yet published, kNoElement = no element
// of the chunk has a nonzero key), the high word the key itself for keys of
// up to 32 bits (wider keys are recomputed from x[index]). It then waits for
// the records of the earlier chunks of its row, all of which belong to CTAs
// that took their tickets before it and so are running; their merge with the
// seed is its carry-in, and phase B follows. No CTA waits on a chain: every
// record is written straight after its CTA's phase A.
//
// Scratch (the argreduce scratch buffer; calls that share it must not run at
// the same time): a ticket and a done counter in the header, and the records
// in the region of argreduce's split counters, which must be all-zero between
// calls. The CTA whose wait finishes last zeroes the records once its own
// scan is done, so both regions are zero again when the kernel ends.
// Every wait is bounded: on expiry the CTA records kErrWaitExpired in the
// scratch error word, counts the missing record as empty and carries on (the
// outputs of that call are then undefined; the counters still wrap and the
// records are still cleared).
// ---------------------------------------------------------------------------
constexpr unsigned kNoElement = 0xffffffffu;
constexpr unsigned kErrBadScratch = 2u;  // a ticket or record out of range: scratch not prepared

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ unsigned inc_relaxed_gpu(unsigned* counter, unsigned wrap) {
    unsigned old;
    asm volatile("atom.relaxed.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(counter), "r"(wrap) : "memory");
    return old;
}

// Wait (bounded) until the record at p is published; an empty record on expiry.
__device__ __forceinline__ unsigned long long wait_record(const unsigned long long* p, unsigned long long limit_ns,
                                                          unsigned* err) {
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        const unsigned long long w = ld_acquire_gpu_u64(p);
        if (static_cast<unsigned>(w) != 0) return w;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrWaitExpired);
            return kNoElement;
        }
        __nanosleep(64);
    }
}

template <class CT>
__device__ __forceinline__ unsigned long long make_record(const KI<CT>& a) {
    if (a.k == CT::identity()) return kNoElement;
    const unsigned long long lo = static_cast<unsigned>(a.i) + 1u;
    if constexpr (sizeof(typename CT::key) <= 4) return (CT::to_bits(a.k) << 32) | lo;
    return lo;
}

// Wait (bounded) until chunk j publishes its inclusive prefix or its
// aggregate, and return whichever is there; an empty record on expiry.
__device__ __forceinline__ unsigned long long wait_either(const unsigned long long* incl,
                                                          const unsigned long long* agg,
                                                          unsigned long long limit_ns, unsigned* err) {
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        unsigned long long w = ld_acquire_gpu_u64(incl);
        if (static_cast<unsigned>(w) != 0) return w;
        w = ld_acquire_gpu_u64(agg);
        if (static_cast<unsigned>(w) != 0) return w;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrWaitExpired);
            return kNoElement;
        }
        __nanosleep(64);
    }
}

// A published record of row `row` as a prefix result (false: none, or not a
// record of this call, which is reported). Index 0 is the seed's: its key is
// the seed key (for a NaN x[0] that is not elem_key's).
template <class CT, int OP>
__device__ __forceinline__ bool decode_record(unsigned long long w, const typename CT::raw* row, int cols,
                                              const KI<CT>& seed, unsigned* err, KI<CT>* e) {
    const unsigned lo = static_cast<unsigned>(w);
    if (lo == 0 || lo == kNoElement) return false;
    if (lo - 1u >= static_cast<unsigned>(cols)) {  // not a record of this call
        atomicOr(err, kErrBadScratch);
        return false;
    }
    e->i = static_cast<int>(lo - 1u);
    if constexpr (sizeof(typename CT::key) <= 4) {
        e->k = CT::from_bits(w >> 32);
    } else {
        e->k = e->i == 0 ? seed.k : CT::template elem_key<OP>(ld_scalar(row + e->i));
    }
    return true;
}

// Split scan, LOOKBACK variant (decoupled look-back): every chunk publishes
// its aggregate and, once its carry-in is known, its inclusive prefix (chunk
// 0 only the latter). A CTA reads the records of the chunks before its own,
// one per thread, nearest first, down to the nearest inclusive prefix, so
// the work per CTA does not grow with the chunk count; merging an inclusive
// prefix with aggregates it already covers is harmless (first_best is
// idempotent). Records: [aggregate, inclusive] per chunk.
template <class CT, int OP, int ITEMS, bool STASH, bool LOOKBACK, bool VEC>
__global__ void __launch_bounds__(1024)
cum_split_kernel(const typename CT::raw* __restrict__ x, int64_t rows, int cols, int chunks,
                 int64_t* __restrict__ out_idx, typename CT::raw* __restrict__ out_val,
                 unsigned char* __restrict__ scratch, int test_expire) {
    using R = typename CT::raw;
    using K = typename CT::key;
    constexpr bool kKeyInRecord = sizeof(K) <= 4;
    extern __shared__ __align__(16) unsigned char cum_smem[];
    __shared__ KI<CT> warp_tot[32];
    __shared__ KI<CT> s_total;
    __shared__ unsigned s_flag;
    __shared__ bool s_dominated;
    __shared__ int s_near;
    __shared__ __align__(8) unsigned long long stash_bar;
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    const unsigned total = static_cast<unsigned>(rows) * static_cast<unsigned>(chunks);
    constexpr unsigned kWords = LOOKBACK ? 2u : 1u;  // record words per chunk
    unsigned* const err = reinterpret_cast<unsigned*>(scratch);
    unsigned* const ticket_ctr = reinterpret_cast<unsigned*>(scratch + kCumTicketOffset);
    unsigned* const done_ctr = reinterpret_cast<unsigned*>(scratch + kCumDoneOffset);
    unsigned long long* const records =
        reinterpret_cast<unsigned long long*>(scratch + cum_records_offset(static_cast<int64_t>(kWords) * total));
    const unsigned long long limit_ns = test_expire ? 2ull * 1000 * 1000 : kWaitLimitNs;

    grid_dependency_wait();  // the previous call's counters and records are settled
    if (t == 0) s_flag = arrive_acq_rel(ticket_ctr, total - 1);
    __syncthreads();
    allow_dependents();
    const unsigned ticket = s_flag;
    if (ticket >= total) {  // only with a scratch buffer that was never prepared
        if (t == 0) atomicOr(err, kErrBadScratch);
        return;
    }
    const int64_t r = ticket / static_cast<unsigned>(chunks);
    const int c = static_cast<int>(ticket % static_cast<unsigned>(chunks));
    const R* row = x + r * static_cast<int64_t>(cols);
    const int cb = static_cast<int>(static_cast<int64_t>(cols) * c / chunks);
    const int ce = static_cast<int>(static_cast<int64_t>(cols) * (c + 1) / chunks);
    const R x0 = ld_scalar(row);
    R v[ITEMS];
    R* stash = nullptr;
    KI<CT> a;
    if constexpr (STASH) {
        stash = stash_fill<CT>(row, cb, ce, cum_smem, &stash_bar, limit_ns, err);
        a = stash_aggregate<CT, OP>(stash, cb, ce, warp_tot);
    } else if constexpr (VEC) {
        a = chunk_aggregate_vec<CT, OP, kCumLoadsVec<R>>(row, cb, ce, warp_tot);
    } else {
        load_first_tile<CT, ITEMS, true>(row, cb, ce, v);
        a = chunk_aggregate<CT, OP, ITEMS, true>(row, cb, ce, v, warp_tot);
    }
    KI<CT> seed;
    seed.k = CT::template seed_key<OP>(x0);
    seed.i = 0;

    unsigned long long* const row_records = records + kWords * (r * chunks);
    KI<CT> acc = ki_identity<CT>();
    if constexpr (LOOKBACK) {
        // Publish: chunk 0 its inclusive prefix (seed and aggregate), the others
        // their aggregate (the test flag leaves chunk 0's record unset).
        if (t == 0 && !(test_expire && c == 0)) {
            if (c == 0)
                st_release_gpu_u64(row_records + 1, make_record(first_best(seed, a)));
            else
                st_release_gpu_u64(row_records + 2 * c, make_record(a));
        }
        // Look back in windows of one chunk per thread, nearest first.
        for (int j_hi = c - 1; j_hi >= 0; j_hi -= nt) {
            const int j = j_hi - t;
            unsigned long long w = 0;
            bool is_incl = false;
            if (j >= 0) {
                w = ld_acquire_gpu_u64(row_records + 2 * j + 1);
                is_incl = static_cast<unsigned>(w) != 0;
                if (!is_incl) w = ld_acquire_gpu_u64(row_records + 2 * j);
            }
            if (t == 0) s_near = nt;
            __syncthreads();
            if (is_incl) atomicMin(&s_near, t);
            __syncthreads();
            const int near = s_near;  // the nearest chunk with an inclusive prefix, if any in this window
            if (j >= 0 && t <= near) {
                if (static_cast<unsigned>(w) == 0)
                    w = wait_either(row_records + 2 * j + 1, row_records + 2 * j, limit_ns, err);
                KI<CT> e;
                if (decode_record<CT, OP>(w, row, cols, seed, err, &e)) acc = first_best(acc, e);
            }
            __syncthreads();  // s_near is rewritten by the next window
            if (near < nt) break;
        }
    } else {
    unsigned long long* const row_rec1 = row_records;
    // Publish (the test flag leaves chunk 0's record unset: every wait on it expires).
    if (t == 0 && !(test_expire && c == 0)) st_release_gpu_u64(row_rec1 + c, make_record(a));

    // Merge the records of chunks 0 .. c-1 (all loads first, then the waits).
    for (int j0 = t; j0 < c; j0 += 4 * nt) {
        unsigned long long w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = j0 + u * nt < c ? ld_acquire_gpu_u64(row_rec1 + j0 + u * nt) : kNoElement;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (static_cast<unsigned>(w[u]) == 0) w[u] = wait_record(row_rec1 + j0 + u * nt, limit_ns, err);
        R xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const unsigned lo = static_cast<unsigned>(w[u]);
            if (lo != kNoElement && lo - 1u >= static_cast<unsigned>(cols)) {  // not a record of this call
                atomicOr(err, kErrBadScratch);
                w[u] = kNoElement;
            }
            if (!kKeyInRecord && static_cast<unsigned>(w[u]) != kNoElement)
                xv[u] = ld_scalar(row + (static_cast<unsigned>(w[u]) - 1u));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const unsigned lo = static_cast<unsigned>(w[u]);
            if (lo != kNoElement) {
                KI<CT> e;
                if constexpr (kKeyInRecord) {
                    e.k = CT::from_bits(w[u] >> 32);
                } else {
                    e.k = CT::template elem_key<OP>(xv[u]);
                }
                e.i = static_cast<int>(lo - 1u);
                acc = first_best(acc, e);
            }
        }
    }
    }
    __syncthreads();  // warp_tot is free again (chunk_aggregate's readers are done)
    acc = block_first_best(acc, warp_tot);
    unsigned done_old = 0;
    if (t < 32) {
        acc = first_best(seed, acc);
        if (t == 0) {
            s_total = acc;
            s_dominated = !(a.k > acc.k);  // the carry-in is at least as good as the chunk's best
            // LOOKBACK: the inclusive prefix of this chunk, for the chunks after it.
            if (LOOKBACK && c > 0) st_release_gpu_u64(row_records + 2 * c + 1, make_record(first_best(acc, a)));
            // Every record this CTA needs has been read (the barrier above);
            // count it done. The result is only needed after the scan.
            fence_acq_rel_gpu();
            done_old = inc_relaxed_gpu(done_ctr, total - 1);
        }
    }
    __syncthreads();
    const KI<CT> carry = s_total;
    __syncthreads();  // s_total / warp_tot are reused by the scan
    const R carry_v = carry.i == 0 ? x0 : ld_scalar(row + carry.i);
    int64_t* const oi_row = out_idx + r * static_cast<int64_t>(cols);
    R* const ov_row = out_val ? out_val + r * static_cast<int64_t>(cols) : nullptr;
    if (s_dominated) {
        fill_chunk<CT>(cb, ce, carry.i, carry_v, oi_row, ov_row);
    } else if constexpr (STASH) {
        scan_stash<CT, OP, ITEMS>(row, stash, cb, ce, carry, carry_v, oi_row, ov_row,
                                  reinterpret_cast<int*>(cum_smem + kCumStashBytes + 16), warp_tot, &s_total);
    } else {
        if constexpr (VEC) load_first_tile<CT, ITEMS>(row, cb, ce, v);  // from L2: phase A kept the chunk there
        scan_chunk<CT, OP, ITEMS>(row, cb, ce, carry, carry_v, v, oi_row, ov_row, cum_smem, warp_tot, &s_total);
    }
    // The CTA that counted last clears the records of the whole launch.
    if (t == 0) {
        s_flag = done_old == total - 1 ? 1u : 0u;
        if (s_flag) fence_acq_rel_gpu();
    }
    __syncthreads();
    if (s_flag)
        for (unsigned j = t; j < kWords * total; j += nt) records[j] = 0ull;
}

// ---------------------------------------------------------------------------
// Streaming scan (ARGR_PATH_CUM_STREAM): a fixed grid of CTAs (about two per
// SM) takes tiles in ticket order, any number of tiles per CTA, each tile
// read once. For a tile the CTA scans it locally (identity-seeded), publishes
// the tile's total as its aggregate, looks back (decoupled look-back, as in
// the split scan's LOOKBACK variant) for its carry-in, publishes its inclusive
// prefix and writes its outputs; the next ticket's tile is being loaded into
// registers all the while. Tickets come from an atomic counter, so a tile
// only waits for tiles with earlier tickets, taken by CTAs that are running.
// Records: [aggregate, inclusive] per tile. The CTA that leaves last clears
// the records and the ticket counter.
// ---------------------------------------------------------------------------
template <class CT, int OP, int ITEMS>
__device__ __forceinline__ void stream_load(const typename CT::raw* x, int cols, int tiles_per_row, unsigned ticket,
                                            typename CT::raw (&v)[ITEMS]) {
    const int nt = blockDim.x;
    const int tile = nt * ITEMS;
    const int64_t r = ticket / static_cast<unsigned>(tiles_per_row);
    const int base = static_cast<int>(ticket % static_cast<unsigned>(tiles_per_row)) * tile;
    const int n = cols - base < tile ? cols - base : tile;
    const typename CT::raw* src = x + r * static_cast<int64_t>(cols) + base;
#pragma unroll
    for (int q = 0; q < ITEMS; ++q)
        if (static_cast<int>(threadIdx.x) + q * nt < n) v[q] = ld_scalar(src + threadIdx.x + q * nt);
}

template <class CT, int OP, int ITEMS>
__global__ void __launch_bounds__(1024)
cum_stream_kernel(const typename CT::raw* __restrict__ x, int64_t rows, int cols, int tiles_per_row,
                  int64_t* __restrict__ out_idx, typename CT::raw* __restrict__ out_val,
                  unsigned char* __restrict__ scratch, int test_expire) {
    using R = typename CT::raw;
    using K = typename CT::key;
    extern __shared__ __align__(16) unsigned char cum_smem[];
    __shared__ KI<CT> warp_tot[32];  // the local scan's warp prefixes
    __shared__ KI<CT> lb_tot[32];    // the look-back's reduction
    __shared__ KI<CT> s_total;
    __shared__ KI<CT> s_carry;
    __shared__ unsigned s_ticket;
    __shared__ int s_near;
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = nt >> 5;
    const int tile = nt * ITEMS;
    const unsigned total = static_cast<unsigned>(rows) * static_cast<unsigned>(tiles_per_row);
    unsigned* const err = reinterpret_cast<unsigned*>(scratch);
    unsigned* const ticket_ctr = reinterpret_cast<unsigned*>(scratch + kCumTicketOffset);
    unsigned* const done_ctr = reinterpret_cast<unsigned*>(scratch + kCumDoneOffset);
    unsigned long long* const records =
        reinterpret_cast<unsigned long long*>(scratch + cum_records_offset(2 * static_cast<int64_t>(total)));
    const unsigned long long limit_ns = test_expire ? 2ull * 1000 * 1000 : kWaitLimitNs;
    R* tin = reinterpret_cast<R*>(cum_smem);
    int* tidx = reinterpret_cast<int*>(cum_smem + static_cast<size_t>(tile) * sizeof(R));

    // Tickets are taken one tile ahead: a CTA holds `ticket` (being scanned)
    // and `next` (being loaded), and asks for the one after during the scan.
    grid_dependency_wait();  // the previous call's counters and records are settled
    if (t == 0) {
        s_ticket = atomicAdd(ticket_ctr, 1u);
        s_near = static_cast<int>(s_ticket < total ? atomicAdd(ticket_ctr, 1u) : total);
    }
    __syncthreads();
    allow_dependents();
    unsigned ticket = s_ticket;
    unsigned next = static_cast<unsigned>(s_near);
    // Each CTA takes at most two tickets past the last tile, so a first ticket
    // at or above total + 2 * grid comes from a scratch buffer never prepared.
    if (ticket >= total + 2 * gridDim.x) {
        if (t == 0) atomicOr(err, kErrBadScratch);
        return;
    }
    __syncthreads();  // s_near is reused by the look-back
    R v[ITEMS];
    if (ticket < total) stream_load<CT, OP, ITEMS>(x, cols, tiles_per_row, ticket, v);
    while (ticket < total) {
        const int64_t r = ticket / static_cast<unsigned>(tiles_per_row);
        const int j = static_cast<int>(ticket % static_cast<unsigned>(tiles_per_row));
        const int base = j * tile;
        const int n = cols - base < tile ? cols - base : tile;
        const R* row = x + r * static_cast<int64_t>(cols);
        unsigned long long* const row_records = records + 2 * (r * tiles_per_row);
#pragma unroll
        for (int q = 0; q < ITEMS; ++q)
            if (t + q * nt < n) tin[t + q * nt] = v[q];
        unsigned after = total;  // thread 0: the ticket after `next`, asked for now, read at the end
        if (t == 0 && next < total) after = atomicAdd(ticket_ctr, 1u);
        __syncthreads();
        if (next < total) stream_load<CT, OP, ITEMS>(x, cols, tiles_per_row, next, v);  // overlaps the rest

        // Local scan: thread prefixes, warp scan, warp totals; s_total = the tile's total.
        KI<CT> p[ITEMS];
        KI<CT> run = ki_identity<CT>();
#pragma unroll
        for (int q = 0; q < ITEMS; ++q) {
            const int jj = t * ITEMS + q;
            if (jj < n) {
                const K k = CT::template elem_key<OP>(tin[jj]);
                if (k > run.k) {
                    run.k = k;
                    run.i = base + jj;
                }
            }
            p[q] = run;
        }
        KI<CT> ws = run;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const KI<CT> o = shfl_up_ki(ws, d);
            if (lane >= d) ws = later(o, ws);
        }
        KI<CT> excl = shfl_up_ki(ws, 1);
        if (lane == 0) excl = ki_identity<CT>();
        if (lane == 31) warp_tot[warp] = ws;
        __syncthreads();
        if (warp == 0) {
            KI<CT> w = lane < nwarps ? warp_tot[lane] : ki_identity<CT>();
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const KI<CT> o = shfl_up_ki(w, d);
                if (lane >= d) w = later(o, w);
            }
            KI<CT> we = shfl_up_ki(w, 1);
            if (lane == 0) we = ki_identity<CT>();
            if (lane < nwarps) warp_tot[lane] = we;  // exclusive prefix of each warp
            if (lane == nwarps - 1) s_total = w;
        }
        __syncthreads();
        const KI<CT> agg = s_total;
        const R x0 = ld_scalar(row);
        KI<CT> seed;
        seed.k = CT::template seed_key<OP>(x0);
        seed.i = 0;

        // Carry-in: the seed for a row's first tile, else the look-back.
        KI<CT> acc = ki_identity<CT>();
        if (j == 0) {
            if (t == 0 && !test_expire) st_release_gpu_u64(row_records + 1, make_record(first_best(seed, agg)));
        } else {
            if (t == 0) st_release_gpu_u64(row_records + 2 * j, make_record(agg));
            for (int j_hi = j - 1; j_hi >= 0; j_hi -= nt) {
                const int jb = j_hi - t;
                unsigned long long w = 0;
                bool is_incl = false;
                if (jb >= 0) {
                    w = ld_acquire_gpu_u64(row_records + 2 * jb + 1);
                    is_incl = static_cast<unsigned>(w) != 0;
                    if (!is_incl) w = ld_acquire_gpu_u64(row_records + 2 * jb);
                }
                if (t == 0) s_near = nt;
                __syncthreads();
                if (is_incl) atomicMin(&s_near, t);
                __syncthreads();
                const int near = s_near;
                if (jb >= 0 && t <= near) {
                    if (static_cast<unsigned>(w) == 0)
                        w = wait_either(row_records + 2 * jb + 1, row_records + 2 * jb, limit_ns, err);
                    KI<CT> e;
                    if (decode_record<CT, OP>(w, row, cols, seed, err, &e)) acc = first_best(acc, e);
                }
                __syncthreads();  // s_near is rewritten by the next window
                if (near < nt) break;
            }
        }
        acc = block_first_best(acc, lb_tot);
        if (t == 0) {
            const KI<CT> carry = first_best(seed, acc);
            s_carry = carry;
            if (j > 0) st_release_gpu_u64(row_records + 2 * j + 1, make_record(first_best(carry, agg)));
        }
        __syncthreads();
        const KI<CT> carry = s_carry;
        const R carry_v = carry.i == 0 ? x0 : ld_scalar(row + carry.i);  // before the tile: an L2 hit

        // Outputs: the carry, the warp's exclusive prefix and the lane's, then the thread's own prefixes.
        const KI<CT> before = later(later(carry, warp_tot[warp]), excl);
#pragma unroll
        for (int q = 0; q < ITEMS; ++q) {
            const int jj = t * ITEMS + q;
            if (jj < n) tidx[jj] = later(before, p[q]).i;
        }
        __syncthreads();
        int64_t* oi = out_idx + r * static_cast<int64_t>(cols) + base;
#pragma unroll
        for (int q = 0; q < ITEMS; ++q)
            if (t + q * nt < n) oi[t + q * nt] = tidx[t + q * nt];
        if (out_val) {
            R* ov = out_val + r * static_cast<int64_t>(cols) + base;
#pragma unroll
            for (int q = 0; q < ITEMS; ++q) {
                if (t + q * nt < n) {
                    const int i = tidx[t + q * nt];
                    ov[t + q * nt] = i >= base ? tin[i - base] : carry_v;
                }
            }
        }
        if (t == 0) s_ticket = after;
        __syncthreads();  // tin, tidx, the shared totals are reused by the next tile
        ticket = next;
        next = s_ticket;
    }
    // The CTA that leaves last clears the records and resets the ticket counter.
    if (t == 0) {
        fence_acq_rel_gpu();
        const unsigned old = inc_relaxed_gpu(done_ctr, gridDim.x - 1);
        s_ticket = old == gridDim.x - 1 ? 1u : 0u;
        if (s_ticket) fence_acq_rel_gpu();
    }
    __syncthreads();
    if (s_ticket) {
        for (unsigned k = t; k < 2 * total; k += nt) records[k] = 0ull;
        if (t == 0) *ticket_ctr = 0u;
    }
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
constexpr int kCumItems = 7;

inline size_t cum_smem_bytes(int block, int es) { return static_cast<size_t>(block) * kCumItems * (es + 4); }

template <class CT, int OP, bool STASH, bool LOOKBACK, bool VEC>
cudaError_t launch_cum_split_s(const argr_plan& p, const Problem& pr) {
    using R = typename CT::raw;
    auto kern = cum_split_kernel<CT, OP, kCumItems, STASH, LOOKBACK, VEC>;
    // Stash: the chunk (16 bytes of slack for its alignment) and the tile indices.
    const size_t smem = STASH ? kCumStashBytes + 16 + static_cast<size_t>(p.block) * kCumItems * 4
                              : cum_smem_bytes(p.block, sizeof(R));
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(pr.rows * p.blocks_per_row));
    return launch_ex_smem(kern, grid, dim3(p.block), 1, smem, p, pr.stream, static_cast<const R*>(pr.x), pr.rows,
                          pr.cols, static_cast<int>(p.blocks_per_row), pr.out_idx, static_cast<R*>(pr.out_val),
                          static_cast<unsigned char*>(pr.scratch), (p.flags & ARGR_PLAN_TEST_EXPIRE) ? 1 : 0);
}

// Chunks of kCumVecTiles tiles or more take the 16-byte phase A (phase B, if
// needed, reloads its first tile from L2); shorter chunks keep their first
// tile in registers from phase A to phase B. Either variant is correct for any
// chunk length; the choice is only one of speed.
template <class CT, int OP>
cudaError_t launch_cum_split(const argr_plan& p, const Problem& pr) {
    if (p.flags & ARGR_PLAN_STASH) return launch_cum_split_s<CT, OP, true, false, false>(p, pr);
    const bool vec = pr.cols / p.blocks_per_row >= static_cast<int64_t>(kCumVecTiles) * p.block * kCumItems;
    if (p.flags & ARGR_PLAN_LOOKBACK)
        return vec ? launch_cum_split_s<CT, OP, false, true, true>(p, pr)
                   : launch_cum_split_s<CT, OP, false, true, false>(p, pr);
    return vec ? launch_cum_split_s<CT, OP, false, false, true>(p, pr)
               : launch_cum_split_s<CT, OP, false, false, false>(p, pr);
}

template <class CT, int OP>
cudaError_t launch_cum_stream(const argr_plan& p, const Problem& pr) {
    using R = typename CT::raw;
    auto kern = cum_stream_kernel<CT, OP, kCumItems>;
    const size_t smem = cum_smem_bytes(p.block, sizeof(R));
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    return launch_ex_smem(kern, dim3(static_cast<unsigned>(p.grid_rows)), dim3(p.block), 1, smem, p, pr.stream,
                          static_cast<const R*>(pr.x), pr.rows, pr.cols, static_cast<int>(p.blocks_per_row),
                          pr.out_idx, static_cast<R*>(pr.out_val), static_cast<unsigned char*>(pr.scratch),
                          (p.flags & ARGR_PLAN_TEST_EXPIRE) ? 1 : 0);
}

template <class CT, int OP>
cudaError_t launch_cum_op(const argr_plan& p, const Problem& pr) {
    using R = typename CT::raw;
    if (p.path == ARGR_PATH_CUM_SPLIT) return launch_cum_split<CT, OP>(p, pr);
    if (p.path == ARGR_PATH_CUM_STREAM) return launch_cum_stream<CT, OP>(p, pr);
    const size_t smem = cum_smem_bytes(p.block, sizeof(R));
    if (p.cluster <= 1) {
        auto kern1 = cum_kernel<CT, OP, kCumItems, false>;
        static KernelLaunchCache cache1;
        cudaError_t e = ensure_smem_limit(kern1, smem, cache1);
        if (e != cudaSuccess) return e;
        return launch_ex_smem(kern1, dim3(1, static_cast<unsigned>(p.grid_rows)), dim3(p.block), 1, smem, p,
                              pr.stream, static_cast<const R*>(pr.x), pr.rows, pr.cols, pr.out_idx,
                              static_cast<R*>(pr.out_val));
    }
    auto kern = cum_kernel<CT, OP, kCumItems, true>;
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    const int C = p.cluster;
    if (C > 8) {
        e = allow_big_cluster(kern, cache);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>(C), static_cast<unsigned>(p.grid_rows));
    bool ok = false;  // refuse a cluster shape the device cannot co-schedule
    e = cluster_fits(kern, grid, p.block, C, smem, cache, &ok);
    if (e != cudaSuccess) return e;
    if (!ok) return cudaErrorInvalidClusterSize;  // reported as ARGR_EUNSUPPORTED
    return launch_ex_smem(kern, grid, dim3(p.block), C, smem, p, pr.stream, static_cast<const R*>(pr.x), pr.rows,
                          pr.cols, pr.out_idx, static_cast<R*>(pr.out_val));
}

template <class CT>
cudaError_t launch_cum_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_cum_op<CT, kOpMax>(p, pr);
        case kOpMin: return launch_cum_op<CT, kOpMin>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace argr

#define ARGR_DEFINE_CUM_LAUNCHER(sfx, CT)                                                                    \
    namespace argr {                                                                                          \
    cudaError_t launch_cum_##sfx(const argr_plan& p, const Problem& pr) { return launch_cum_t<CT>(p, pr); }   \
    }
