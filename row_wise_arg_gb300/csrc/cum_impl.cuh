// cummax / cummin with indices along the last axis (argreduce_cum).
//
// For every row and position j the output is the row's ArgMax (ArgMin) over
// x[0..j] under the same rules as argreduce(): seed (x[0], 0), a later element
// replaces the candidate only when strictly better, so ties keep the earlier
// index and a NaN after x[0] is never chosen (Paddle issue #79670, "Possible
// fixes": a scan with argmax semantics whose ties take the earlier index).
//
// Comparisons use ordered integer keys: monotone in the value (reversed for
// the min op), +0.0 and -0.0 equal, NaN elements key 0 (never better than
// anything), a NaN x[0] the all-ones key (nothing is better, so every output
// stays (x[0], 0)). The combine of an earlier prefix a and a later part b is
// "b if b.key > a.key, else a": associative, so any scan tree reproduces the
// sequential scan, and key-0 elements act as its identity.
//
// Decomposition: a row is cut into C contiguous chunks, one CTA each (a
// thread-block cluster when C > 1). Phase A (C > 1): every CTA reduces its
// chunk to an aggregate and pushes it into the shared memory of every later
// CTA of the cluster; after one cluster barrier each CTA folds the aggregates
// before it into its carry-in. Phase B: the CTA scans its chunk tile by tile
// (NT threads x ITEMS elements; tiles loaded and stored through shared memory
// so that global accesses are coalesced, ITEMS odd so that a thread's run of
// consecutive elements spreads over the banks), carrying the running prefix.
#pragma once

#include "device_common.cuh"
#include "internal.h"

namespace argr {

// Ordered keys for the scan. Key type u32 for elements up to 4 bytes, u64 for 8.
struct CumF32 {
    using raw = float;
    using key = unsigned;
    template <int OP> static __device__ __forceinline__ unsigned ordered(unsigned b) {
        unsigned u = (b & 0x7fffffffu) == 0 ? 0x80000000u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
        return kIsMin<OP> ? ~u : u;
    }
    template <int OP> static __device__ __forceinline__ unsigned elem_key(float v) {
        const unsigned b = __float_as_uint(v);
        return (b & 0x7fffffffu) > 0x7f800000u ? 0u : ordered<OP>(b);
    }
    template <int OP> static __device__ __forceinline__ unsigned seed_key(float v) {
        const unsigned b = __float_as_uint(v);
        return (b & 0x7fffffffu) > 0x7f800000u ? ~0u : ordered<OP>(b);
    }
};
template <unsigned kInf>
struct Cum16 {
    using raw = uint16_t;
    using key = unsigned;
    template <int OP> static __device__ __forceinline__ unsigned ordered(unsigned b) {
        unsigned u = (b & 0x7fffu) == 0 ? 0x8000u : ((b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u));
        return kIsMin<OP> ? (~u & 0xffffu) : u;
    }
    template <int OP> static __device__ __forceinline__ unsigned elem_key(uint16_t v) {
        return (v & 0x7fffu) > kInf ? 0u : ordered<OP>(v);
    }
    template <int OP> static __device__ __forceinline__ unsigned seed_key(uint16_t v) {
        return (v & 0x7fffu) > kInf ? ~0u : ordered<OP>(v);
    }
};
using CumF16 = Cum16<0x7c00u>;
using CumBF16 = Cum16<0x7f80u>;
struct CumF64 {
    using raw = unsigned long long;  // binary64 bit patterns
    using key = unsigned long long;
    template <int OP> static __device__ __forceinline__ unsigned long long elem_key(unsigned long long b) {
        return TagF64::elem_key<OP>(b);
    }
    template <int OP> static __device__ __forceinline__ unsigned long long seed_key(unsigned long long b) {
        return TagF64::seed_key<OP>(b);
    }
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
};
using CumI32 = CumInt<int, unsigned>;
using CumI64 = CumInt<long long, unsigned long long>;

template <class CT>
struct Pfx {
    typename CT::key k;
    int i;
    typename CT::raw v;
};

// The later part b replaces the earlier prefix a only when strictly better.
template <class CT>
__device__ __forceinline__ Pfx<CT> later(const Pfx<CT>& a, const Pfx<CT>& b) {
    return b.k > a.k ? b : a;
}

template <class CT>
__device__ __forceinline__ Pfx<CT> pfx_identity() {
    Pfx<CT> p;
    p.k = 0;
    p.i = 0;
    p.v = typename CT::raw(0);
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
__device__ __forceinline__ Pfx<CT> shfl_up_pfx(const Pfx<CT>& p, int d) {
    Pfx<CT> q;
    q.k = shfl_up_any(p.k, d);
    q.i = __shfl_up_sync(0xffffffffu, p.i, d);
    q.v = shfl_up_any(p.v, d);
    return q;
}

constexpr int kCumMaxCluster = 16;

template <class CT, int OP, int ITEMS>
__global__ void __launch_bounds__(1024)
cum_kernel(const typename CT::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
           typename CT::raw* __restrict__ out_val) {
    using R = typename CT::raw;
    using K = typename CT::key;
    extern __shared__ __align__(16) unsigned char cum_smem[];
    __shared__ Pfx<CT> warp_tot[32];
    __shared__ Pfx<CT> s_total;
    __shared__ __align__(16) uint4 agg_slots[2][kCumMaxCluster];  // aggregates pushed by earlier CTAs
    const int nt = blockDim.x;
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = nt >> 5;
    const int C = gridDim.x;
    const int b = blockIdx.x;
    const int tile = nt * ITEMS;
    R* tin = reinterpret_cast<R*>(cum_smem);                                                  // tile input
    int* tidx = reinterpret_cast<int*>(cum_smem + static_cast<size_t>(tile) * sizeof(R));   // tile indices
    R* tval = reinterpret_cast<R*>(cum_smem + static_cast<size_t>(tile) * (sizeof(R) + 4)); // tile values
    bool started = false;
    if (C > 1) cluster_started_arrive();
    grid_dependency_wait();
    allow_dependents();
    int parity = 0;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y, parity ^= 1) {
        const R* row = x + r * static_cast<int64_t>(cols);
        const int cb = static_cast<int>(static_cast<int64_t>(cols) * b / C);
        const int ce = static_cast<int>(static_cast<int64_t>(cols) * (b + 1) / C);
        const R x0 = ld_scalar(row);
        Pfx<CT> carry;
        carry.k = CT::template seed_key<OP>(x0);
        carry.i = 0;
        carry.v = x0;
        if (C > 1) {
            // Phase A: this chunk's aggregate (first best element), identity-seeded.
            Pfx<CT> a = pfx_identity<CT>();
            for (int j = cb + t; j < ce; j += nt) {
                const R v = ld_scalar(row + j);
                const K k = CT::template elem_key<OP>(v);
                if (k > a.k) {
                    a.k = k;
                    a.i = j;
                    a.v = v;
                }
            }
            // CTA merge: higher key wins, equal keys keep the lower index.
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                Pfx<CT> o;
                o.k = __shfl_xor_sync(0xffffffffu, a.k, off);
                o.i = __shfl_xor_sync(0xffffffffu, a.i, off);
                o.v = shfl_xor_any(a.v, off);
                if (o.k > a.k || (o.k == a.k && o.i < a.i)) a = o;
            }
            if (lane == 0) warp_tot[warp] = a;
            __syncthreads();
            if (warp == 0) {
                a = lane < nwarps ? warp_tot[lane] : pfx_identity<CT>();
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    Pfx<CT> o;
                    o.k = __shfl_xor_sync(0xffffffffu, a.k, off);
                    o.i = __shfl_xor_sync(0xffffffffu, a.i, off);
                    o.v = shfl_xor_any(a.v, off);
                    if (o.k > a.k || (o.k == a.k && o.i < a.i)) a = o;
                }
            }
            if (!started) {  // every CTA of the cluster runs before the first remote write
                cluster_started_wait();
                started = true;
            }
            if (t < C - b - 1) {
                // Push this chunk's aggregate (key and index; the winner's raw
                // value is reloaded by whoever needs it) to the later CTA b + 1 + t.
                const uint64_t kk = static_cast<uint64_t>(a.k);
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
                Pfx<CT> e;
                e.k = static_cast<K>(static_cast<uint64_t>(pk.x) | (static_cast<uint64_t>(pk.y) << 32));
                e.i = static_cast<int>(pk.z);
                if (e.k > carry.k) {
                    carry.k = e.k;
                    carry.i = e.i;
                    carry.v = ld_scalar(row + e.i);  // the winner's raw bits (an L2 hit)
                }
            }
        }
        // Phase B: tiles of this chunk, in order.
        for (int base = cb; base < ce; base += tile) {
            const int n = ce - base < tile ? ce - base : tile;
            for (int j = t; j < n; j += nt) tin[j] = ld_scalar(row + base + j);
            __syncthreads();
            // thread-local inclusive prefixes of ITEMS consecutive elements
            Pfx<CT> p[ITEMS];
            Pfx<CT> run = pfx_identity<CT>();
#pragma unroll
            for (int q = 0; q < ITEMS; ++q) {
                const int j = t * ITEMS + q;
                if (j < n) {
                    const R v = tin[j];
                    const K k = CT::template elem_key<OP>(v);
                    if (k > run.k) {
                        run.k = k;
                        run.i = base + j;
                        run.v = v;
                    }
                }
                p[q] = run;
            }
            // warp inclusive scan of the thread totals
            Pfx<CT> ws = run;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const Pfx<CT> o = shfl_up_pfx(ws, d);
                if (lane >= d) ws = later(o, ws);
            }
            Pfx<CT> excl = shfl_up_pfx(ws, 1);
            if (lane == 0) excl = pfx_identity<CT>();
            if (lane == 31) warp_tot[warp] = ws;
            __syncthreads();
            if (warp == 0) {
                Pfx<CT> w = lane < nwarps ? warp_tot[lane] : pfx_identity<CT>();
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const Pfx<CT> o = shfl_up_pfx(w, d);
                    if (lane >= d) w = later(o, w);
                }
                Pfx<CT> we = shfl_up_pfx(w, 1);
                if (lane == 0) we = pfx_identity<CT>();
                if (lane < nwarps) warp_tot[lane] = we;  // exclusive prefix of each warp
                if (lane == nwarps - 1) s_total = w;
            }
            __syncthreads();
            const Pfx<CT> before = later(later(carry, warp_tot[warp]), excl);
#pragma unroll
            for (int q = 0; q < ITEMS; ++q) {
                const int j = t * ITEMS + q;
                if (j < n) {
                    const Pfx<CT> o = later(before, p[q]);
                    tidx[j] = o.i;
                    tval[j] = o.v;
                }
            }
            carry = later(carry, s_total);
            __syncthreads();
            int64_t* oi = out_idx + r * static_cast<int64_t>(cols) + base;
            for (int j = t; j < n; j += nt) oi[j] = tidx[j];
            if (out_val) {
                R* ov = out_val + r * static_cast<int64_t>(cols) + base;
                for (int j = t; j < n; j += nt) ov[j] = tval[j];
            }
            __syncthreads();  // the tile buffers are reused by the next tile
        }
    }
    if (C > 1 && !started) cluster_started_wait();  // complete the start phase even with no rows
}

// ---------------------------------------------------------------------------
// Launcher.
// ---------------------------------------------------------------------------
constexpr int kCumItems = 7;

inline size_t cum_smem_bytes(int block, int es) { return static_cast<size_t>(block) * kCumItems * (2 * es + 4); }

template <class CT, int OP>
cudaError_t launch_cum_op(const argr_plan& p, const Problem& pr) {
    using R = typename CT::raw;
    auto kern = cum_kernel<CT, OP, kCumItems>;
    const size_t smem = cum_smem_bytes(p.block, sizeof(R));
    static thread_local size_t smem_set = 0;
    if (smem > 48 * 1024 && smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    const int C = p.cluster > 1 ? p.cluster : 1;
    if (C > 8) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>(C), static_cast<unsigned>(p.grid_rows));
    if (C > 1) {
        // Refuse a cluster shape the device cannot co-schedule (checked once per shape).
        static thread_local int checked_block = 0, checked_cluster = 0, checked_ok = 0;
        if (checked_block != p.block || checked_cluster != C) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = grid;
            cfg.blockDim = dim3(p.block);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(C);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess) return e;
            checked_block = p.block;
            checked_cluster = C;
            checked_ok = n > 0;
        }
        if (!checked_ok) return cudaErrorInvalidClusterSize;  // reported as ARGR_EUNSUPPORTED
    }
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
