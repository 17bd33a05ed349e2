// argreduce kernels, templated on element tag, op and geometry. Each
// kernels_<dtype>.cu instantiates them for one element type.
//
// Paths (onnxruntime #32092 Approach, #31694 Description):
//  * rows_kernel    - G lanes per row (G = 1: one thread per row, G = 32: one
//                     warp per row), many rows per CTA, rows 16-byte aligned
//                     (VEC) or not (scalar loads). For narrow and medium rows.
//  * split_kernel   - one or more CTAs per row. A row spread over several CTAs
//                     is merged through a small global scratch: each CTA
//                     writes a partial, fences, and bumps the row's arrival
//                     counter; the CTA that arrives last merges the partials.
//                     The counter is bumped with a wrapping increment, so it
//                     is back at zero after every row and needs no memset.
//  * cluster_push_kernel - one thread-block cluster per row, a row slot per
//                     row: every warp pushes its candidate into CTA 0's shared
//                     memory (st.async on an mbarrier) and all CTAs but CTA 0
//                     leave at once; CTA 0 waits (bounded) and merges. No scratch.
//  * cluster_kernel - the same with fewer row slots than rows (CTAs loop over
//                     rows) or CTAs of more than 512 threads: CTAs store their
//                     candidates into CTA 0 and meet at a cluster barrier.
//  * cluster_bulk_kernel - a cluster per row with each CTA's share copied into
//                     shared memory by bulk (TMA) copies (forced plans).
//  * stream_kernel  - every warp owns a contiguous range of rows and streams
//                     them through its own shared-memory stages with bulk
//                     (TMA) copies, several in flight; rows that fit a stage
//                     are scanned G lanes per row, wider rows piece by piece
//                     by the whole warp. Rows must start on 16-byte boundaries.
//  * axis_kernel    - reduction over a non-last axis, x[outer][R][inner] over R.
//
// Index arithmetic: within a row every position is an int in [0, cols) with
// cols <= INT32_MAX. Loops are written with differences (remaining = end -
// position, and a step is only taken when it is smaller than what remains), so
// no sum can leave [0, cols) (#32092 review follow-up on the overflowing scan).
// Row offsets are 64-bit.
#pragma once

#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "tma.cuh"

namespace argr {

// ---------------------------------------------------------------------------
// G lanes per row.
// ---------------------------------------------------------------------------
template <class Tag, int OP, int G, bool VEC, int U, bool PIPE>
__global__ void __launch_bounds__(PIPE ? kPipeMaxBlock : 1024)
rows_kernel(const typename Tag::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
            typename Tag::raw* __restrict__ out_val, unsigned prefetch_bytes) {
    using R = typename Tag::raw;
    constexpr int E = 16 / sizeof(R);
    const int lg = threadIdx.x & (G - 1);
    const int lane = threadIdx.x & 31;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    const int groups_per_block = blockDim.x / G;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * groups_per_block;
    if (prefetch_bytes) {
        // the rows of this CTA's grid-stride steps, up to prefetch_bytes,
        // before waiting for the previous grid
        allow_dependents();
        const int64_t row_bytes = static_cast<int64_t>(cols) * static_cast<int64_t>(sizeof(R));
        int64_t budget = static_cast<int64_t>(prefetch_bytes);
        for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * groups_per_block; r0 < rows && budget > 0;
             r0 += stride) {
            const int64_t r1 = rows - r0 > groups_per_block ? r0 + groups_per_block : rows;
            prefetch_l2_range(x + r0 * cols, x + r1 * cols, static_cast<uintptr_t>(budget));
            budget -= (r1 - r0) * row_bytes;
        }
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        allow_dependents();
    }

    for (int64_t r = static_cast<int64_t>(blockIdx.x) * groups_per_block + threadIdx.x / G; r < rows;
         r += stride) {
        const R* row = x + r * static_cast<int64_t>(cols);
        Cand<Tag> c;
        if constexpr (VEC) {
            // Every row starts on a 16-byte boundary and cols % E == 0.
            const uint4* rv = reinterpret_cast<const uint4*>(row);
            const int nvec = cols / E;
            int v0 = lg;
            int rem = nvec - v0;
            uint4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) buf[u] = (u * G < rem) ? ld_stream16(rv + v0 + u * G) : make_uint4(0, 0, 0, 0);
            // Lane 0 of the group always holds vector 0, whose first element is x[0].
            c = make_cand<Tag, OP>(shfl_raw(gmask, vec_elem<R>(buf[0], 0), 0, G), 0);
            // The pipelined binary32 loop measured faster with the element-by-
            // element scanner ([2048,8192] f32 12.7 against 13.5 us).
            using Scan = std::conditional_t<PIPE && std::is_same<Tag, TagF32>::value, VecScanElems<Tag, OP>,
                                            VecScan<Tag, OP>>;
            Scan scan(c);
            if constexpr (PIPE) {
                // Software pipeline: the next batch's loads are issued before
                // the current batch is scanned, so a lane always has loads in
                // flight while it compares.
                for (;;) {
                    const bool more = rem > G * U;
                    uint4 nxt[U];
                    int v1 = v0, rem1 = 0;
                    if (more) {
                        v1 = v0 + G * U;
                        rem1 = nvec - v1;
#pragma unroll
                        for (int u = 0; u < U; ++u)
                            nxt[u] = (u * G < rem1) ? ld_stream16(rv + v1 + u * G) : make_uint4(0, 0, 0, 0);
                    }
                    #pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * G < rem) scan.visit(buf[u], (v0 + u * G) * E);
                    if (!more) break;
                    v0 = v1;
                    rem = rem1;
#pragma unroll
                    for (int u = 0; u < U; ++u) buf[u] = nxt[u];
                }
            } else {
                #pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * G < rem) scan.visit(buf[u], (v0 + u * G) * E);
                while (rem > G * U) {
                    v0 += G * U;
                    rem = nvec - v0;
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * G < rem) buf[u] = ld_stream16(rv + v0 + u * G);
                    #pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * G < rem) scan.visit(buf[u], (v0 + u * G) * E);
                }
            }
            c = scan.finish();
        } else {
            int j0 = lg;
            int rem = cols - j0;
            R buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) buf[u] = (u * G < rem) ? ld_scalar(row + j0 + u * G) : R(0);
            c = make_cand<Tag, OP>(shfl_raw(gmask, buf[0], 0, G), 0);  // lane 0 loaded x[0]
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u * G < rem) visit<Tag, OP>(c, buf[u], j0 + u * G);
            while (rem > G * U) {
                j0 += G * U;
                rem = cols - j0;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u * G < rem) buf[u] = ld_scalar(row + j0 + u * G);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u * G < rem) visit<Tag, OP>(c, buf[u], j0 + u * G);
            }
        }
        c = group_merge<Tag, OP, G>(c, gmask);
        if (lg == 0) {
            out_idx[r] = c.i;
            if (out_val) out_val[r] = cand_value<Tag>(c, row);
        }
    }
}

// ---------------------------------------------------------------------------
// Scan of this CTA's share of one row (shared by the split and cluster paths).
// The row is cut into a scalar head up to the first 16-byte boundary, a body
// of 16-byte vectors and a scalar tail. CTA b of nb owns a contiguous chunk of
// the body; CTA 0 also owns the head and CTA nb-1 the tail. Each thread visits
// its elements in increasing index order (head, body, tail).
// ---------------------------------------------------------------------------
struct ShareBounds {
    int head;  // elements before the first 16-byte boundary of the row
    int nvec;  // 16-byte vectors of the body
    int vb;    // this CTA's body vectors: [vb, ve)
    int ve;
};

template <typename R>
__device__ __forceinline__ ShareBounds share_bounds(const R* row, int cols, int b, int nb) {
    constexpr int E = 16 / sizeof(R);
    ShareBounds s;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    s.head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(R));
    if (s.head > cols) s.head = cols;
    s.nvec = (cols - s.head) / E;
    const int chunk = s.nvec / nb + (s.nvec % nb != 0);
    s.vb = b * chunk < s.nvec ? b * chunk : s.nvec;
    s.ve = s.nvec - s.vb > chunk ? s.vb + chunk : s.nvec;
    return s;
}

// L2 prefetch of CTA b's body vectors of a row (ARGR_PLAN_PREFETCH).
template <typename R>
__device__ __forceinline__ void prefetch_share(const R* row, int cols, int b, int nb) {
    const ShareBounds s = share_bounds(row, cols, b, nb);
    const uint4* rv = reinterpret_cast<const uint4*>(row + s.head);
    prefetch_l2_range(rv + s.vb, rv + s.ve);
}

template <class Tag, int OP, int U>
__device__ __forceinline__ Cand<Tag> scan_share(const typename Tag::raw* __restrict__ row, int cols, int b, int nb,
                                                typename Tag::raw x0) {
    using R = typename Tag::raw;
    constexpr int E = 16 / sizeof(R);
    const ShareBounds sb = share_bounds(row, cols, b, nb);
    const int head = sb.head, nvec = sb.nvec, vb = sb.vb, ve = sb.ve;
    const int tail0 = head + nvec * E;
    const uint4* rv = reinterpret_cast<const uint4*>(row + head);

    Cand<Tag> c = make_cand<Tag, OP>(x0, 0);
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    if (b == 0 && t < head) visit<Tag, OP>(c, ld_scalar(row + t), t);

    int v0 = vb + t;
    if (v0 < ve) {
        VecScan<Tag, OP> scan(c);
        for (;;) {
            const int rem = ve - v0;
            uint4 buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u * nt < rem) buf[u] = ld_stream16(rv + v0 + u * nt);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (u * nt < rem) scan.visit(buf[u], head + (v0 + u * nt) * E);
            if (rem <= U * nt) break;
            v0 += U * nt;
        }
        c = scan.finish();
    }
    if (b == nb - 1 && t < cols - tail0) visit<Tag, OP>(c, ld_scalar(row + tail0 + t), tail0 + t);
    return c;
}

template <class Tag>
__device__ __forceinline__ uint4 pack_cand(const Cand<Tag>& c) {
    using R = typename Tag::raw;
    uint64_t bits = 0;
    if constexpr (sizeof(R) == 8)
        bits = c.v;
    else if constexpr (sizeof(R) == 4)
        bits = __float_as_uint(c.v);
    else
        bits = c.v;
    return make_uint4(static_cast<uint32_t>(bits), static_cast<uint32_t>(bits >> 32), static_cast<uint32_t>(c.i), 0u);
}

template <class Tag, int OP>
__device__ __forceinline__ Cand<Tag> unpack_cand(const uint4& p) {
    using R = typename Tag::raw;
    R v;
    if constexpr (sizeof(R) == 8)
        v = static_cast<unsigned long long>(p.y) << 32 | p.x;
    else if constexpr (sizeof(R) == 4)
        v = __uint_as_float(p.x);
    else
        v = static_cast<uint16_t>(p.x);
    return make_cand<Tag, OP>(v, static_cast<int>(p.z));
}

// Arrival at a row's counter: a wrapping increment with acquire-release
// semantics at GPU scope. Release publishes this CTA's partial (stored before
// by the same thread); acquire lets the last arrival read every partial.
__device__ __forceinline__ unsigned arrive_acq_rel(unsigned* counter, unsigned wrap) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(counter), "r"(wrap) : "memory");
    return old;
}

__device__ __forceinline__ uint4 ld_relaxed_gpu(const uint4* p) {
    uint4 r;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p)
                 : "memory");
    return r;
}

// ---------------------------------------------------------------------------
// One or more CTAs per row; grid = (blocks_per_row, row_slots).
// With blocks_per_row > 1 every row has its own slot (row_slots >= rows).
// ---------------------------------------------------------------------------
template <class Tag, int OP, int U>
__global__ void __launch_bounds__(1024)
split_kernel(const typename Tag::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
             typename Tag::raw* __restrict__ out_val, unsigned char* __restrict__ scratch, bool prefetch) {
    using R = typename Tag::raw;
    __shared__ Cand<Tag> smem[32];
    const int nb = gridDim.x;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31;
    if (prefetch) {
        allow_dependents();
        if (blockIdx.y < rows) prefetch_share(x + static_cast<int64_t>(blockIdx.y) * cols, cols, b, nb);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        allow_dependents();
    }
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        const R* row = x + r * static_cast<int64_t>(cols);
        const R x0 = ld_scalar(row);
        const Cand<Tag> seed = make_cand<Tag, OP>(x0, 0);
        Cand<Tag> c = scan_share<Tag, OP, U>(row, cols, b, nb, x0);
        c = block_merge<Tag, OP>(c, smem, seed);  // merged candidate in warp 0
        if (threadIdx.x < 32) {
            if (nb == 1) {
                if (lane == 0) {
                    out_idx[r] = c.i;
                    if (out_val) out_val[r] = cand_value<Tag>(c, row);
                }
            } else {
                // Multi-CTA row: publish the partial, then arrive. The arrival
                // that returns nb-1 is the last one; the wrapping increment has
                // left the counter at zero for the next call.
                unsigned* counter = reinterpret_cast<unsigned*>(scratch + kCounterOffset) + blockIdx.y;
                uint4* parts = reinterpret_cast<uint4*>(scratch + kPartialsOffset) +
                               static_cast<size_t>(blockIdx.y) * nb;
                unsigned old = 0;
                if (lane == 0) {
                    parts[b] = pack_cand<Tag>(c);
                    old = arrive_acq_rel(counter, static_cast<unsigned>(nb - 1));
                }
                old = __shfl_sync(0xffffffffu, old, 0);
                __syncwarp();
                if (old == static_cast<unsigned>(nb - 1)) {
                    Cand<Tag> m = seed;
                    for (int k = lane; k < nb; k += 32) m = merge<Tag, OP>(m, unpack_cand<Tag, OP>(ld_relaxed_gpu(parts + k)));
                    m = group_merge<Tag, OP, 32>(m, 0xffffffffu);
                    if (lane == 0) {
                        out_idx[r] = m.i;
                        if (out_val) out_val[r] = cand_value<Tag>(m, row);
                    }
                }
            }
        }
        __syncthreads();  // shared memory is reused by the next row
    }
}

// ---------------------------------------------------------------------------
// One cluster of gridDim.x CTAs per row; grid = (cluster, row_slots).
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_addr(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Distributed shared memory of another CTA may only be accessed once that CTA
// is running. Every cluster kernel arrives on the cluster barrier when it
// starts (cluster_started_arrive) and completes that phase (cluster_started_wait)
// before its first remote access; by then all CTAs have long arrived, so the
// wait costs nothing on the critical path.
__device__ __forceinline__ void cluster_started_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_started_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <class Tag, int OP, int U>
__global__ void __launch_bounds__(1024)
cluster_kernel(const typename Tag::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
               typename Tag::raw* __restrict__ out_val, bool prefetch) {
    using R = typename Tag::raw;
    __shared__ Cand<Tag> smem[32];
    __shared__ __align__(16) uint4 slots[2][16];  // written by every CTA of the cluster into CTA 0
    const int nb = gridDim.x;   // the cluster spans the grid's x dimension
    const int b = blockIdx.x;   // == rank in the cluster
    int parity = 0;
    bool started = false;
    cluster_started_arrive();
    if (prefetch) {
        allow_dependents();
        if (blockIdx.y < rows) prefetch_share(x + static_cast<int64_t>(blockIdx.y) * cols, cols, b, nb);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        allow_dependents();
    }
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y, parity ^= 1) {
        const R* row = x + r * static_cast<int64_t>(cols);
        const R x0 = ld_scalar(row);
        const Cand<Tag> seed = make_cand<Tag, OP>(x0, 0);
        Cand<Tag> c = scan_share<Tag, OP, U>(row, cols, b, nb, x0);
        c = block_merge<Tag, OP>(c, smem, seed);
        if (!started) {  // every CTA of the cluster is running before the first push
            cluster_started_wait();
            started = true;
        }
        if (threadIdx.x == 0) {
            const uint4 p = pack_cand<Tag>(c);
            unsigned remote;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                         : "=r"(remote)
                         : "r"(smem_addr(&slots[parity][b])), "r"(0));
            asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(p.x), "r"(p.y),
                         "r"(p.z), "r"(p.w)
                         : "memory");
        }
        // Release the pushes, acquire everyone else's. Reuse of a slot two rows
        // later is ordered by the barrier of the row in between.
        cluster_barrier();
        if (b == 0 && threadIdx.x < 32) {
            Cand<Tag> m = threadIdx.x < nb ? unpack_cand<Tag, OP>(slots[parity][threadIdx.x]) : seed;
            m = group_merge<Tag, OP, 32>(m, 0xffffffffu);
            if (threadIdx.x == 0) {
                out_idx[r] = m.i;
                if (out_val) out_val[r] = cand_value<Tag>(m, row);
            }
        }
        __syncthreads();
    }
    if (!started) cluster_started_wait();  // complete the start phase even with no rows
}

// ---------------------------------------------------------------------------
// One cluster per row, each CTA with exactly one row (gridDim.y >= rows):
// the push merge. Instead of a CTA merge and a cluster barrier, every warp
// merges its lanes and pushes its 16-byte candidate into CTA 0's shared
// memory with st.async, which also counts the bytes on an mbarrier of CTA 0.
// A CTA other than 0 exits as soon as its warps have pushed (st.async takes
// its data from registers, so nothing of the exiting CTA is read later); CTA
// 0 stays until its barrier has counted every candidate of the cluster
// (a bounded wait) and merges them. No release fence, no cluster barrier
// after the start, and the SMs of a row's other CTAs are free for the next
// grid while CTA 0 merges.
// ---------------------------------------------------------------------------
constexpr int kPushMaxSlots = 16 * 32;  // CTAs of a cluster x warps of a CTA

__device__ __forceinline__ unsigned cluster_addr(unsigned local_smem, unsigned rank) {
    unsigned remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_smem), "r"(rank));
    return remote;
}

// Store 16 bytes into shared memory of a CTA of the cluster and count them on
// that CTA's mbarrier (both addresses from cluster_addr()).
__device__ __forceinline__ void st_async_v4(unsigned remote, const uint4& v, unsigned remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     remote),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
                 : "memory");
}

// try_wait with acquire at cluster scope: the candidates were written by
// other CTAs of the cluster.
__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

constexpr int kPushMaxBlock = 512;  // threads per CTA of the push merge kernel

// At most 512 threads and at least two CTAs per SM (64 registers a thread).
// PF (ARGR_PLAN_PREFETCH) and VAL (out_val given) are template parameters and
// every CTA has a row (gridDim.y == rows): each runtime test of these, kept
// live through the scan, measured 0.12-0.26 us slower per call.
template <class Tag, int OP, int U, bool PF, bool VAL>
__global__ void __launch_bounds__(kPushMaxBlock, 2)
cluster_push_kernel(const typename Tag::raw* __restrict__ x, int cols, int64_t* __restrict__ out_idx,
                    typename Tag::raw* __restrict__ out_val, int flags) {
    using R = typename Tag::raw;
    __shared__ __align__(16) uint4 slots[kPushMaxSlots];  // CTA 0: candidate of warp w of CTA b at b * nwarps + w
    __shared__ __align__(8) unsigned long long bar;
    const int nb = gridDim.x;  // the cluster spans the grid's x dimension
    const int b = blockIdx.x;  // == rank in the cluster
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const unsigned bar_local = smem_u32(&bar);
    if (b == 0 && t == 0) {
        // One phase: the arrival below plus every candidate's bytes. Test hook
        // (ARGR_PLAN_TEST_EXPIRE): 16 bytes more than the cluster pushes, so
        // CTA 0's wait (2 ms under the flag) expires.
        mbar_init(bar_local, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(bar_local, static_cast<unsigned>(nb * nwarps) * 16u +
                                             ((flags & ARGR_PLAN_TEST_EXPIRE) ? 16u : 0u));
    }
    cluster_started_arrive();  // after the barrier's initialisation (released by the fence above)
    const int64_t r = blockIdx.y;
    const R* row = x + r * static_cast<int64_t>(cols);
    if constexpr (PF) {
        allow_dependents();
        prefetch_share(row, cols, b, nb);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        allow_dependents();
    }
    const R x0 = ld_scalar(row);
    const Cand<Tag> seed = make_cand<Tag, OP>(x0, 0);
    Cand<Tag> c = scan_share<Tag, OP, U>(row, cols, b, nb, x0);
    c = group_merge<Tag, OP, 32>(c, 0xffffffffu);  // the warp's candidate, in every lane
    cluster_started_wait();  // every CTA of the cluster runs: CTA 0's barrier is initialised
    if (lane == 0)
        st_async_v4(cluster_addr(smem_u32(&slots[b * nwarps + warp]), 0), pack_cand<Tag>(c),
                    cluster_addr(bar_local, 0));
    if (b != 0 || warp != 0) return;
    // CTA 0, warp 0: wait (bounded) until every candidate has landed, then
    // merge. Every push of the cluster lands whether or not the wait expires
    // (the CTAs of a cluster run together), so CTA 0 never leaves with a
    // store into it still in flight.
    const unsigned long long limit_ns = (flags & ARGR_PLAN_TEST_EXPIRE) ? 2ull * 1000 * 1000 : kWaitLimitNs;
    bool ok = mbar_try_wait_cluster(bar_local, 0);
    if (!ok) {
        const unsigned long long t0 = global_timer_ns();
        while (!(ok = mbar_try_wait_cluster(bar_local, 0)) && global_timer_ns() - t0 <= limit_ns) {
        }
    }
    if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_device_error(kErrWaitExpired);
        return;
    }
    Cand<Tag> m = seed;
    for (int k = lane; k < nb * nwarps; k += 32) m = merge<Tag, OP>(m, unpack_cand<Tag, OP>(slots[k]));
    m = group_merge<Tag, OP, 32>(m, 0xffffffffu);
    if (lane == 0) {
        out_idx[r] = m.i;
        if constexpr (VAL) out_val[r] = cand_value<Tag>(m, row);
    }
}

// ---------------------------------------------------------------------------
// One cluster per row, with every CTA's share fetched by bulk copies.
//
// Same decomposition and merge as cluster_kernel, but CTA b's part of the
// row's 16-byte-aligned body (at most kBulkMaxPieces * kBulkPieceBytes bytes)
// is copied into shared memory by up to eight bulk copies issued at once, each
// completing on its own mbarrier, so the whole share is in flight at the start
// instead of a few loads per thread. Threads scan piece p as soon as it lands.
// The scalar head and tail are read directly as in scan_share().
// If a bounded wait expires the CTA records the error and skips its scans but
// keeps the control flow (merges, cluster barriers) of the other CTAs.
// ---------------------------------------------------------------------------
constexpr int kBulkPieceBytes = 16384;
constexpr int kBulkMaxPieces = 8;

template <class Tag, int OP>
__global__ void __launch_bounds__(1024)
cluster_bulk_kernel(const typename Tag::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
                    typename Tag::raw* __restrict__ out_val) {
    using R = typename Tag::raw;
    constexpr int E = 16 / sizeof(R);
    extern __shared__ __align__(128) unsigned char bulk_smem[];
    __shared__ Cand<Tag> smem[32];
    __shared__ __align__(16) uint4 slots[2][16];
    __shared__ __align__(8) unsigned long long bars[kBulkMaxPieces];
    grid_dependency_wait();
    allow_dependents();
    const int nb = gridDim.x;  // the cluster spans the grid's x dimension
    const int b = blockIdx.x;  // == rank in the cluster
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    const unsigned buf = smem_u32(bulk_smem);
    const unsigned bar0 = smem_u32(bars);
    bool started = false;
    cluster_started_arrive();
    if (t == 0) {
        for (int p = 0; p < kBulkMaxPieces; ++p) mbar_init(bar0 + 8 * p, 1);
        mbar_init_fence();
    }
    __syncthreads();

    bool abort = false;         // CTA-uniform from one row to the next
    unsigned phase_bits = 0;    // bit p: parity of barrier p's next phase
    unsigned pending = 0;       // bit p: a copy on barrier p not yet waited for (thread 0)
    int parity = 0;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y, parity ^= 1) {
        const R* row = x + r * static_cast<int64_t>(cols);
        const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
        int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(R));
        if (head > cols) head = cols;
        const int nvec = (cols - head) / E;
        const int tail0 = head + nvec * E;
        const uint4* rv = reinterpret_cast<const uint4*>(row + head);
        const int chunk = nvec / nb + (nvec % nb != 0);
        const int vb = b * chunk < nvec ? b * chunk : nvec;
        const int ve = nvec - vb > chunk ? vb + chunk : nvec;
        const int nbytes = (ve - vb) * 16;
        const int npieces = (nbytes + kBulkPieceBytes - 1) / kBulkPieceBytes;
        if (t == 0 && !abort) {
            fence_proxy_async_smem();  // earlier reads of the buffer come before the copies that overwrite it
            for (int p = 0; p < npieces; ++p) {
                const int off = p * kBulkPieceBytes;
                const int bytes = nbytes - off < kBulkPieceBytes ? nbytes - off : kBulkPieceBytes;
                mbar_arrive_expect_tx(bar0 + 8 * p, static_cast<unsigned>(bytes));
                bulk_copy_g2s(buf + off, reinterpret_cast<const unsigned char*>(rv + vb) + off,
                              static_cast<unsigned>(bytes), bar0 + 8 * p);
                pending |= 1u << p;
            }
        }
        const R x0 = ld_scalar(row);
        const Cand<Tag> seed = make_cand<Tag, OP>(x0, 0);
        Cand<Tag> c = seed;
        if (b == 0 && t < head) visit<Tag, OP>(c, ld_scalar(row + t), t);
        for (int p = 0; p < npieces; ++p) {
            const unsigned par = (phase_bits >> p) & 1u;
            if (!abort) {
                if (mbar_wait_bounded(bar0 + 8 * p, par)) {
                    const int off = p * kBulkPieceBytes;
                    const int nvp = (nbytes - off < kBulkPieceBytes ? nbytes - off : kBulkPieceBytes) >> 4;
                    const int v0 = vb + (off >> 4);
                    for (int v = t; v < nvp; v += nt)
                        visit_vec<Tag, OP>(c, ld_shared16(buf + off + 16u * v), head + (v0 + v) * E);
                } else {
                    record_device_error(kErrWaitExpired);
                    abort = true;
                }
            }
        }
        if (b == nb - 1 && t < cols - tail0) visit<Tag, OP>(c, ld_scalar(row + tail0 + t), tail0 + t);
        c = block_merge<Tag, OP>(c, smem, seed);
        if (!started) {  // every CTA of the cluster is running before the first push
            cluster_started_wait();
            started = true;
        }
        if (t == 0) {
            const uint4 pk = pack_cand<Tag>(c);
            unsigned remote;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(&slots[parity][b])), "r"(0));
            asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(pk.x), "r"(pk.y),
                         "r"(pk.z), "r"(pk.w)
                         : "memory");
        }
        cluster_barrier();
        if (b == 0 && t < 32) {
            Cand<Tag> m = t < nb ? unpack_cand<Tag, OP>(slots[parity][t]) : seed;
            m = group_merge<Tag, OP, 32>(m, 0xffffffffu);
            if (t == 0) {
                out_idx[r] = m.i;
                if (out_val) out_val[r] = m.v;
            }
        }
        const bool was_aborted = abort;
        abort = __syncthreads_or(abort) != 0;  // also: the buffer is free for the next row
        if (!was_aborted && !abort) {
            // every piece of this row was waited for: its barrier moved one phase
            phase_bits ^= (npieces >= 32 ? ~0u : ((1u << npieces) - 1u));
            if (t == 0) pending = 0;
        }
    }
    if (!started) cluster_started_wait();  // complete the start phase even with no rows
    if (abort && t == 0) {
        // Copies still in flight into this CTA's buffer: wait for them, bounded.
        for (int p = 0; p < kBulkMaxPieces; ++p)
            if (pending & (1u << p)) mbar_wait_bounded(bar0 + 8 * p, (phase_bits >> p) & 1u);
    }
}

// ---------------------------------------------------------------------------
// Reduction over a non-last axis: x[outer][R][inner] over R.
//
// A warp is CG column lanes by 32/CG lanes along R. Column lane cl owns V
// consecutive inner positions (V per lane: a 16-byte vector for 4- and 8-byte
// elements, 8 bytes for 16-bit ones, one element when the columns are not
// aligned), so a CTA tile is CG * V columns and each step along R reads
// segments of CG * V elements. The R lanes of a column take interleaved steps
// of the warp's part of R and merge with shuffles; the Y warps of a CTA take
// contiguous parts of R and merge per column through shared memory; with a
// cluster of C CTAs, R is first cut into C parts and the CTAs merge through
// distributed shared memory into CTA 0. Every lane visits its steps in
// increasing r. grid = (C, column tiles, outer slots); outer loops over the
// slots when C == 1.
// ---------------------------------------------------------------------------
template <typename R, int V>
struct AxisVec;
template <typename R>
struct AxisVec<R, 1> {
    static __device__ __forceinline__ void load(const R* p, R (&v)[1]) { v[0] = ld_scalar(p); }
};
template <>
struct AxisVec<float, 4> {
    static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
        const uint4 q = ld_stream16(p);
        v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y); v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
    }
};
template <>
struct AxisVec<unsigned long long, 2> {
    static __device__ __forceinline__ void load(const unsigned long long* p, unsigned long long (&v)[2]) {
        const uint4 q = ld_stream16(p);
        v[0] = static_cast<unsigned long long>(q.y) << 32 | q.x;
        v[1] = static_cast<unsigned long long>(q.w) << 32 | q.z;
    }
};
template <>
struct AxisVec<uint16_t, 4> {
    static __device__ __forceinline__ uint2 load_words(const uint16_t* p) {
        uint2 q;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(q.x), "=r"(q.y) : "l"(p));
        return q;
    }
    static __device__ __forceinline__ void load(const uint16_t* p, uint16_t (&v)[4]) {
        const uint2 q = load_words(p);
        v[0] = static_cast<uint16_t>(q.x & 0xffffu); v[1] = static_cast<uint16_t>(q.x >> 16);
        v[2] = static_cast<uint16_t>(q.y & 0xffffu); v[3] = static_cast<uint16_t>(q.y >> 16);
    }
};

template <class Tag, int OP, int V, int U, int CG>
__global__ void __launch_bounds__(1024)
axis_kernel(const typename Tag::raw* __restrict__ x, int64_t outer, int nred, int64_t inner,
            int64_t* __restrict__ out_idx, typename Tag::raw* __restrict__ out_val) {
    using R = typename Tag::raw;
    constexpr int RG = 32 / CG;  // lanes of a warp along R for each column lane
    extern __shared__ __align__(16) uint4 axis_smem[];  // [Y][CG][V] CTA merge, then [C][CG][V] cluster slots
    grid_dependency_wait();
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int cl = lane % CG;   // column lane
    const int rl = lane / CG;   // R lane
    const int y = threadIdx.x >> 5;
    const int Y = blockDim.x >> 5;
    const int C = gridDim.x;
    const int b = blockIdx.x;  // rank in the cluster (the cluster spans x)
    uint4* cta_slots = axis_smem;
    uint4* cl_slots = axis_smem + Y * CG * V;
    bool started = false;
    if (C > 1) cluster_started_arrive();
    const int64_t i0 = (static_cast<int64_t>(blockIdx.y) * CG + cl) * V;  // this lane's first column
    const bool active = i0 < inner;
    // This warp's part of R: CTA part b of C, then warp part y of Y; its R
    // lanes take every RG-th step of that part.
    const int64_t cb = static_cast<int64_t>(nred) * b / C, ce = static_cast<int64_t>(nred) * (b + 1) / C;
    const int rs = static_cast<int>(cb + (ce - cb) * y / Y);
    const int re = static_cast<int>(cb + (ce - cb) * (y + 1) / Y);
    for (int64_t o = blockIdx.z; o < outer; o += gridDim.z) {
        const R* col = x + (o * nred) * inner + i0;
        Cand<Tag> c[V];
        R v0[V];
        if (active) AxisVec<R, V>::load(col, v0);  // row r = 0 seeds every candidate
#pragma unroll
        for (int v = 0; v < V; ++v) c[v] = make_cand<Tag, OP>(active ? v0[v] : R(0), 0);
        if constexpr (sizeof(R) == 2 && V == 4) {
            // 16-bit columns, two to a 32-bit word: two independent scans per
            // packed step (pair_step), both with the row's index. A column
            // whose x[0] is NaN keeps (x[0], 0) (nothing displaces it), which
            // is restored after the loop since the packed max moves its key.
            if (active) {
                uint32_t kv0 = static_cast<uint32_t>(v0[0]) | static_cast<uint32_t>(v0[1]) << 16;
                uint32_t kv1 = static_cast<uint32_t>(v0[2]) | static_cast<uint32_t>(v0[3]) << 16;
                int ix[4] = {0, 0, 0, 0};
                int r = rs + rl;
                while (r < re) {
                    const int rem = re - r;  // > 0
                    uint2 buf[U];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * RG < rem) buf[u] = AxisVec<R, 4>::load_words(col + static_cast<int64_t>(r + u * RG) * inner);
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (u * RG < rem) {
                            pair_step<Tag, OP>(kv0, ix[0], ix[1], buf[u].x, r + u * RG);
                            pair_step<Tag, OP>(kv1, ix[2], ix[3], buf[u].y, r + u * RG);
                        }
                    if (rem <= U * RG) break;
                    r += U * RG;
                }
                const uint32_t keys[4] = {kv0 & 0xffffu, kv0 >> 16, kv1 & 0xffffu, kv1 >> 16};
#pragma unroll
                for (int v = 0; v < V; ++v)
                    if (c[v].k == c[v].k) c[v] = make_cand<Tag, OP>(static_cast<R>(keys[v]), ix[v]);
            }
        } else if (active) {
            int r = rs + rl;
            while (r < re) {
                const int rem = re - r;  // > 0
                R buf[U][V];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u * RG < rem) AxisVec<R, V>::load(col + static_cast<int64_t>(r + u * RG) * inner, buf[u]);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (u * RG < rem) {
#pragma unroll
                        for (int v = 0; v < V; ++v) visit<Tag, OP>(c[v], buf[u][v], r + u * RG);
                    }
                if (rem <= U * RG) break;
                r += U * RG;
            }
        }
        // Merge the R lanes of each column lane (lanes cl, cl + CG, ...).
#pragma unroll
        for (int off = CG; off < 32; off <<= 1) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const Cand<Tag> other = make_cand<Tag, OP>(shfl_xor_raw(0xffffffffu, c[v].v, off, 32),
                                                           __shfl_xor_sync(0xffffffffu, c[v].i, off, 32));
                c[v] = merge<Tag, OP>(c[v], other);
            }
        }
        // Merge the Y warps of this CTA, column by column (warp 0).
        if (rl == 0 && active) {
#pragma unroll
            for (int v = 0; v < V; ++v) cta_slots[(y * CG + cl) * V + v] = pack_cand<Tag>(c[v]);
        }
        __syncthreads();
        const bool writer = y == 0 && rl == 0 && active;
        if (writer) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                Cand<Tag> m = c[v];
                for (int w = 1; w < Y; ++w) m = merge<Tag, OP>(m, unpack_cand<Tag, OP>(cta_slots[(w * CG + cl) * V + v]));
                c[v] = m;
            }
        }
        if (C > 1) {
            if (!started) {  // every CTA of the cluster is running before the first push
                cluster_started_wait();
                started = true;
            }
            if (writer) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const uint4 pk = pack_cand<Tag>(c[v]);
                    unsigned remote;
                    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                                 : "=r"(remote)
                                 : "r"(smem_addr(&cl_slots[(b * CG + cl) * V + v])), "r"(0));
                    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(pk.x),
                                 "r"(pk.y), "r"(pk.z), "r"(pk.w)
                                 : "memory");
                }
            }
            cluster_barrier();
            if (b == 0 && writer) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    Cand<Tag> m = unpack_cand<Tag, OP>(cl_slots[cl * V + v]);
                    for (int k = 1; k < C; ++k) m = merge<Tag, OP>(m, unpack_cand<Tag, OP>(cl_slots[(k * CG + cl) * V + v]));
                    c[v] = m;
                }
            }
        }
        if (b == 0 && writer) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                if (i0 + v < inner) {
                    out_idx[o * inner + i0 + v] = c[v].i;
                    if (out_val) {
                        R val = c[v].v;
                        // the packed 16-bit scan may keep a zero of the other sign: read zeros back
                        if constexpr (sizeof(R) == 2 && V == 4) {
                            if ((val & 0x7fffu) == 0) val = ld_scalar(col + static_cast<int64_t>(c[v].i) * inner + v);
                        }
                        out_val[o * inner + i0 + v] = val;
                    }
                }
            }
        }
        __syncthreads();  // the CTA merge slots are reused by the next outer index
    }
    if (C > 1 && !started) cluster_started_wait();  // complete the start phase even with no work
}

// ---------------------------------------------------------------------------
// Per-warp streaming through shared memory with bulk copies.
// ---------------------------------------------------------------------------
constexpr int kMaxStreamWarps = 32;
constexpr int kMaxStreamStages = 4;

// Where piece q of a warp's row range [r0, r1) comes from.
struct Piece {
    int64_t row;      // first row of the piece
    int64_t off;      // byte offset of the piece inside that row (wide rows)
    int bytes;        // bytes in the piece
    int nrows;        // whole rows in the piece (rows that fit a stage)
    bool row_end;     // the piece ends its row (wide rows)
};

__device__ __forceinline__ Piece stream_piece(int64_t q, int64_t r0, int64_t r1, int64_t row_bytes, int stage_bytes,
                                              int rows_per_piece, int pieces_per_row) {
    Piece p;
    if (rows_per_piece > 0) {
        p.row = r0 + q * rows_per_piece;
        const int64_t left = r1 - p.row;
        p.nrows = static_cast<int>(left < rows_per_piece ? left : rows_per_piece);
        p.off = 0;
        p.bytes = static_cast<int>(p.nrows * row_bytes);
        p.row_end = true;
    } else {
        const int64_t k = q / pieces_per_row;
        const int64_t j = q - k * pieces_per_row;
        p.row = r0 + k;
        p.off = j * stage_bytes;
        const int64_t left = row_bytes - p.off;
        p.bytes = static_cast<int>(left < stage_bytes ? left : stage_bytes);
        p.nrows = 1;
        p.row_end = j == pieces_per_row - 1;
    }
    return p;
}

template <class Tag, int OP, int G>
__global__ void __launch_bounds__(1024)
stream_kernel(const typename Tag::raw* __restrict__ x, int64_t rows, int cols, int64_t* __restrict__ out_idx,
              typename Tag::raw* __restrict__ out_val, int stages, int stage_bytes, int flags) {
    using R = typename Tag::raw;
    constexpr int E = 16 / sizeof(R);
    extern __shared__ __align__(128) unsigned char stream_smem[];
    __shared__ __align__(8) unsigned long long bars[kMaxStreamWarps * kMaxStreamStages];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * W;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * W + w;
    const int64_t r0 = rows * gw / nw;
    const int64_t r1 = rows * (gw + 1) / nw;
    if (flags & ARGR_PLAN_PREFETCH) {
        // the CTA's rows (contiguous: its warps' ranges follow one another),
        // up to kPrefetchMaxBytes, before waiting for the previous grid
        allow_dependents();
        const int64_t c0 = rows * (static_cast<int64_t>(blockIdx.x) * W) / nw;
        const int64_t c1 = rows * (static_cast<int64_t>(blockIdx.x + 1) * W) / nw;
        prefetch_l2_range(x + c0 * cols, x + c1 * cols);
        grid_dependency_wait();
    } else {
        grid_dependency_wait();
        allow_dependents();
    }
    const int64_t row_bytes = static_cast<int64_t>(cols) * static_cast<int64_t>(sizeof(R));
    // Rows that fit a stage travel whole (rows_per_piece > 0); wider rows in pieces.
    const int rows_per_piece = row_bytes <= stage_bytes ? static_cast<int>(stage_bytes / row_bytes) : 0;
    const int pieces_per_row = rows_per_piece > 0 ? 1 : static_cast<int>((row_bytes + stage_bytes - 1) / stage_bytes);
    const int64_t nrows = r1 - r0;
    const int64_t total = rows_per_piece > 0 ? (nrows + rows_per_piece - 1) / rows_per_piece : nrows * pieces_per_row;

    const unsigned my_smem = smem_u32(stream_smem) + static_cast<unsigned>(w * stages * stage_bytes);
    const unsigned my_bar = smem_u32(bars) + static_cast<unsigned>(w * kMaxStreamStages * 8);
    const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(my_bar + 8 * s, 1);
        mbar_init_fence();
    }
    __syncwarp();
    // Test hook (ARGR_PLAN_TEST_EXPIRE): the first piece's barrier expects 16
    // bytes more than are copied, so its phase never completes and the bounded
    // wait (shortened to 2 ms) runs out. The copy itself lands.
    const bool expire = (flags & ARGR_PLAN_TEST_EXPIRE) != 0;
    const unsigned long long limit_ns = expire ? 2ull * 1000 * 1000 : kWaitLimitNs;
    auto issue = [&](int64_t q) {
        const Piece p = stream_piece(q, r0, r1, row_bytes, stage_bytes, rows_per_piece, pieces_per_row);
        const int s = static_cast<int>(q % stages);
        const unsigned bar = my_bar + 8 * s;
        mbar_arrive_expect_tx(bar, static_cast<unsigned>(p.bytes) + (expire && q == 0 ? 16u : 0u));
        bulk_copy_g2s(my_smem + static_cast<unsigned>(s * stage_bytes), xb + p.row * row_bytes + p.off,
                      static_cast<unsigned>(p.bytes), bar);
    };
    if (lane == 0)
        for (int64_t q = 0; q < total && q < stages; ++q) issue(q);

    const int lg = lane & (G - 1);
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    bool abort = false;
    int64_t waited = 0;  // pieces whose barrier this warp has passed
    Cand<Tag> c = make_cand<Tag, OP>(R(0), 0);
    for (int64_t q = 0; q < total; ++q) {
        const int s = static_cast<int>(q % stages);
        const unsigned parity = static_cast<unsigned>((q / stages) & 1);
        if (!abort) {
            const bool ok = mbar_wait_bounded(my_bar + 8 * s, parity, limit_ns);
            abort = __any_sync(0xffffffffu, !ok);
            if (abort) {
                if (lane == 0) record_device_error(kErrWaitExpired);
            } else {
                waited = q + 1;
            }
        }
        if (!abort) {
            const Piece p = stream_piece(q, r0, r1, row_bytes, stage_bytes, rows_per_piece, pieces_per_row);
            const unsigned base = my_smem + static_cast<unsigned>(s * stage_bytes);
            if (rows_per_piece > 0) {
                // Whole rows: G lanes per row, 32 / G rows at a time.
                const int nv = static_cast<int>(row_bytes >> 4);
                for (int rr = lane / G; rr < p.nrows; rr += 32 / G) {
                    const unsigned rbase = base + static_cast<unsigned>(rr * row_bytes);
                    Cand<Tag> rc = make_cand<Tag, OP>(vec_elem<R>(ld_shared16(rbase), 0), 0);
                    for (int v = lg; v < nv; v += G) visit_vec<Tag, OP>(rc, ld_shared16(rbase + 16u * v), v * E);
                    rc = group_merge<Tag, OP, G>(rc, gmask);
                    if (lg == 0) {
                        out_idx[p.row + rr] = rc.i;
                        if (out_val) out_val[p.row + rr] = rc.v;
                    }
                }
            } else {
                // A piece of a wide row: the whole warp, a running candidate.
                const int v0 = static_cast<int>(p.off >> 4);
                if (p.off == 0) c = make_cand<Tag, OP>(vec_elem<R>(ld_shared16(base), 0), 0);
                const int nvp = p.bytes >> 4;
                for (int v = lane; v < nvp; v += 32) visit_vec<Tag, OP>(c, ld_shared16(base + 16u * v), (v0 + v) * E);
                if (p.row_end) {
                    c = group_merge<Tag, OP, 32>(c, 0xffffffffu);
                    if (lane == 0) {
                        out_idx[p.row] = c.i;
                        if (out_val) out_val[p.row] = c.v;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && !abort && q + stages < total) {
            fence_proxy_async_smem();  // this stage's reads come before the copy that overwrites it
            issue(q + stages);
        }
    }
    if (abort && lane == 0) {
        // Copies issued but not waited for: wait for them (bounded) before leaving.
        const int64_t issued = total < waited + stages ? total : waited + stages;
        for (int64_t q = waited; q < issued; ++q)
            mbar_wait_bounded(my_bar + 8 * static_cast<int>(q % stages), static_cast<unsigned>((q / stages) & 1),
                              limit_ns);
    }
}

// ---------------------------------------------------------------------------
// Per-device launch facts: a kernel's raised dynamic shared memory limit, its
// permission for 16-CTA clusters, and whether a cluster shape fits the device.
// Kernel attributes belong to the current device, so each is recorded per
// device; the records are shared by every host thread (atomics, or a mutex
// for the occupancy answers).
// ---------------------------------------------------------------------------
constexpr int kLaunchCacheDevices = 64;

struct KernelLaunchCache {
    std::atomic<size_t> smem_limit[kLaunchCacheDevices];  // dynamic shared memory already allowed
    std::atomic<bool> big_cluster[kLaunchCacheDevices];   // non-portable cluster size allowed
    struct Fit {
        int dev, block, cluster;
        size_t smem;
        bool ok;
    };
    std::mutex mu;
    Fit fits[16];
    int n_fits;
};

inline cudaError_t launch_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e == cudaSuccess && (*dev < 0 || *dev >= kLaunchCacheDevices)) *dev = -1;  // not cached
    return e;
}

// Raise the kernel's dynamic shared memory limit to `smem` on the current device if needed.
template <class K>
cudaError_t ensure_smem_limit(K kern, size_t smem, KernelLaunchCache& c) {
    if (smem <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = launch_device(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && c.smem_limit[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && dev >= 0) {
        size_t cur = c.smem_limit[dev].load(std::memory_order_relaxed);
        while (cur < smem && !c.smem_limit[dev].compare_exchange_weak(cur, smem, std::memory_order_release)) {
        }
    }
    return e;
}

// Allow clusters of more than 8 CTAs for the kernel on the current device.
template <class K>
cudaError_t allow_big_cluster(K kern, KernelLaunchCache& c) {
    int dev = 0;
    cudaError_t e = launch_device(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && c.big_cluster[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && dev >= 0) c.big_cluster[dev].store(true, std::memory_order_release);
    return e;
}

// Whether the current device can co-schedule clusters of `cluster` CTAs of
// `block` threads with `smem` bytes of dynamic shared memory (answers cached).
template <class K>
cudaError_t cluster_fits(K kern, dim3 grid, int block, int cluster, size_t smem, KernelLaunchCache& c, bool* ok) {
    int dev = 0;
    cudaError_t e = launch_device(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lk(c.mu);
        for (int i = 0; i < c.n_fits && i < 16; ++i) {
            const KernelLaunchCache::Fit& f = c.fits[i];
            if (f.dev == dev && f.block == block && f.cluster == cluster && f.smem == smem) {
                *ok = f.ok;
                return cudaSuccess;
            }
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(cluster);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    *ok = n > 0;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lk(c.mu);
        c.fits[c.n_fits % 16] = KernelLaunchCache::Fit{dev, block, cluster, smem, *ok};
        ++c.n_fits;
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Launchers. Every launch goes through cudaLaunchKernelEx so that it can carry
// the programmatic-dependent-launch attribute (plan flag ARGR_PLAN_PDL) and,
// on the cluster path, the cluster shape.
// ---------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
cudaError_t launch_ex_smem(void (*kern)(KArgs...), dim3 grid, dim3 block, int cluster, size_t smem,
                           const argr_plan& p, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (p.flags & ARGR_PLAN_PDL) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, int cluster, const argr_plan& p,
                      cudaStream_t stream, Args... args) {
    return launch_ex_smem(kern, grid, block, cluster, 0, p, stream, args...);
}
template <class Tag, int OP, int G, int U>
cudaError_t launch_rows_gu(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    const dim3 grid(static_cast<unsigned>(p.grid_rows));
    const R* x = static_cast<const R*>(pr.x);
    R* ov = static_cast<R*>(pr.out_val);
    // bytes each CTA prefetches before its dependency wait (0: none)
    const unsigned pf = !(p.flags & ARGR_PLAN_PREFETCH)    ? 0u
                        : (p.flags & ARGR_PLAN_PREFETCH_HEAD) ? static_cast<unsigned>(kPrefetchHeadBytes)
                                                              : static_cast<unsigned>(kPrefetchMaxBytes);
    if constexpr (G >= 16) {
        if (p.flags & ARGR_PLAN_PIPELINE)  // check_plan admits it only with vec and G >= 16
            return launch_ex(rows_kernel<Tag, OP, G, true, U, true>, grid, dim3(p.block), 1, p, pr.stream, x,
                             pr.rows, pr.cols, pr.out_idx, ov, pf);
    }
    if (p.vec)
        return launch_ex(rows_kernel<Tag, OP, G, true, U, false>, grid, dim3(p.block), 1, p, pr.stream, x, pr.rows,
                         pr.cols, pr.out_idx, ov, pf);
    return launch_ex(rows_kernel<Tag, OP, G, false, U, false>, grid, dim3(p.block), 1, p, pr.stream, x, pr.rows,
                     pr.cols, pr.out_idx, ov, pf);
}

template <class Tag, int OP, int G>
cudaError_t launch_rows_g(const argr_plan& p, const Problem& pr) {
    return p.unroll == 8 ? launch_rows_gu<Tag, OP, G, 8>(p, pr) : launch_rows_gu<Tag, OP, G, 4>(p, pr);
}

template <class Tag, int OP>
cudaError_t launch_rows_op(const argr_plan& p, const Problem& pr) {
    switch (p.group) {
        case 1: return launch_rows_g<Tag, OP, 1>(p, pr);
        case 2: return launch_rows_g<Tag, OP, 2>(p, pr);
        case 4: return launch_rows_g<Tag, OP, 4>(p, pr);
        case 8: return launch_rows_g<Tag, OP, 8>(p, pr);
        case 16: return launch_rows_g<Tag, OP, 16>(p, pr);
        case 32: return launch_rows_g<Tag, OP, 32>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag>
cudaError_t launch_rows_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_rows_op<Tag, kOpMax>(p, pr);
        case kOpMin: return launch_rows_op<Tag, kOpMin>(p, pr);
        case kOpMaxLast: return launch_rows_op<Tag, kOpMaxLast>(p, pr);
        case kOpMinLast: return launch_rows_op<Tag, kOpMinLast>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag, int OP, int U>
cudaError_t launch_split_u(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    const dim3 grid(static_cast<unsigned>(p.blocks_per_row), static_cast<unsigned>(p.grid_rows));
    return launch_ex(split_kernel<Tag, OP, U>, grid, dim3(p.block), 1, p, pr.stream, static_cast<const R*>(pr.x),
                     pr.rows, pr.cols, pr.out_idx, static_cast<R*>(pr.out_val),
                     static_cast<unsigned char*>(pr.scratch), (p.flags & ARGR_PLAN_PREFETCH) != 0);
}

template <class Tag, int OP>
cudaError_t launch_split_op(const argr_plan& p, const Problem& pr) {
    switch (p.unroll) {
        case 1: return launch_split_u<Tag, OP, 1>(p, pr);
        case 2: return launch_split_u<Tag, OP, 2>(p, pr);
        case 4: return launch_split_u<Tag, OP, 4>(p, pr);
        case 8: return launch_split_u<Tag, OP, 8>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag>
cudaError_t launch_split_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_split_op<Tag, kOpMax>(p, pr);
        case kOpMin: return launch_split_op<Tag, kOpMin>(p, pr);
        case kOpMaxLast: return launch_split_op<Tag, kOpMaxLast>(p, pr);
        case kOpMinLast: return launch_split_op<Tag, kOpMinLast>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

// Before launching a cluster kernel: enable cluster sizes above 8 for it and
// check that the device can co-schedule the plan's cluster shape.
template <class K>
cudaError_t prepare_cluster_launch(K kern, KernelLaunchCache& cache, const argr_plan& p) {
    if (p.cluster > 8) {
        // Cluster sizes above the portable 8 must be enabled per kernel.
        cudaError_t e = allow_big_cluster(kern, cache);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>(p.cluster), static_cast<unsigned>(p.grid_rows));
    bool ok = false;  // refuse a cluster shape the device cannot co-schedule
    cudaError_t e = cluster_fits(kern, grid, p.block, p.cluster, 0, cache, &ok);
    if (e != cudaSuccess) return e;
    if (!ok) return cudaErrorInvalidClusterSize;  // reported as ARGR_EUNSUPPORTED
    return cudaSuccess;
}

template <class Tag, int OP, int U, bool PF, bool VAL>
cudaError_t launch_push(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    auto kern = cluster_push_kernel<Tag, OP, U, PF, VAL>;
    static KernelLaunchCache cache;
    cudaError_t e = prepare_cluster_launch(kern, cache, p);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(p.cluster), static_cast<unsigned>(p.grid_rows));
    return launch_ex(kern, grid, dim3(p.block), p.cluster, p, pr.stream, static_cast<const R*>(pr.x), pr.cols,
                     pr.out_idx, static_cast<R*>(pr.out_val), static_cast<int>(p.flags));
}

template <class Tag, int OP, int U>
cudaError_t launch_cluster_u(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    const bool pf = (p.flags & ARGR_PLAN_PREFETCH) != 0;
    if (p.grid_rows == pr.rows && p.block <= kPushMaxBlock) {
        // one row per CTA: the push merge
        if (pr.out_val)
            return pf ? launch_push<Tag, OP, U, true, true>(p, pr) : launch_push<Tag, OP, U, false, true>(p, pr);
        return pf ? launch_push<Tag, OP, U, true, false>(p, pr) : launch_push<Tag, OP, U, false, false>(p, pr);
    }
    // rows looping over fewer row slots, spare row slots, or CTAs of more than
    // 512 threads: the barrier merge
    auto kern = cluster_kernel<Tag, OP, U>;
    static KernelLaunchCache cache;
    cudaError_t e = prepare_cluster_launch(kern, cache, p);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(p.cluster), static_cast<unsigned>(p.grid_rows));
    return launch_ex(kern, grid, dim3(p.block), p.cluster, p, pr.stream, static_cast<const R*>(pr.x), pr.rows,
                     pr.cols, pr.out_idx, static_cast<R*>(pr.out_val), pf);
}

// Dynamic shared memory the bulk cluster kernel needs: the largest share of a
// row's 16-byte-aligned body one CTA can own.
inline size_t cluster_bulk_smem(const argr_plan& p, int cols, int es) {
    const int64_t nvec = static_cast<int64_t>(cols) * es / 16;
    return static_cast<size_t>((nvec + p.cluster - 1) / p.cluster) * 16;
}

template <class Tag, int OP>
cudaError_t launch_cluster_bulk(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    auto kern = cluster_bulk_kernel<Tag, OP>;
    const size_t smem = cluster_bulk_smem(p, pr.cols, sizeof(R));
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    if (p.cluster > 8) {
        e = allow_big_cluster(kern, cache);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(static_cast<unsigned>(p.cluster), static_cast<unsigned>(p.grid_rows));
    bool ok = false;
    e = cluster_fits(kern, grid, p.block, p.cluster, smem, cache, &ok);
    if (e != cudaSuccess) return e;
    if (!ok) return cudaErrorInvalidClusterSize;  // reported as ARGR_EUNSUPPORTED
    return launch_ex_smem(kern, grid, dim3(p.block), p.cluster, smem, p, pr.stream, static_cast<const R*>(pr.x),
                          pr.rows, pr.cols, pr.out_idx, static_cast<R*>(pr.out_val));
}

template <class Tag, int OP>
cudaError_t launch_cluster_op(const argr_plan& p, const Problem& pr) {
    if (p.flags & ARGR_PLAN_BULK) return launch_cluster_bulk<Tag, OP>(p, pr);
    switch (p.unroll) {
        case 1: return launch_cluster_u<Tag, OP, 1>(p, pr);
        case 2: return launch_cluster_u<Tag, OP, 2>(p, pr);
        case 4: return launch_cluster_u<Tag, OP, 4>(p, pr);
        case 8: return launch_cluster_u<Tag, OP, 8>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag>
cudaError_t launch_cluster_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_cluster_op<Tag, kOpMax>(p, pr);
        case kOpMin: return launch_cluster_op<Tag, kOpMin>(p, pr);
        case kOpMaxLast: return launch_cluster_op<Tag, kOpMaxLast>(p, pr);
        case kOpMinLast: return launch_cluster_op<Tag, kOpMinLast>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag, int OP, int G>
cudaError_t launch_stream_g(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    auto kern = stream_kernel<Tag, OP, G>;
    const size_t smem = static_cast<size_t>(p.block / 32) * p.stages * p.stage_bytes;
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    return launch_ex_smem(kern, dim3(static_cast<unsigned>(p.grid_rows)), dim3(p.block), 1, smem, p, pr.stream,
                          static_cast<const R*>(pr.x), pr.rows, pr.cols, pr.out_idx, static_cast<R*>(pr.out_val),
                          p.stages, p.stage_bytes, p.flags);
}

template <class Tag, int OP>
cudaError_t launch_stream_op(const argr_plan& p, const Problem& pr) {
    switch (p.group) {
        case 1: return launch_stream_g<Tag, OP, 1>(p, pr);
        case 2: return launch_stream_g<Tag, OP, 2>(p, pr);
        case 4: return launch_stream_g<Tag, OP, 4>(p, pr);
        case 8: return launch_stream_g<Tag, OP, 8>(p, pr);
        case 16: return launch_stream_g<Tag, OP, 16>(p, pr);
        case 32: return launch_stream_g<Tag, OP, 32>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag>
cudaError_t launch_stream_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_stream_op<Tag, kOpMax>(p, pr);
        case kOpMin: return launch_stream_op<Tag, kOpMin>(p, pr);
        case kOpMaxLast: return launch_stream_op<Tag, kOpMaxLast>(p, pr);
        case kOpMinLast: return launch_stream_op<Tag, kOpMinLast>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag, int OP, int V, int U, int CG>
cudaError_t launch_axis_vug(const argr_plan& p, const Problem& pr) {
    using R = typename Tag::raw;
    auto kern = axis_kernel<Tag, OP, V, U, CG>;
    const int Y = p.block / 32;
    const int C = p.cluster > 1 ? p.cluster : 1;
    const size_t smem = static_cast<size_t>(Y + (C > 1 ? C : 0)) * CG * V * sizeof(uint4);
    static KernelLaunchCache cache;
    cudaError_t e = ensure_smem_limit(kern, smem, cache);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = allow_big_cluster(kern, cache);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = (pr.inner + CG * V - 1) / (CG * V);
    const dim3 grid(static_cast<unsigned>(C), static_cast<unsigned>(tiles), static_cast<unsigned>(p.grid_rows));
    if (C > 1) {
        bool ok = false;  // refuse a cluster shape the device cannot co-schedule
        e = cluster_fits(kern, grid, p.block, C, smem, cache, &ok);
        if (e != cudaSuccess) return e;
        if (!ok) return cudaErrorInvalidClusterSize;  // reported as ARGR_EUNSUPPORTED
    }
    return launch_ex_smem(kern, grid, dim3(p.block), C, smem, p, pr.stream, static_cast<const R*>(pr.x), pr.rows,
                          pr.cols, pr.inner, pr.out_idx, static_cast<R*>(pr.out_val));
}

template <class Tag, int OP, int V, int U>
cudaError_t launch_axis_vu(const argr_plan& p, const Problem& pr) {
    switch (p.group) {
        case 1: return launch_axis_vug<Tag, OP, V, U, 1>(p, pr);
        case 2: return launch_axis_vug<Tag, OP, V, U, 2>(p, pr);
        case 4: return launch_axis_vug<Tag, OP, V, U, 4>(p, pr);
        case 8: return launch_axis_vug<Tag, OP, V, U, 8>(p, pr);
        case 16: return launch_axis_vug<Tag, OP, V, U, 16>(p, pr);
        case 32: return launch_axis_vug<Tag, OP, V, U, 32>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

template <class Tag, int OP, int V>
cudaError_t launch_axis_v(const argr_plan& p, const Problem& pr) {
    return p.unroll == 8 ? launch_axis_vu<Tag, OP, V, 8>(p, pr) : launch_axis_vu<Tag, OP, V, 4>(p, pr);
}

template <class Tag, int OP>
cudaError_t launch_axis_op(const argr_plan& p, const Problem& pr) {
    constexpr int VV = sizeof(typename Tag::raw) == 8 ? 2 : 4;
    return p.vec ? launch_axis_v<Tag, OP, VV>(p, pr) : launch_axis_v<Tag, OP, 1>(p, pr);
}

template <class Tag>
cudaError_t launch_axis_t(const argr_plan& p, const Problem& pr) {
    switch (pr.op) {
        case kOpMax: return launch_axis_op<Tag, kOpMax>(p, pr);
        case kOpMin: return launch_axis_op<Tag, kOpMin>(p, pr);
        case kOpMaxLast: return launch_axis_op<Tag, kOpMaxLast>(p, pr);
        case kOpMinLast: return launch_axis_op<Tag, kOpMinLast>(p, pr);
        default: return cudaErrorInvalidValue;
    }
}

// The device error word of this translation unit: read it, then clear it.
static inline cudaError_t read_and_clear_error_t(unsigned* out) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    *out = v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace argr

#define ARGR_DEFINE_LAUNCHERS(sfx, Tag)                                                                       \
    namespace argr {                                                                                          \
    cudaError_t launch_rows_##sfx(const argr_plan& p, const Problem& pr) { return launch_rows_t<Tag>(p, pr); } \
    cudaError_t launch_split_##sfx(const argr_plan& p, const Problem& pr) {                                  \
        return launch_split_t<Tag>(p, pr);                                                                    \
    }                                                                                                         \
    cudaError_t launch_cluster_##sfx(const argr_plan& p, const Problem& pr) {                                \
        return launch_cluster_t<Tag>(p, pr);                                                                  \
    }                                                                                                         \
    cudaError_t launch_stream_##sfx(const argr_plan& p, const Problem& pr) {                                 \
        return launch_stream_t<Tag>(p, pr);                                                                   \
    }                                                                                                         \
    cudaError_t read_and_clear_error_##sfx(unsigned* out) { return read_and_clear_error_t(out); }           \
    }

// The non-last-axis launcher lives in its own translation unit per type.
#define ARGR_DEFINE_AXIS_LAUNCHER(sfx, Tag)                                                                  \
    namespace argr {                                                                                          \
    cudaError_t launch_axis_##sfx(const argr_plan& p, const Problem& pr) { return launch_axis_t<Tag>(p, pr); } \
    }
