// Split-row online softmax with the chunks streamed through a shared-memory
// ring [Triton Kernel 实现练习 §2.5 split_online_softmax; 第 6 讲 §7.2 Online
// Softmax]. The same two passes as online_softmax_kernels.cuh (partials, then
// merge + normalise), but each CTA keeps `nbuf` chunks in flight by bulk
// asynchronous copies (cp.async.bulk, completion counted on one mbarrier per
// ring slot) instead of register loads, so the memory pipe stays busy while a
// chunk is reduced, merged or written.
//
// Work item k of a pass is chunk (k mod nchunks) of row k / nchunks; a chunk
// is exactly TPR * VPT 16-byte vectors (N a multiple of the chunk, rows
// 16-byte aligned). Thread t reads vectors t + j * TPR of a slot.
//   Pass 1: m_c = max over the chunk (NaN-propagating), d_c = sum exp(x - m_c)
//           (0 for a chunk of -inf only) -> partials[k].
//   Pass 2 (items in reverse order, so that its first chunks are the ones pass
//           1 read last, still in L2): thread q folds the row's partials q, q +
//           TPR, ..., two group reductions give m = max m_c (over d_c > 0) and
//           d = sum d_c exp(m_c - m) in one fixed order (the same for every
//           chunk of the row), y = exp(x - m) / d.
// A wait that gives up (bounded) is reported through the workspace status
// word after the CTA's copies in flight have landed.
//
// Pass 2 is launched as a programmatic dependent of pass 1: each pass-1 CTA
// signals once it has issued its last copy, so pass-2 CTAs start as pass-1
// CTAs leave and fill their rings with x (which pass 1 does not write); they
// wait for pass 1 to complete (griddepcontrol.wait) before reading a partial
// or writing y. Launched the ordinary way, the wait returns at once.
#pragma once

#include "online_softmax_kernels.cuh"
#include "reduce_kernels.cuh"
#include "row_pipeline.cuh"

namespace rowops {

__device__ __forceinline__ int64_t split_chunk_offset(int64_t item, int64_t nchunks, int64_t chunk, int64_t ld) {
    const int64_t r = item / nchunks;
    return r * ld + (item - r * nchunks) * chunk;
}

// Producer (thread 0): the copy of work item `item` into slot s.
template <typename T, int TPR, int VPT>
__device__ __forceinline__ void split_issue(const RowRing& ring, int s, int64_t item, const T* x, int64_t nchunks,
                                            int64_t ld, int64_t stall_row) {
    constexpr int64_t kChunk = int64_t(TPR) * VPT * Elem<T>::kVec;
    tma_load_row(ring.slot(s), x + split_chunk_offset(item, nchunks, kChunk, ld), uint32_t(TPR) * VPT * 16u,
                 ring.bar + s, stall_extra(item, stall_row));
}

// CTA start: barriers, then the first nbuf items of this CTA (iteration i is
// item `order(first + i * stride)`).
template <typename T, int TPR, int VPT, class Order>
__device__ __forceinline__ void split_start(const RowRing& ring, const T* x, int64_t items, int64_t nchunks,
                                            int64_t ld, int64_t stall_row, Order order) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ring.nbuf; ++s) mbar_init(ring.bar + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int s = 0; s < ring.nbuf; ++s) {
            const int64_t k = int64_t(blockIdx.x) + int64_t(s) * gridDim.x;
            if (k < items) split_issue<T, TPR, VPT>(ring, s, order(k), x, nchunks, ld, stall_row);
        }
}

// After iteration i's first group barrier every thread has read slot s: refill
// it with iteration i + nbuf.
template <typename T, int TPR, int VPT, class Order>
__device__ __forceinline__ void split_refill(const RowRing& ring, int s, int64_t i, const T* x, int64_t items,
                                             int64_t nchunks, int64_t ld, int64_t stall_row, Order order) {
    if (threadIdx.x != 0) return;
    const int64_t k = int64_t(blockIdx.x) + (i + ring.nbuf) * int64_t(gridDim.x);
    if (k < items) {
        fence_proxy_async_smem();  // the slot was last read through the generic proxy
        split_issue<T, TPR, VPT>(ring, s, order(k), x, nchunks, ld, stall_row);
    }
}

// Error exit: thread 0 waits (bounded) for the copies still in flight, then
// records the timeout in the workspace status word.
__device__ __forceinline__ void split_abandon(const RowRing& ring, int64_t i, int64_t items, unsigned* status,
                                              unsigned long long wait_ns) {
    if (threadIdx.x != 0) return;
    drain_ring(ring, i, blockIdx.x, gridDim.x, items, wait_ns);
    atomicExch(status, kDeviceErrTimeout);
}

struct SplitForward {
    __device__ __forceinline__ int64_t operator()(int64_t k) const { return k; }
};
struct SplitReverse {
    int64_t items;
    __device__ __forceinline__ int64_t operator()(int64_t k) const { return items - 1 - k; }
};

template <typename T, int TPR, int VPT>
__global__ void __launch_bounds__(TPR)
    split_partial_tma_kernel(const T* x, int64_t items, int64_t nchunks, int64_t ld, unsigned* status,
                             float2* partials, int nbuf, unsigned long long wait_ns, int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    static_assert(TPR % 64 == 0, "at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red[2][2][TPR / 32];
    const RowRing ring{reinterpret_cast<uint64_t*>(smem), smem + kRingHeader, uint32_t(TPR) * VPT * 16u, nbuf};
    const int t = threadIdx.x;
    if (blockIdx.x == 0 && t == 0) *status = 0u;
    const SplitForward order;
    split_start<T, TPR, VPT>(ring, x, items, nchunks, ld, stall_row, order);

    bool signalled = false;
    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t k = int64_t(blockIdx.x) + i * gridDim.x;
        if (k >= items) break;
        if (!signalled && k + int64_t(nbuf) * gridDim.x >= items) {  // no copy left to issue
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            signalled = true;
        }
        const int s = rc.slot;
        int fail = !mbar_wait(ring.bar + s, rc.parity, wait_ns);
        const char* sb = ring.slot(s);
        float v[VPT][V];
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            E::unpack(lds16(sb + size_t(t + j * TPR) * 16), v[j]);
#pragma unroll
            for (int e = 0; e < V; ++e) m = fmax_nan(m, v[j][e]);
        }
        m = row_reduce<TPR>(m, red[0][i & 1], 1, RowMax(), fail);
        if (fail) {
            split_abandon(ring, i, items, status, wait_ns);
            return;
        }
        split_refill<T, TPR, VPT>(ring, s, i, x, items, nchunks, ld, stall_row, order);
        float d = 0.f;
        if (m != -INFINITY) {
#pragma unroll
            for (int j = 0; j < VPT; ++j)
#pragma unroll
                for (int e = 0; e < V; ++e) d += exp_shifted(v[j][e], m);
        }
        d = row_reduce<TPR>(d, red[1][i & 1], 1, OpSum(), fail);
        if (t == 0) partials[order(k)] = make_float2(m, d);
    }
}

template <typename T, int TPR, int VPT>
__global__ void __launch_bounds__(TPR)
    split_normalise_tma_kernel(const T* x, T* y, int64_t items, int64_t nchunks, int64_t ld,
                               const float2* partials, unsigned* status, int nbuf, unsigned long long wait_ns,
                               int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int64_t kChunk = int64_t(TPR) * VPT * V;
    static_assert(TPR % 64 == 0, "at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red[2][2][TPR / 32];
    const RowRing ring{reinterpret_cast<uint64_t*>(smem), smem + kRingHeader, uint32_t(TPR) * VPT * 16u, nbuf};
    const int t = threadIdx.x;
    const SplitReverse order{items};
    split_start<T, TPR, VPT>(ring, x, items, nchunks, ld, stall_row, order);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // pass 1's partials are complete and visible

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t k = int64_t(blockIdx.x) + i * gridDim.x;
        if (k >= items) break;
        const int64_t item = order(k), r = item / nchunks;
        const int s = rc.slot;
        // this thread's share of the row's partials (issued before the wait)
        MD pm{-INFINITY, 0.f};
        for (int64_t q = t; q < nchunks; q += TPR) {
            const float2 pv = partials[r * nchunks + q];
            pm = md_merge(pm, MD{pv.x, pv.y});
        }
        int fail = !mbar_wait(ring.bar + s, rc.parity, wait_ns);
        const char* sb = ring.slot(s);
        float v[VPT][V];
#pragma unroll
        for (int j = 0; j < VPT; ++j) E::unpack(lds16(sb + size_t(t + j * TPR) * 16), v[j]);
        const float mr = row_reduce<TPR>(pm.d == 0.f ? -INFINITY : pm.m, red[0][i & 1], 1, OpMax(), fail);
        if (fail) {
            split_abandon(ring, i, items, status, wait_ns);
            return;
        }
        split_refill<T, TPR, VPT>(ring, s, i, x, items, nchunks, ld, stall_row, order);
        const float dr = row_reduce<TPR>(pm.d == 0.f ? 0.f : pm.d * ex2_approx((pm.m - mr) * kLog2eF),
                                         red[1][i & 1], 1, OpSum(), fail);
        const float mm = dr > 0.f ? mr : 0.f;
        const float inv = safe_inverse(dr);
        T* yc = y + split_chunk_offset(item, nchunks, kChunk, ld);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = exp_shifted(v[j][e], mm) * inv;
            st_stream16(yc + size_t(t + j * TPR) * V, E::pack(o));
        }
    }
}

}  // namespace rowops
