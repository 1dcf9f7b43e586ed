// TMA-fed row pipeline: one CTA works on one row at a time while the next
// rows stream into a ring of shared-memory buffers.
//
// Thread 0 copies each whole row with one bulk asynchronous copy
// (cp.async.bulk, global -> shared, completion counted in bytes on an
// mbarrier). Every thread waits on the buffer's mbarrier, reads its own 16-byte
// vectors out of shared memory, and after the row's first CTA-wide reduction
// (by which point every thread holds its data in registers) thread 0 refills
// that buffer with the row `nbuf` iterations ahead. So `nbuf` rows per CTA are
// always in flight regardless of how long the arithmetic of the current row
// takes: the memory system never waits for the compute of a row.
//
// The bulk copy moves whole 16-byte vectors between 16-byte-aligned addresses,
// so it takes each row's aligned body; the kernels on the pipeline load the
// unaligned head and tail of a row themselves (tma_row_kernels.cuh).
//
// Waits are bounded (2 s unless the launch gives a shorter limit). If a
// buffer's copy has not landed in time, the thread records it; the row
// group's next barrier (bar.red.or) tells every thread of the group, the group
// stops processing rows, its producer waits (again bounded) for the copies it
// still has in flight and sets the library's device error word, and the group
// returns.
#pragma once

#include "rowops_device.cuh"

namespace rowops {

constexpr unsigned kDeviceErrTimeout = 5u;  // value of ROWOPS_ERR_TIMEOUT
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// make the initialised barriers visible to the async (copy) proxy
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity: false after `limit_ns`
// (or 2^26 polls, whichever comes first).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Thread 0: expect `bytes` (+ `extra`) on `bar`, then copy `bytes` global ->
// shared. A nonzero `extra` is the test hook that makes the phase never
// complete, so the bounded wait on it runs out (the copy itself completes).
__device__ __forceinline__ void tma_load_row(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                             uint32_t extra = 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes + extra)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// One plain arrival (no bytes): completes a phase that expects nothing else.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// The same in two steps, for several copies completing on one barrier: one
// expect of their total bytes, then each copy.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_copy_row(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Order this thread's earlier shared-memory reads before later async-proxy
// writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds16(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// One 16-byte shared-memory load of four floats, as an asm statement: issued
// whole and kept in program order with the ring's loads. The exact-GELU form
// reads its staged w, b this way (bf16 65536 x 8192 measured side by side:
// 405 -> 375 us); the tanh form keeps the compiler's own loads, which it
// schedules better there (330 us against 340).
__device__ __forceinline__ float4 ldsf4(const float4* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

// Row-group reductions for the pipeline kernels. A row is owned by the TPR
// threads of group g = threadIdx.x / TPR (TPR a multiple of 64); the group
// synchronises on its own named barrier 1 + g (0 is __syncthreads), so row
// groups of one CTA run independently. The barrier also ORs a per-thread
// failure flag across the group. `red` is the group's slice of TPR / 32 floats
// (2 * TPR / 32 for the two-value form).
__device__ __forceinline__ int group_bar_or(int id, int nthreads, int flag) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(flag), "r"(id), "r"(nthreads)
        : "memory");
    return r;
}

template <int TPR, class Op>
__device__ __forceinline__ float row_reduce(float v, float* red, int bar_id, Op op, int& fail) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    constexpr int W = TPR / 32;
    const int w = (threadIdx.x % TPR) >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    fail = group_bar_or(bar_id, TPR, fail);
    v = red[0];
#pragma unroll
    for (int i = 1; i < W; ++i) v = op(v, red[i]);
    return v;
}

template <int TPR>
__device__ __forceinline__ void row_reduce_sum2(float& a, float& b, float* red, int bar_id, int& fail) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    constexpr int W = TPR / 32;
    const int w = (threadIdx.x % TPR) >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[2 * w] = a;
        red[2 * w + 1] = b;
    }
    fail = group_bar_or(bar_id, TPR, fail);
    a = red[0];
    b = red[1];
#pragma unroll
    for (int i = 1; i < W; ++i) {
        a += red[2 * i];
        b += red[2 * i + 1];
    }
}

// row_reduce_sum2 on packed pairs: one add per butterfly step and per warp
// partial for both sums (the additions in the order of two separate sums), and
// two warps' partials per 16-byte load. `red`: 16-byte aligned, TPR / 32 pairs.
// (The row pipelines of the forward kernels keep the scalar form: at their
// register caps the packed one spilled and ran slower.)
template <int TPR>
__device__ __forceinline__ void row_reduce_sum2_packed(float& a, float& b, float2* red, int bar_id, int& fail) {
    float2 v = make_float2(a, b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = f2_add(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o)));
    constexpr int W = TPR / 32;
    static_assert(W % 2 == 0, "pairs of warps");
    const int w = (threadIdx.x % TPR) >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    fail = group_bar_or(bar_id, TPR, fail);
    const float4* r4 = reinterpret_cast<const float4*>(red);
    float4 q = r4[0];
    v = f2_add(make_float2(q.x, q.y), make_float2(q.z, q.w));
#pragma unroll
    for (int i = 1; i < W / 2; ++i) {
        q = r4[i];
        v = f2_add(f2_add(v, make_float2(q.x, q.y)), make_float2(q.z, q.w));
    }
    a = v.x;
    b = v.y;
}

// The ring: nbuf buffers of `row_bytes` (a multiple of 128) after the barriers.
struct RowRing {
    uint64_t* bar;    // nbuf mbarriers
    char* buf;        // nbuf * row_bytes
    uint32_t row_bytes;
    int nbuf;
    __device__ __forceinline__ char* slot(int s) const { return buf + size_t(s) * row_bytes; }
};

// Ring slot and phase parity of iteration i (i % nbuf and (i / nbuf) & 1),
// advanced one iteration at a time: the loops over rows would otherwise pay a
// 64-bit division by the run-time ring depth per row and thread.
struct RingCursor {
    int slot = 0;
    uint32_t parity = 0;
    __device__ __forceinline__ void next(int nbuf) {
        if (++slot == nbuf) {
            slot = 0;
            parity ^= 1u;
        }
    }
};

// Bytes of dynamic shared memory before the row buffers: the mbarriers of all
// row groups' rings (ROWS * nbuf <= 32), padded.
constexpr uint32_t kRingHeader = 256;
constexpr int kMaxRingBuffers = 16;

__host__ __device__ constexpr uint32_t ring_row_bytes(int64_t N, int es) {
    return uint32_t((N * es + 127) / 128 * 128);
}

// Thread 0, on an error exit: wait (bounded) for every copy still in flight so
// that none lands in shared memory after the CTA is gone.
__device__ __forceinline__ void drain_ring(const RowRing& ring, int64_t first_row_iter, int64_t row0,
                                           int64_t stride, int64_t M, unsigned long long limit_ns) {
    for (int d = 0; d < ring.nbuf; ++d) {
        const int64_t i = first_row_iter + d;
        const int64_t row = row0 + i * stride;
        if (row >= M) break;
        mbar_wait(ring.bar + (i % ring.nbuf), uint32_t((i / ring.nbuf) & 1), limit_ns);
    }
}

}  // namespace rowops
