// Tensor memory (TMEM) as per-thread scratch, through the tcgen05 PTX
// instructions of sm_100a / sm_103a.
//
// TMEM is 128 lanes x 512 columns of 32-bit cells per SM, outside the register
// file and shared memory. A CTA allocates a power-of-two number of columns
// (>= 32) with one warp, and that warp frees them before the CTA exits. The
// 32x32b access shape gives lane i of a warp TMEM lane (32 q + i), q = warp
// index mod 4, and n consecutive columns: for that warp a private array of n
// 32-bit values per thread, read and written with one instruction each.
#pragma once

#include <cstdint>

namespace rowops {

__device__ __forceinline__ uint32_t tmem_smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One whole warp: allocate `cols` columns and write their base address to *dst
// (shared memory); give up the right to allocate again, so that other CTAs on
// the SM are not held back.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_smem_addr(dst)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// The warp that allocated: free the columns (after every access has completed
// and a CTA barrier between them, fenced by tmem_fence_before / _after).
__device__ __forceinline__ void tmem_free(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// Order TMEM accesses and allocation around a thread barrier.
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Complete this thread's earlier stores.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Complete this thread's earlier loads. The registers a load wrote are passed
// through the wait as read-write operands, so the compiler cannot move their
// uses above it (the load's outputs are not valid until the wait).
template <int N>
__device__ __forceinline__ void tmem_wait_ld(float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_wait_ld<8>(float (&v)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7])
                 :
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_wait_ld<16>(float (&v)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                   "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]), "+f"(v[15])
                 :
                 : "memory");
}

// Whole warp: v[0..N) <- columns addr .. addr + N - 1 of this thread's lane
// (valid after tmem_wait_ld on v).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t addr, float (&v)[N]);
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t addr, const float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t addr, float (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "r"(addr)
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t addr, float (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]),
          "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(addr)
        : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<8>(uint32_t addr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(addr),
                 "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t addr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(addr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
        "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
        : "memory");
}

}  // namespace rowops
