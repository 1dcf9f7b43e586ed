/*
 * What raises the shared-load bank-conflict counter of the row pipelines?
 *
 * Each kernel has the same seven reader warps per CTA issue conflict-free
 * 16-byte shared loads (lane l reads bytes [16 l, 16 l + 16) of a 512-byte
 * window, 4 wavefronts per warp instruction). Warp 0 adds one kind of other
 * traffic:
 *   lds_only                      nothing
 *   lds_with_global_stores        st.global.cs.v4, 512 contiguous bytes per warp
 *                                 instruction, 128-byte aligned
 *   lds_with_global_stores_off16  the same 16 bytes off a 128-byte boundary
 *                                 (as the unaligned rows' bodies)
 *   lds_with_global_loads         ld.global.nc.L1::no_allocate.v4
 *   lds_with_bulk_copies          cp.async.bulk global -> shared, 16 KB each,
 *                                 two buffers on mbarriers
 * Under ncu, compare l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum
 * across the kernels: the readers' own pattern has none.
 *
 * Build and run (one GPU):
 *   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o smem_conflict_probe tests/native/smem_conflict_probe.cu
 *   ./smem_conflict_probe
 * Every wait on an mbarrier is bounded; a wait that runs out sets an error flag
 * and the program exits 1.
 */
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

namespace {

constexpr int kThreads = 256;         // warp 0: other traffic; warps 1-7: readers
constexpr int kReadIters = 2048;      // 16-byte shared loads per reader thread
constexpr int kStoreIters = 1024;     // 512-byte warp accesses of warp 0
constexpr size_t kSpan = size_t(1) << 20;  // global bytes per CTA
constexpr int kCopyBytes = 16384;     // per bulk copy
constexpr int kCopies = 256;          // bulk copies per CTA
constexpr int kCopySmem = 2 * kCopyBytes + 128;  // two buffers + alignment slack
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ bool try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t n = 0; n < kSpinLimit; ++n)
        if (try_wait(bar, parity)) return true;
    return false;
}

// the readers' loop: conflict-free 16-byte loads from a 4 KB table
__device__ __forceinline__ float read_loop(const float* table) {
    float acc = 0.f;
    const int t = threadIdx.x - 32;
    for (int i = 0; i < kReadIters; ++i) {
        float a, b, c, d;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
                     : "r"(smem_u32(table + 4 * ((t + i) & 255))));
        acc += a + b + c + d;
    }
    return acc;
}

// MODE 0: no other traffic; 1: global stores; 2: global loads (OFF: byte offset)
template <int MODE, int OFF>
__device__ __forceinline__ void global_mix(char* g, float* out) {
    __shared__ __align__(16) float table[1024];
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) table[i] = float(i);
    __syncthreads();
    if (threadIdx.x >= 32) {
        out[blockIdx.x * blockDim.x + threadIdx.x] = read_loop(table);
        return;
    }
    char* base = g + size_t(blockIdx.x) * kSpan + OFF;
    float acc = 0.f;
    for (int i = 0; i < kStoreIters; ++i) {
        // 16-byte aligned offsets below kSpan - 1024, so OFF + 16 bytes stay in the CTA's span
        char* q = base + (size_t(i) * 512 + threadIdx.x * 16) % (kSpan - 1024);
        if (MODE == 1) {
            asm volatile("st.global.cs.v4.f32 [%0], {%1, %1, %1, %1};" ::"l"(q), "f"(float(i)) : "memory");
        } else if (MODE == 2) {
            float a, b, c, d;
            asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
                         : "l"(q));
            acc += a + b + c + d;
        }
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

__global__ void __launch_bounds__(kThreads) lds_only(char* g, float* out) { global_mix<0, 0>(g, out); }
__global__ void __launch_bounds__(kThreads) lds_with_global_stores(char* g, float* out) { global_mix<1, 0>(g, out); }
__global__ void __launch_bounds__(kThreads) lds_with_global_stores_off16(char* g, float* out) {
    global_mix<1, 16>(g, out);
}
__global__ void __launch_bounds__(kThreads) lds_with_global_loads(char* g, float* out) { global_mix<2, 0>(g, out); }

__global__ void __launch_bounds__(kThreads) lds_with_bulk_copies(const char* src, float* out, unsigned* err) {
    extern __shared__ __align__(128) char raw[];
    __shared__ __align__(16) float table[1024];
    __shared__ __align__(8) uint64_t bar[2];
    char* buf = raw + ((128u - (smem_u32(raw) & 127u)) & 127u);  // 128-byte aligned, 2 x kCopyBytes
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) table[i] = float(i);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[0])));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[1])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x >= 32) {
        out[blockIdx.x * blockDim.x + threadIdx.x] = read_loop(table);
        return;
    }
    if (threadIdx.x != 0) return;
    int issued = 0;
    for (int c = 0; c < kCopies; ++c) {
        const int s = c & 1;
        // buffer s's previous copy (use (c >> 1) - 1 of that barrier) must have landed
        if (c >= 2 && !wait_bounded(&bar[s], uint32_t(((c >> 1) - 1) & 1))) {
            atomicExch(err, 1u);
            break;
        }
        const char* from = src + size_t((blockIdx.x * kCopies + c) % 4096) * kCopyBytes;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bar[s])),
                     "r"(kCopyBytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_u32(buf + s * kCopyBytes)),
            "l"(from), "r"(kCopyBytes), "r"(smem_u32(&bar[s]))
            : "memory");
        issued = c + 1;
    }
    // the last copy into each buffer lands before the CTA exits
    for (int c = issued - 2; c < issued; ++c)
        if (c >= 0 && !wait_bounded(&bar[c & 1], uint32_t((c >> 1) & 1))) atomicExch(err, 2u);
}

}  // namespace

int main() {
    const int blocks = 152 * 4;
    char* g = nullptr;
    float* out = nullptr;
    unsigned* err = nullptr;
    const size_t gbytes = size_t(blocks) * kSpan;  // >= 4096 * kCopyBytes for the bulk-copy source
    if (cudaMalloc(&g, gbytes) != cudaSuccess || cudaMalloc(&out, size_t(blocks) * kThreads * 4) != cudaSuccess ||
        cudaMalloc(&err, 4) != cudaSuccess) {
        fprintf(stderr, "allocation failed\n");
        return 1;
    }
    cudaMemset(g, 1, gbytes);
    cudaMemset(err, 0, 4);
    cudaFuncSetAttribute(lds_with_bulk_copies, cudaFuncAttributeMaxDynamicSharedMemorySize, kCopySmem);
    lds_only<<<blocks, kThreads>>>(g, out);
    lds_with_global_stores<<<blocks, kThreads>>>(g, out);
    lds_with_global_stores_off16<<<blocks, kThreads>>>(g, out);
    lds_with_global_loads<<<blocks, kThreads>>>(g, out);
    lds_with_bulk_copies<<<blocks, kThreads, kCopySmem>>>(g, out, err);
    const cudaError_t e = cudaDeviceSynchronize();
    unsigned h = 0;
    cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
    printf("smem_conflict_probe: %s, wait flag %u\n", cudaGetErrorString(e), h);
    cudaFree(g);
    cudaFree(out);
    cudaFree(err);
    return (e == cudaSuccess && h == 0) ? 0 : 1;
}
