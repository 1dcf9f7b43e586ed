// Elementwise GELU, exact or tanh approximation ["Triton Kernel 实现练习" §3.4
// Approx Activation: gelu_exact(x) = 0.5 x (1 + erf(x / sqrt(2))), gelu_approx
// with tanh(sqrt(2 / pi) (x + 0.044715 x^3))], on n contiguous elements: 16-byte
// vectors over the aligned body, the unaligned head and tail one element per
// thread; x and y at different offsets modulo 16 bytes go element by element.
#include "ln_gelu_kernels.cuh"
#include "rowops_launch.h"

namespace rowops {

template <typename T, bool ERF, int BLOCK>
__global__ void __launch_bounds__(BLOCK) gelu_kernel(const T* x, T* y, int64_t n, bool scalar) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    const int64_t tid = int64_t(blockIdx.x) * BLOCK + threadIdx.x;
    const int64_t nthreads = int64_t(gridDim.x) * BLOCK;
    if (scalar) {
        for (int64_t i = tid; i < n; i += nthreads) E::store(y + i, gelu_of<ERF>(E::load(x + i)));
        return;
    }
    const RowGeom geo = row_geometry<T>(x, n);
    if (tid < geo.extras()) {
        const int64_t c = extra_col(geo, int(tid), V);
        E::store(y + c, gelu_of<ERF>(E::load(x + c)));
    }
    const T* xv = x + geo.head;
    T* yv = y + geo.head;
    for (int64_t k = tid; k < geo.nvec; k += nthreads) {
        float v[V];
        E::unpack(ld_stream16(xv + k * V), v);
#pragma unroll
        for (int e = 0; e < V; ++e) v[e] = gelu_of<ERF>(v[e]);
        st_stream16(yv + k * V, E::pack(v));
    }
}

template <typename T, bool ERF>
cudaError_t launch_gelu(const void* x, void* y, int64_t n, const LaunchCfg& cfg) {
    constexpr int BLOCK = 256;
    auto kern = gelu_kernel<T, ERF, BLOCK>;
    const bool scalar = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) != 0;
    const int64_t work = scalar ? n : (n + Elem<T>::kVec - 1) / Elem<T>::kVec;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, 0, (work + BLOCK - 1) / BLOCK, cfg);
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), n, scalar);
    return cudaGetLastError();
}

GeluLaunch gelu_f32(bool erf) { return erf ? launch_gelu<float, true> : launch_gelu<float, false>; }
GeluLaunch gelu_bf16(bool erf) { return erf ? launch_gelu<bf16_t, true> : launch_gelu<bf16_t, false>; }

}  // namespace rowops
