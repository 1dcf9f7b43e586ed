// Elementwise GELU, exact or tanh approximation ["Triton Kernel 实现练习" §3.4
// Approx Activation: gelu_exact(x) = 0.5 x (1 + erf(x / sqrt(2))), gelu_approx
// with tanh(sqrt(2 / pi) (x + 0.044715 x^3))], on n contiguous elements: 16-byte
// vectors over the aligned body, the unaligned head and tail one element per
// thread; x and y at different offsets modulo 16 bytes go element by element.
// Also the fused residual + bias + GELU over rows.
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

// Fused residual + bias + GELU ["Triton Kernel 实现练习" §3.4, "fused residual +
// bias + GELU"]: y = GELU((x + b) + residual) in fp32, b per column, residual
// and b optional. One row per CTA iteration (grid-stride over rows). VEC: rows
// of x, residual and y 16-byte aligned, N a multiple of the vector, b 16-byte
// aligned: UNROLL 16-byte vectors of x and the residual in flight per thread,
// arithmetic on packed fp32 pairs; otherwise one element at a time.
template <typename T, bool ERF, int BLOCK, int UNROLL, bool VEC>
__global__ void __launch_bounds__(BLOCK)
    bias_residual_gelu_kernel(const T* x, const T* r, const T* b, T* y, int64_t M, int64_t N, int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    const int t = threadIdx.x;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const T* xr = x + row * ld;
        const T* rr = r ? r + row * ld : nullptr;
        T* yr = y + row * ld;
        if constexpr (VEC) {
            const int64_t nvec = N / V;
            for (int64_t k0 = t; k0 < nvec; k0 += int64_t(BLOCK) * UNROLL) {
                uint4 xa[UNROLL], ra[UNROLL];
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int64_t k = k0 + int64_t(u) * BLOCK;
                    if (k < nvec) {
                        xa[u] = ld_stream16(xr + k * V);
                        if (rr) ra[u] = ld_stream16(rr + k * V);
                    }
                }
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int64_t k = k0 + int64_t(u) * BLOCK;
                    if (k < nvec) {
                        float xv[V], rv[V], bv[V];
                        E::unpack(xa[u], xv);
                        if (rr) E::unpack(ra[u], rv);
                        if (b) E::unpack(*reinterpret_cast<const uint4*>(b + k * V), bv);
                        float o[V];
#pragma unroll
                        for (int e = 0; e < V; e += 2) {
                            float2 s = make_float2(xv[e], xv[e + 1]);
                            if (b) s = f2_add(s, make_float2(bv[e], bv[e + 1]));
                            if (rr) s = f2_add(s, make_float2(rv[e], rv[e + 1]));
                            const float2 g = gelu_of2<ERF>(s);
                            o[e] = g.x;
                            o[e + 1] = g.y;
                        }
                        st_stream16(yr + k * V, E::pack(o));
                    }
                }
            }
        } else {
            for (int64_t c = t; c < N; c += BLOCK) {
                float s = E::load(xr + c);
                if (b) s += E::load(b + c);
                if (rr) s += E::load(rr + c);
                E::store(yr + c, gelu_of<ERF>(s));
            }
        }
    }
}

template <typename T, bool ERF, bool VEC>
cudaError_t launch_brg(const void* x, const void* r, const void* b, void* y, int64_t M, int64_t N, int64_t ld,
                       const LaunchCfg& cfg) {
    constexpr int BLOCK = 256, UNROLL = 4;
    auto kern = bias_residual_gelu_kernel<T, ERF, BLOCK, UNROLL, VEC>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, 0, M, cfg);
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(r),
                                         static_cast<const T*>(b), static_cast<T*>(y), M, N, ld);
    return cudaGetLastError();
}

template <typename T>
BiasResidualGeluLaunch brg_table(bool erf, bool vec) {
    if (vec) return erf ? launch_brg<T, true, true> : launch_brg<T, false, true>;
    return erf ? launch_brg<T, true, false> : launch_brg<T, false, false>;
}

BiasResidualGeluLaunch bias_residual_gelu_f32(bool erf, bool vec) { return brg_table<float>(erf, vec); }
BiasResidualGeluLaunch bias_residual_gelu_bf16(bool erf, bool vec) { return brg_table<bf16_t>(erf, vec); }

}  // namespace rowops
