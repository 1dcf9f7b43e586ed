// Fused LayerNorm -> affine -> tanh-approximation GELU kernels.
//
// Definition [PyTorch 自定义 CUDA 算子与 Triton 编程 §三 _layer_norm_gelu_kernel;
// Triton Kernel 实现练习 §4.1 LayerNorm]: mean = sum(x)/N, var = sum((x-mean)^2)/N,
// z = (x - mean) / sqrt(var + eps) * w + b, y = 0.5 z (1 + tanh(k0 (z + k1 z^3)))
// with k0 = 0.79788456, k1 = 0.044715 [CS336 Kernels, Triton notes "Triton
// GeLU"]. The row stays in registers between the two reductions (the variance
// is taken over the centred values, padding excluded), so x is read from HBM
// once; w and b are staged once per CTA in shared memory as fp32.
#pragma once

#include "rowops_device.cuh"

namespace rowops {

// 0.5 z (1 + tanh(u)) = z * sigmoid(2u) = z / (1 + exp(-2u)), u = k0 (z + k1 z^3).
// exp(-2u) = 2^(z (c0 + c1 z^2)) with c0 = -2 k0 log2(e), c1 = c0 k1. For z -> -inf
// the exponential overflows to +inf and the result is -0; for z -> +inf it is z.
// This is the tanh form itself, rearranged so that nothing cancels or overflows
// to NaN (the pages' (e^{2u} - 1) / (e^{2u} + 1) gives inf/inf for large u).
__device__ __forceinline__ float gelu_tanh_approx(float z) {
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    const float a = fmaf(c1, z * z, c0) * z;
    return z * rcp_approx(1.f + ex2_approx(a));
}

// Exact GELU ["Triton Kernel 实现练习" §3.4]: z Phi(z), Phi(z) = 0.5 (1 + erf(z /
// sqrt(2))). Evaluated in the shape of the tanh form above, Phi(z) ~ 1 / (1 +
// exp(-P(z))), with P an odd polynomial of degree 13 instead of 3: c_k are the
// minimax fit of the GELU's absolute error over |z| <= 8 (printed by
// row_wise_reduction_gb300/gelu_erf_fit.py; P increasing beyond, so the limits
// z -> +-inf are those of GELU). The fit is within 7e-8 of z Phi(z); the fp32
// evaluation adds the same kind of rounding as the tanh form (its exp2
// argument |z| (2.3 + 0.105 z^2) carries a relative error of ~2^-24). One exp2
// and one reciprocal per value, like the tanh form: an erfc approximation needs
// a reciprocal and an exponential as well and a longer polynomial, and these
// kernels are bound by issue when they take the exact form.
// exp(-P(z)) = 2^(z q(z^2)), q_k = -log2(e) c_k.
struct GeluErfFit {
    static constexpr double c0 = 1.595768432225e+00, c1 = 7.266856705396e-02, c2 = -6.626000741970e-05,
                            c3 = -1.104803108419e-04, c4 = 7.938218056236e-06, c5 = -2.668927628528e-07,
                            c6 = 3.611231485973e-09;
    static constexpr float q0 = float(-kLog2e * c0), q1 = float(-kLog2e * c1), q2 = float(-kLog2e * c2),
                           q3 = float(-kLog2e * c3), q4 = float(-kLog2e * c4), q5 = float(-kLog2e * c5),
                           q6 = float(-kLog2e * c6);
};

__device__ __forceinline__ float gelu_erf(float z) {
    using F = GeluErfFit;
    const float z2 = z * z;
    float q = fmaf(z2, F::q6, F::q5);
    q = fmaf(z2, q, F::q4);
    q = fmaf(z2, q, F::q3);
    q = fmaf(z2, q, F::q2);
    q = fmaf(z2, q, F::q1);
    q = fmaf(z2, q, F::q0);
    return z * rcp_approx(1.f + ex2_approx(q * z));
}

// The GELU of the fused kernels: exact (ERF) or the tanh approximation.
template <bool ERF>
__device__ __forceinline__ float gelu_of(float z) {
    if constexpr (ERF) return gelu_erf(z);
    else return gelu_tanh_approx(z);
}

// The same two functions on a pair of values with packed fp32 arithmetic (the
// same operations per value, half the instructions).
__device__ __forceinline__ float2 gelu_tanh_approx2(float2 z) {
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    const float2 a = f2_mul(f2_fma(f2(c1), f2_mul(z, z), f2(c0)), z);
    const float2 d = f2_add(make_float2(ex2_approx(a.x), ex2_approx(a.y)), f2(1.f));
    return f2_mul(z, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

__device__ __forceinline__ float2 gelu_erf2(float2 z) {
    using F = GeluErfFit;
    const float2 z2 = f2_mul(z, z);
    float2 q = f2_fma(z2, f2(F::q6), f2(F::q5));
    q = f2_fma(z2, q, f2(F::q4));
    q = f2_fma(z2, q, f2(F::q3));
    q = f2_fma(z2, q, f2(F::q2));
    q = f2_fma(z2, q, f2(F::q1));
    q = f2_fma(z2, q, f2(F::q0));
    const float2 a = f2_mul(q, z);
    const float2 d = f2_add(make_float2(ex2_approx(a.x), ex2_approx(a.y)), f2(1.f));
    return f2_mul(z, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

template <bool ERF>
__device__ __forceinline__ float2 gelu_of2(float2 z) {
    if constexpr (ERF) return gelu_erf2(z);
    else return gelu_tanh_approx2(z);
}

// Shared-memory staging of w, b as fp32 (absent -> 1, 0). `sw` and `sb` hold
// round_up(N, 4) floats each.
template <typename T>
__device__ __forceinline__ void stage_affine(const T* w, const T* b, int N, float* sw, float* sb) {
    using E = Elem<T>;
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        sw[j] = w ? E::load(w + j) : 1.f;
        sb[j] = b ? E::load(b + j) : 0.f;
    }
}

__host__ __device__ constexpr int affine_pad(int n) { return (n + 3) & ~3; }

// Unaligned rows: (w, b) as fp32 pairs in column order with one unused pair
// after every 8 columns (column c at pair c + c / 8). A warp's threads read
// column c0 + V*v + j of their vectors v, pair 9v + const: 32 different bank
// pairs for any c0, where plain column order gives an 8-way conflict.
__device__ __forceinline__ int affine_pair(int c) { return c + (c >> 3); }

template <typename T>
__device__ __forceinline__ void stage_affine_pairs(const T* w, const T* b, int N, float2* swb) {
    using E = Elem<T>;
    for (int c = threadIdx.x; c < N; c += blockDim.x)
        swb[affine_pair(c)] = make_float2(w ? E::load(w + c) : 1.f, b ? E::load(b + c) : 0.f);
}

// ALIGNED: every row starts on a 16-byte boundary (head = 0), so the columns of
// a vector are a multiple of 4 and w, b are read from shared memory as float4.
// DIRECT (ALIGNED only; w, b 16-byte aligned or absent): no staging; each
// thread loads the w, b vectors of its columns from global memory where it
// uses them (L1 hits after the SM's first row group). For launches where a CTA
// takes one or two row groups, the staging (a shared-memory fill and a CTA
// barrier before the first load of x) is a large share of its critical path.
template <typename T, int TPR, int VPT, int BLOCK, bool ALIGNED, bool ERF = false, bool DIRECT = false>
__global__ void __launch_bounds__(BLOCK)
    ln_gelu_reg_kernel(const T* x, T* y, const T* w, const T* b, float eps, int64_t M, int N,
                       int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int ROWS = BLOCK / TPR;
    static_assert(BLOCK % TPR == 0 && TPR >= 16, "row group must be at least a half warp");
    static_assert(ALIGNED || !DIRECT, "direct w, b loads need 16-byte vectors of columns");
    extern __shared__ float4 smem_affine[];
    float* sw = reinterpret_cast<float*>(smem_affine);
    float* sb = sw + affine_pad(N);
    __shared__ float red_a[BLOCK / 32 > 0 ? BLOCK / 32 : 1];
    __shared__ float red_b[BLOCK / 32 > 0 ? 2 * BLOCK / 32 : 2];

    const float2* swb = reinterpret_cast<const float2*>(smem_affine);
    if constexpr (!DIRECT) {
        if constexpr (ALIGNED) stage_affine(w, b, N, sw, sb);
        else stage_affine_pairs(w, b, N, reinterpret_cast<float2*>(smem_affine));
        __syncthreads();
    }

    const int t = threadIdx.x % TPR;
    const int slot = threadIdx.x / TPR;
    const int64_t ngroups = (M + ROWS - 1) / ROWS;
    // 1/N once instead of three divisions per row (the mean's rounding is
    // taken out by the residual either way); arithmetic on packed fp32 pairs
    const float inv_n = 1.f / float(N);

    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const int64_t row = g * ROWS + slot;
        const bool live = row < M;
        const T* xr = x + (live ? row : 0) * ld;
        T* yr = y + (live ? row : 0) * ld;
        RowGeom geo = row_geometry<T>(xr, N);
        if (!live) geo = RowGeom{0, 0, 0};
        const T* xv = xr + geo.head;
        T* yv = yr + geo.head;

        uint4 raw[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) raw[i] = ld_stream16(xv + k * V);
        }
        const bool has_ex = t < geo.extras();
        const int ecol = has_ex ? int(extra_col(geo, t, V)) : 0;
        float ex = has_ex ? E::load(xr + ecol) : 0.f;

        // mean (padding contributes 0)
        float v[VPT][V];
        float2 s2 = make_float2(ex, 0.f);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                E::unpack(raw[i], v[i]);
            } else {
#pragma unroll
                for (int j = 0; j < V; ++j) v[i][j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < V; j += 2) s2 = f2_add(s2, make_float2(v[i][j], v[i][j + 1]));
        }
        const float s = group_reduce<TPR>(s2.x + s2.y, red_a, OpSum());
        const float mean = s * inv_n;

        // variance of the centred values; padding stays out of it. The fp32
        // mean carries a rounding error of order |mean| 2^-24; the residual
        // r = sum(x - mean) measures it, delta = r / N, so that
        // x - true mean = (x - mean) - delta and var = q / N - delta^2.
        float2 q2 = f2(0.f), r2 = f2(0.f);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            const bool ok = k < geo.nvec;
#pragma unroll
            for (int j = 0; j < V; j += 2) {
                float2 d = f2_add(make_float2(v[i][j], v[i][j + 1]), f2(-mean));
                if (!ok) d = f2(0.f);
                v[i][j] = d.x;
                v[i][j + 1] = d.y;
                q2 = f2_fma(d, d, q2);
                r2 = f2_add(r2, d);
            }
        }
        float q = q2.x + q2.y, r = r2.x + r2.y;
        ex = has_ex ? ex - mean : 0.f;
        q = fmaf(ex, ex, q);
        r += ex;
        group_reduce_sum2<TPR>(q, r, red_b);
        const float delta = r * inv_n;
        const float rstd = rsqrtf(fmaxf(q * inv_n - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;  // (x - mean - delta) * rstd = fma(x - mean, rstd, shift)

        // affine + GELU + store
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                const int c0 = geo.head + int(k) * V;
                float o[V];
                if constexpr (DIRECT) {
                    float wf[V], bf[V];
                    if (w) {
                        E::unpack(__ldg(reinterpret_cast<const uint4*>(w + c0)), wf);
                    } else {
#pragma unroll
                        for (int j = 0; j < V; ++j) wf[j] = 1.f;
                    }
                    if (b) {
                        E::unpack(__ldg(reinterpret_cast<const uint4*>(b + c0)), bf);
                    } else {
#pragma unroll
                        for (int j = 0; j < V; ++j) bf[j] = 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < V; j += 2) {
                        const float2 z = f2_fma(make_float2(v[i][j], v[i][j + 1]), f2(rstd), f2(shift));
                        const float2 g = gelu_of2<ERF>(
                            f2_fma(z, make_float2(wf[j], wf[j + 1]), make_float2(bf[j], bf[j + 1])));
                        o[j] = g.x;
                        o[j + 1] = g.y;
                    }
                } else if constexpr (ALIGNED) {
#pragma unroll
                    for (int j = 0; j < V; j += 4) {
                        const float4 ww = *reinterpret_cast<const float4*>(sw + c0 + j);
                        const float4 bb = *reinterpret_cast<const float4*>(sb + c0 + j);
                        const float2 z0 = f2_fma(make_float2(v[i][j], v[i][j + 1]), f2(rstd), f2(shift));
                        const float2 z1 = f2_fma(make_float2(v[i][j + 2], v[i][j + 3]), f2(rstd), f2(shift));
                        const float2 g0 = gelu_of2<ERF>(f2_fma(z0, make_float2(ww.x, ww.y), make_float2(bb.x, bb.y)));
                        const float2 g1 = gelu_of2<ERF>(f2_fma(z1, make_float2(ww.z, ww.w), make_float2(bb.z, bb.w)));
                        o[j + 0] = g0.x;
                        o[j + 1] = g0.y;
                        o[j + 2] = g1.x;
                        o[j + 3] = g1.y;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < V; j += 2) {
                        const float2 wb0 = swb[affine_pair(c0 + j)], wb1 = swb[affine_pair(c0 + j + 1)];
                        const float2 z = f2_fma(make_float2(v[i][j], v[i][j + 1]), f2(rstd), f2(shift));
                        const float2 g = gelu_of2<ERF>(f2_fma(z, make_float2(wb0.x, wb1.x), make_float2(wb0.y, wb1.y)));
                        o[j] = g.x;
                        o[j + 1] = g.y;
                    }
                }
                st_stream16(yv + k * V, E::pack(o));
            }
        }
        if (has_ex) {
            const float2 wb = DIRECT    ? make_float2(w ? E::load(w + ecol) : 1.f, b ? E::load(b + ecol) : 0.f)
                              : ALIGNED ? make_float2(sw[ecol], sb[ecol])
                                        : swb[affine_pair(ecol)];
            E::store(yr + ecol, gelu_of<ERF>(fmaf(fmaf(ex, rstd, shift), wb.x, wb.y)));
        }
    }
}

// One CTA per row, any N. Pass 1: shifted sums around the row's first entry,
// S1 = sum(x - x0), S2 = sum((x - x0)^2), so mean = x0 + S1/N and
// var = S2/N - (S1/N)^2 without cancellation for rows whose mean is far from 0.
// Pass 2 re-reads x and writes y; w and b come from global memory (L1/L2).
// `scalar`: x and y rows differ in their offset modulo 16 bytes; one element
// at a time.
template <typename T, int BLOCK, int UNROLL, bool ERF = false>
__global__ void __launch_bounds__(BLOCK)
    ln_gelu_looped_kernel(const T* x, T* y, const T* w, const T* b, float eps, int64_t M, int64_t N,
                          int64_t ld, bool scalar) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    __shared__ float red_a[2][BLOCK / 32];
    __shared__ float red_b[2][BLOCK / 32];
    const int t = threadIdx.x;
    int parity = 0;
    const float fN = float(N);

    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, parity ^= 1) {
        const T* xr = x + row * ld;
        T* yr = y + row * ld;
        const RowGeom geo = scalar ? RowGeom{0, 0, 0} : row_geometry<T>(xr, N);
        const T* xv = xr + geo.head;
        T* yv = yr + geo.head;
        const float x0 = E::load(xr);

        float s1 = 0.f, s2 = 0.f;
        if (scalar) {
            for (int64_t c = t; c < N; c += BLOCK) {
                const float d = E::load(xr + c) - x0;
                s1 += d;
                s2 = fmaf(d, d, s2);
            }
        }
        if (t < geo.extras()) {
            const float d = E::load(xr + extra_col(geo, t, V)) - x0;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
        for (int64_t k0 = t; k0 < geo.nvec; k0 += int64_t(BLOCK) * UNROLL) {
            uint4 raw[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t k = k0 + int64_t(u) * BLOCK;
                if (k < geo.nvec) raw[u] = ld_stream16(xv + k * V);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t k = k0 + int64_t(u) * BLOCK;
                if (k < geo.nvec) {
                    float f[V];
                    E::unpack(raw[u], f);
#pragma unroll
                    for (int j = 0; j < V; ++j) {
                        const float d = f[j] - x0;
                        s1 += d;
                        s2 = fmaf(d, d, s2);
                    }
                }
            }
        }
        s1 = group_reduce<BLOCK>(s1, red_a[parity], OpSum());
        s2 = group_reduce<BLOCK>(s2, red_b[parity], OpSum());
        const float m1 = s1 / fN;
        const float mean = x0 + m1;
        const float var = fmaxf(s2 / fN - m1 * m1, 0.f);
        const float rstd = rsqrtf(var + eps);

        auto affine_gelu = [&](float xv_, int64_t c) {
            const float wj = w ? E::load(w + c) : 1.f;
            const float bj = b ? E::load(b + c) : 0.f;
            return gelu_of<ERF>(fmaf((xv_ - mean) * rstd, wj, bj));
        };
        if (scalar)
            for (int64_t c = t; c < N; c += BLOCK) E::store(yr + c, affine_gelu(E::load(xr + c), c));
        if (t < geo.extras()) {
            const int64_t c = extra_col(geo, t, V);
            E::store(yr + c, affine_gelu(E::load(xr + c), c));
        }
        for (int64_t k0 = t; k0 < geo.nvec; k0 += int64_t(BLOCK) * UNROLL) {
            uint4 raw[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t k = k0 + int64_t(u) * BLOCK;
                if (k < geo.nvec) raw[u] = ld_stream16(xv + k * V);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t k = k0 + int64_t(u) * BLOCK;
                if (k < geo.nvec) {
                    float f[V];
                    E::unpack(raw[u], f);
                    const int64_t c0 = geo.head + k * V;
#pragma unroll
                    for (int j = 0; j < V; ++j) f[j] = affine_gelu(f[j], c0 + j);
                    st_stream16(yv + k * V, E::pack(f));
                }
            }
        }
    }
}

}  // namespace rowops
