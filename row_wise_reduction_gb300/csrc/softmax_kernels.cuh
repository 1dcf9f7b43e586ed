// Stable row softmax kernels.
//
// Definition [Triton Kernel 实现练习 §2.4; CS336 Kernels, Triton notes "Triton
// Softmax（单行 reduction）"]: m = max_j x_j, y_j = exp(x_j - m) / sum_k exp(x_k - m).
// The pages run one Triton program per row with the whole row padded to a
// power of two. Here a row is owned by a group of TPR threads (a half warp up
// to a whole 1024-thread CTA), each holding VPT 16-byte vectors of the row in
// registers, so x is read from HBM once and y written once; the CTA loops over
// row groups (persistent grid, no partial last wave). Rows too long for
// registers take the looped kernel: an in-CTA online (m, d) pass over the row
// [第 6 讲 §7.2 Online Softmax] and a second pass that writes y.
#pragma once

#include "rowops_device.cuh"

namespace rowops {

// exp(x - m) as 2^((x - m) log2 e). The difference is taken first: folding m
// into an FMA as x log2e - m log2e would round m log2e at the scale of m, which
// for |m| ~ 1e4 is already a 3e-4 relative error in the result.
__device__ __forceinline__ float exp_shifted(float x, float m) { return ex2_approx((x - m) * kLog2eF); }

// 1 / d, with a row of no unmasked entry (d = 0) mapped to 0 and NaN kept
__device__ __forceinline__ float safe_inverse(float d) {
    return d > 0.f ? 1.f / d : (d == 0.f ? 0.f : d);
}

template <typename T, int TPR, int VPT, int BLOCK>
__global__ void __launch_bounds__(BLOCK)
    softmax_reg_kernel(const T* x, T* y, int64_t M, int N, int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int ROWS = BLOCK / TPR;
    static_assert(BLOCK % TPR == 0 && TPR >= 16, "row group must be at least a half warp");
    __shared__ float red_max[BLOCK / 32 > 0 ? BLOCK / 32 : 1];
    __shared__ float red_sum[BLOCK / 32 > 0 ? BLOCK / 32 : 1];

    const int t = threadIdx.x % TPR;
    const int slot = threadIdx.x / TPR;
    const int64_t ngroups = (M + ROWS - 1) / ROWS;

    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const int64_t row = g * ROWS + slot;
        const bool live = row < M;
        const T* xr = x + (live ? row : 0) * ld;
        T* yr = y + (live ? row : 0) * ld;
        RowGeom geo = row_geometry<T>(xr, N);
        if (!live) geo = RowGeom{0, 0, 0};
        const T* xv = xr + geo.head;
        T* yv = yr + geo.head;

        // load: all VPT vectors in flight before any use
        uint4 raw[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) raw[i] = ld_stream16(xv + k * V);
        }
        const bool has_ex = t < geo.extras();
        const int64_t ecol = has_ex ? extra_col(geo, t, V) : 0;
        float ex = has_ex ? E::load(xr + ecol) : -INFINITY;

        // row max (padding is -inf)
        float v[VPT][V];
        float mx = ex;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                E::unpack(raw[i], v[i]);
            } else {
#pragma unroll
                for (int j = 0; j < V; ++j) v[i][j] = -INFINITY;
            }
#pragma unroll
            for (int j = 0; j < V; ++j) mx = fmaxf(mx, v[i][j]);
        }
        mx = group_reduce<TPR>(mx, red_max, OpMax());
        if (mx == -INFINITY) mx = 0.f;  // no unmasked entry: every exp below is 0

        // sum of exp(x - m); the exponentials stay in registers
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
#pragma unroll
            for (int j = 0; j < V; ++j) {
                v[i][j] = exp_shifted(v[i][j], mx);
                s += v[i][j];
            }
        }
        ex = exp_shifted(ex, mx);
        s += ex;
        s = group_reduce<TPR>(s, red_sum, OpSum());
        const float inv = safe_inverse(s);

        // normalise and store
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                float o[V];
#pragma unroll
                for (int j = 0; j < V; ++j) o[j] = v[i][j] * inv;
                st_stream16(yv + k * V, E::pack(o));
            }
        }
        if (has_ex) E::store(yr + ecol, ex * inv);
    }
}

// One CTA per row, any N. Pass 1 folds the row into per-thread (m, d) states,
// UNROLL vectors at a time, and merges them across the CTA; pass 2 re-reads x
// and writes y. `scalar`: x and y rows sit at different offsets modulo 16
// bytes, so no 16-byte vector serves both; every element goes one at a time.
template <typename T, int BLOCK, int UNROLL>
__global__ void __launch_bounds__(BLOCK)
    softmax_looped_kernel(const T* x, T* y, int64_t M, int64_t N, int64_t ld, bool scalar) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    __shared__ float red_m[2][BLOCK / 32];
    __shared__ float red_d[2][BLOCK / 32];
    const int t = threadIdx.x;
    int parity = 0;

    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, parity ^= 1) {
        const T* xr = x + row * ld;
        T* yr = y + row * ld;
        const RowGeom geo = scalar ? RowGeom{0, 0, 0} : row_geometry<T>(xr, N);
        const T* xv = xr + geo.head;
        T* yv = yr + geo.head;

        MD s{-INFINITY, 0.f};
        if (scalar)
            for (int64_t c = t; c < N; c += BLOCK) s = md_push(s, E::load(xr + c));
        if (t < geo.extras()) s = md_push(s, E::load(xr + extra_col(geo, t, V)));
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
                    float vm = f[0];
#pragma unroll
                    for (int j = 1; j < V; ++j) vm = fmaxf(vm, f[j]);
                    if (vm == -INFINITY) continue;  // all masked
                    if (vm > s.m) {
                        s.d *= ex2_approx((s.m - vm) * kLog2eF);
                        s.m = vm;
                    }
#pragma unroll
                    for (int j = 0; j < V; ++j) s.d += exp_shifted(f[j], s.m);
                }
            }
        }
        s = group_merge<BLOCK>(s, red_m[parity], red_d[parity]);
        const float m = s.d > 0.f ? s.m : 0.f;
        const float inv = safe_inverse(s.d);

        if (scalar)
            for (int64_t c = t; c < N; c += BLOCK) E::store(yr + c, exp_shifted(E::load(xr + c), m) * inv);
        if (t < geo.extras()) {
            const int64_t c = extra_col(geo, t, V);
            E::store(yr + c, exp_shifted(E::load(xr + c), m) * inv);
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
                    for (int j = 0; j < V; ++j) f[j] = exp_shifted(f[j], m) * inv;
                    st_stream16(yv + k * V, E::pack(f));
                }
            }
        }
    }
}

// Causal softmax, any layout ["Triton Kernel 实现练习" §5.1 causal mask, §2.4
// softmax]: one CTA per row; row r keeps its first kept = clamp((r mod period)
// + offset + 1, 0, N) columns. Pass 1 folds the kept entries into a per-thread
// online (m, d) state (element-wise, coalesced), merged across the CTA; pass 2
// re-reads them and writes y, and writes 0 on the masked columns without
// reading them.
template <typename T, int BLOCK>
__global__ void __launch_bounds__(BLOCK)
    softmax_causal_looped_kernel(const T* x, T* y, int64_t M, int64_t N, int64_t ld, int64_t period,
                                 int64_t offset) {
    using E = Elem<T>;
    __shared__ float red_m[2][BLOCK / 32];
    __shared__ float red_d[2][BLOCK / 32];
    int parity = 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x, parity ^= 1) {
        int64_t kept = row % period + offset + 1;
        kept = kept < 0 ? 0 : (kept > N ? N : kept);
        const T* xr = x + row * ld;
        T* yr = y + row * ld;
        MD s{-INFINITY, 0.f};
        for (int64_t c = threadIdx.x; c < kept; c += BLOCK) s = md_push(s, E::load(xr + c));
        s = group_merge<BLOCK>(s, red_m[parity], red_d[parity]);
        const float m = s.d > 0.f ? s.m : 0.f;
        const float inv = safe_inverse(s.d);
        for (int64_t c = threadIdx.x; c < N; c += BLOCK)
            E::store(yr + c, c < kept ? exp_shifted(E::load(xr + c), m) * inv : 0.f);
    }
}

}  // namespace rowops
