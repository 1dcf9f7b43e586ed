// Split-row online softmax [Triton Kernel 实现练习 §2.5 split_online_softmax;
// 第 6 讲 §7.2 Online Softmax].
//
// Each row is cut into chunks of `chunk` columns; work item i = r * nchunks + c
// is chunk c of row r. Pass 1 (split_partial_kernel): one CTA per item folds
// its chunk into a partial state (m_c, d_c) = (max, sum exp(x - m_c)) and
// stores it. Pass 2 (split_normalise_kernel): one CTA per item merges all
// partials of its row, m = max_c m_c, d = sum_c d_c exp(m_c - m) (partials with
// d_c = 0 skipped), in one fixed order so every chunk of a row gets the same
// (m, d), then writes y = exp(x - m) / d over its chunk. `scalar`: x and y
// rows differ in their offset modulo 16 bytes; one element at a time.
#pragma once

#include "softmax_kernels.cuh"

namespace rowops {

// Workspace layout (bytes): [0, 256) header, word 0 = status; then float2
// partials[M][nchunks].
constexpr size_t kWorkspaceHeader = 256;

template <typename T, int BLOCK, int UNROLL>
__global__ void __launch_bounds__(BLOCK)
    split_partial_kernel(const T* x, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                         int64_t nchunks, bool scalar, unsigned* status, float2* partials) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    __shared__ float red_m[2][BLOCK / 32];
    __shared__ float red_d[2][BLOCK / 32];
    const int t = threadIdx.x;
    if (blockIdx.x == 0 && t == 0) *status = 0u;
    int parity = 0;
    const int64_t items = M * nchunks;

    for (int64_t item = blockIdx.x; item < items; item += gridDim.x, parity ^= 1) {
        const int64_t r = item / nchunks, c = item - r * nchunks;
        const int64_t col0 = c * chunk;
        const int64_t n = (N - col0) < chunk ? (N - col0) : chunk;
        const T* xs = x + r * ld + col0;
        const RowGeom geo = scalar ? RowGeom{0, 0, 0} : row_geometry<T>(xs, n);
        const T* xv = xs + geo.head;

        MD s{-INFINITY, 0.f};
        if (scalar)
            for (int64_t cc = t; cc < n; cc += BLOCK) s = md_push(s, E::load(xs + cc));
        if (t < geo.extras()) s = md_push(s, E::load(xs + extra_col(geo, t, V)));
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
                    if (vm == -INFINITY) continue;
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
        if (t == 0) partials[item] = make_float2(s.m, s.d);
    }
}

// Merge the nchunks partials of row r. Thread q takes partials q, q + BLOCK, ...
// in order, then the CTA combines them in a fixed tree, so every CTA of a row
// computes bit-identical (m, d).
template <int BLOCK>
__device__ __forceinline__ MD merge_row_partials(const float2* p, int64_t nchunks, float* red_m,
                                                 float* red_d) {
    MD s{-INFINITY, 0.f};
    for (int64_t q = threadIdx.x; q < nchunks; q += BLOCK) {
        const float2 v = p[q];
        s = md_merge(s, MD{v.x, v.y});
    }
    return group_merge<BLOCK>(s, red_m, red_d);
}

template <typename T, int BLOCK, int UNROLL>
__global__ void __launch_bounds__(BLOCK)
    split_normalise_kernel(const T* x, T* y, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                           int64_t nchunks, bool scalar, const float2* partials) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    __shared__ float red_m[2][BLOCK / 32];
    __shared__ float red_d[2][BLOCK / 32];
    const int t = threadIdx.x;
    int parity = 0;
    const int64_t items = M * nchunks;

    for (int64_t k = blockIdx.x; k < items; k += gridDim.x, parity ^= 1) {
        // last chunks first: the partial pass read them last, so they are the
        // ones still in L2 when this pass starts
        const int64_t item = items - 1 - k;
        const int64_t r = item / nchunks, c = item - r * nchunks;
        const int64_t col0 = c * chunk;
        const int64_t n = (N - col0) < chunk ? (N - col0) : chunk;
        const T* xs = x + r * ld + col0;
        T* ys = y + r * ld + col0;
        const RowGeom geo = scalar ? RowGeom{0, 0, 0} : row_geometry<T>(xs, n);
        const T* xv = xs + geo.head;
        T* yv = ys + geo.head;

        // issue this chunk's loads before the merge so they overlap it
        uint4 raw[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t k = t + int64_t(u) * BLOCK;
            if (k < geo.nvec) raw[u] = ld_stream16(xv + k * V);
        }

        const MD s = merge_row_partials<BLOCK>(partials + r * nchunks, nchunks, red_m[parity],
                                               red_d[parity]);
        const float m = s.d > 0.f ? s.m : 0.f;
        const float inv = safe_inverse(s.d);

        if (scalar)
            for (int64_t cc = t; cc < n; cc += BLOCK) E::store(ys + cc, exp_shifted(E::load(xs + cc), m) * inv);
        if (t < geo.extras()) {
            const int64_t cc = extra_col(geo, t, V);
            E::store(ys + cc, exp_shifted(E::load(xs + cc), m) * inv);
        }
        for (int64_t k0 = t;; k0 += int64_t(BLOCK) * UNROLL) {
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
            const int64_t next = k0 + int64_t(BLOCK) * UNROLL;
            if (next >= geo.nvec) break;
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int64_t k = next + int64_t(u) * BLOCK;
                if (k < geo.nvec) raw[u] = ld_stream16(xv + k * V);
            }
        }
    }
}

}  // namespace rowops
