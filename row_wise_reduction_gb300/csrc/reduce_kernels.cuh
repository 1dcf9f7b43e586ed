// Row-wise sum and row-wise max ["Triton Kernel 实现练习" §2.2 Row-wise Sum,
// §2.3 Row-wise Max; "CS336 Kernels, Triton" notes, "Triton Row Sum" (the
// looped "baby tiling" form for rows longer than one block)]:
//   out[i] = sum_j x[i, j]     (padding contributes 0)
//   out[i] = max_j x[i, j]     (padding is -inf; a NaN makes the result NaN)
// fp32 accumulation, fp32 results. Three forms, as for softmax: the TMA-fed
// row pipeline (rows of 64..4096 16-byte vectors), register row groups for
// shorter rows, and a looped CTA-per-row kernel for everything else.
#pragma once

#include "tma_row_kernels.cuh"

namespace rowops {

// max that propagates NaN (fmaxf drops it)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

struct RowSum {
    static constexpr float kIdentity = 0.f;
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};
struct RowMax {
    static constexpr float kIdentity = -INFINITY;
    __device__ __forceinline__ float operator()(float a, float b) const { return fmax_nan(a, b); }
};

template <class Op, int V>
__device__ __forceinline__ float fold_vec(float acc, const float* v, Op op) {
#pragma unroll
    for (int e = 0; e < V; ++e) acc = op(acc, v[e]);
    return acc;
}

// Row pipeline: one row group of TPR threads per CTA, one group reduction per
// row (two alternating buffers); the group's first thread writes the result.
template <typename T, int TPR, int VPT, bool FULL, class Op>
__global__ void __launch_bounds__(TPR)
    reduce_tma_kernel(const T* x, float* out, int64_t M, int N, int64_t ld, int nbuf, unsigned* err,
                      unsigned long long wait_ns, int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red[2][TPR / 32];
    const Op op;
    const GroupPipe p = make_group<TPR, 1>(smem, N, E::kBytes, nbuf);
    const int t = threadIdx.x;
    start_pipes<T, FULL, 1>(smem, p, x, M, N, ld, stall_row);

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = rc.slot;
        const T* xr = x + row * ld;
        const RowSpan sp = row_span<T, FULL>(xr, N);
        const bool has_ex = !FULL && t < sp.head + sp.tail;
        float acc = has_ex ? E::load(xr + span_extra_col(sp, t, V)) : Op::kIdentity;
        int fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
        const char* sb = p.ring.slot(s);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
                float v[V];
                E::unpack(lds16(sb + size_t(k) * 16), v);
                acc = fold_vec<Op, V>(acc, v, op);
            }
        }
        acc = row_reduce<TPR>(acc, red[i & 1], p.bar_id, op, fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            return;
        }
        refill<T, FULL>(p, s, row, x, M, N, ld, stall_row);
        if (t == 0) out[row] = acc;
    }
}

// Register row groups (TPR threads per row, BLOCK / TPR rows per CTA, VPT
// 16-byte vectors per thread): every load of the row is issued before the
// first fold.
template <typename T, int TPR, int VPT, int BLOCK, class Op>
__global__ void __launch_bounds__(BLOCK)
    reduce_reg_kernel(const T* x, float* out, int64_t M, int N, int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int ROWS = BLOCK / TPR;
    static_assert(BLOCK % TPR == 0 && TPR >= 16, "row group must be at least a half warp");
    __shared__ float red[2][BLOCK / 32 > 0 ? BLOCK / 32 : 1];
    const Op op;
    const int t = threadIdx.x % TPR;
    const int slot = threadIdx.x / TPR;
    const int64_t ngroups = (M + ROWS - 1) / ROWS;
    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const int64_t row = g * ROWS + slot;
        const bool live = row < M;
        const T* xr = x + (live ? row : 0) * ld;
        RowGeom geo = row_geometry<T>(xr, N);
        if (!live) geo = RowGeom{0, 0, 0};
        uint4 raw[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t k = t + int64_t(j) * TPR;
            if (k < geo.nvec) raw[j] = ld_stream16(xr + geo.head + k * V);
        }
        float acc = t < geo.extras() ? E::load(xr + extra_col(geo, t, V)) : Op::kIdentity;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t k = t + int64_t(j) * TPR;
            if (k < geo.nvec) {
                float v[V];
                E::unpack(raw[j], v);
                acc = fold_vec<Op, V>(acc, v, op);
            }
        }
        acc = group_reduce<TPR>(acc, red[(g / gridDim.x) & 1], op);
        if (live && t == 0) out[row] = acc;
    }
}

// One CTA per row, any N and layout: the "baby tiling" loop, UNROLL 16-byte
// vectors in flight per thread per step, then one CTA reduction.
template <typename T, int BLOCK, int UNROLL, class Op>
__global__ void __launch_bounds__(BLOCK)
    reduce_looped_kernel(const T* x, float* out, int64_t M, int64_t N, int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    __shared__ float red[2][BLOCK / 32];
    const Op op;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const T* xr = x + row * ld;
        const RowGeom geo = row_geometry<T>(xr, N);
        const T* xv = xr + geo.head;
        float acc = threadIdx.x < geo.extras() ? E::load(xr + extra_col(geo, threadIdx.x, V)) : Op::kIdentity;
        for (int64_t k0 = threadIdx.x; k0 < geo.nvec; k0 += int64_t(BLOCK) * UNROLL) {
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
                    float v[V];
                    E::unpack(raw[u], v);
                    acc = fold_vec<Op, V>(acc, v, op);
                }
            }
        }
        acc = group_reduce<BLOCK>(acc, red[(row / gridDim.x) & 1], op);
        if (threadIdx.x == 0) out[row] = acc;
    }
}

}  // namespace rowops
