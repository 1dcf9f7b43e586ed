// Softmax and LayerNorm+GELU on the TMA-fed row pipeline (row_pipeline.cuh).
//
// A CTA holds ROWS independent row groups of TPR threads. Group g works on
// rows gg, gg + GG, gg + 2 GG, ... (gg = blockIdx.x * ROWS + g, GG = gridDim.x *
// ROWS) with its own ring of nbuf row buffers, its own producer thread (the
// group's first thread) and its own named barrier, so groups never wait for
// each other; they share only the staged w, b of LayerNorm+GELU, which is what
// lets one CTA keep many rows in flight without a copy of w, b per row. Each
// thread owns vectors k = t + j * TPR (j < VPT) of its row, so a warp's reads
// of a row buffer are contiguous and free of bank conflicts. FULL: the row is
// exactly TPR * VPT vectors (no per-element predicates).
//
// The arithmetic is that of the register-resident kernels (softmax_kernels.cuh,
// ln_gelu_kernels.cuh): stable softmax [Triton Kernel 实现练习 §2.4]; LayerNorm
// with the variance of the centred row and the residual correction of the fp32
// mean, then z / (1 + exp(-2u)) GELU [PyTorch 自定义 CUDA 算子与 Triton 编程 §三].
#pragma once

#include "ln_gelu_kernels.cuh"
#include "row_pipeline.cuh"
#include "softmax_kernels.cuh"

namespace rowops {

// Per-group view of the pipeline state.
struct GroupPipe {
    RowRing ring;
    int64_t first, stride;  // rows first + i * stride, i = 0, 1, ...
    int bar_id;             // named barrier of the group
    bool producer;          // the group's first thread issues its copies
};

template <int TPR, int ROWS>
__device__ __forceinline__ GroupPipe make_group(char* smem, int64_t N, int es, int nbuf) {
    const int g = threadIdx.x / TPR;
    const uint32_t rb = ring_row_bytes(N, es);
    GroupPipe p;
    p.ring = RowRing{reinterpret_cast<uint64_t*>(smem) + g * nbuf, smem + kRingHeader + size_t(g) * nbuf * rb, rb,
                     nbuf};
    p.first = int64_t(blockIdx.x) * ROWS + g;
    p.stride = int64_t(gridDim.x) * ROWS;
    p.bar_id = 1 + g;
    p.producer = (threadIdx.x % TPR) == 0;
    return p;
}

// CTA start: thread 0 initialises every group's barriers; then each group's
// producer issues the copies of its first nbuf rows.
// Test hook: the copy of row `stall_row` is expected to bring 16 bytes more than
// it does, so the wait on it runs out (-1: no such row).
__device__ __forceinline__ uint32_t stall_extra(int64_t row, int64_t stall_row) { return row == stall_row ? 16u : 0u; }

template <int ROWS>
__device__ __forceinline__ void start_pipes(char* smem, const GroupPipe& p, const void* x, int64_t M, int64_t ld,
                                            int es, uint32_t bytes, int64_t stall_row) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROWS * p.ring.nbuf; ++s) mbar_init(reinterpret_cast<uint64_t*>(smem) + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (p.producer)
        for (int s = 0; s < p.ring.nbuf; ++s) {
            const int64_t row = p.first + s * p.stride;
            if (row < M)
                tma_load_row(p.ring.slot(s), static_cast<const char*>(x) + size_t(row * ld) * es, bytes, p.ring.bar + s,
                             stall_extra(row, stall_row));
        }
}

// After the group's first reduction: refill buffer s with the row nbuf
// iterations ahead (every thread of the group has its data in registers).
__device__ __forceinline__ void refill(const GroupPipe& p, int s, int64_t row, const void* x, int64_t M, int64_t ld,
                                       int es, uint32_t bytes, int64_t stall_row) {
    if (!p.producer) return;
    const int64_t nxt = row + int64_t(p.ring.nbuf) * p.stride;
    if (nxt < M) {
        fence_proxy_async_smem();
        tma_load_row(p.ring.slot(s), static_cast<const char*>(x) + size_t(nxt * ld) * es, bytes, p.ring.bar + s,
                     stall_extra(nxt, stall_row));
    }
}

// Error exit of a group whose wait gave up: its producer waits (bounded) for
// the copies still in flight and records the timeout.
__device__ __forceinline__ void abandon(const GroupPipe& p, int64_t i, int64_t M, unsigned* err,
                                        unsigned long long wait_ns) {
    if (!p.producer) return;
    drain_ring(p.ring, i, p.first, p.stride, M, wait_ns);
    atomicExch(err, kDeviceErrTimeout);
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL>
__global__ void __launch_bounds__(TPR * ROWS)
    softmax_tma_kernel(const T* x, T* y, int64_t M, int N, int64_t ld, int nbuf, unsigned* err,
                       unsigned long long wait_ns, int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_max[ROWS][TPR / 32];
    __shared__ float red_sum[ROWS][TPR / 32];
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    const uint32_t bytes = uint32_t(N) * E::kBytes;
    const int nvec = N / V;
    start_pipes<ROWS>(smem, p, x, M, ld, E::kBytes, bytes, stall_row);

    for (int64_t i = 0;; ++i) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = int(i % nbuf);
        int fail = !mbar_wait(p.ring.bar + s, uint32_t((i / nbuf) & 1), wait_ns);
        const char* sb = p.ring.slot(s);

        float v[VPT][V];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < nvec) {
                E::unpack(lds16(sb + size_t(k) * 16), v[j]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[j][e] = -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) mx = fmaxf(mx, v[j][e]);
        }
        mx = row_reduce<TPR>(mx, red_max[g], p.bar_id, OpMax(), fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            return;
        }
        refill(p, s, row, x, M, ld, E::kBytes, bytes, stall_row);
        if (mx == -INFINITY) mx = 0.f;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = exp_shifted(v[j][e], mx);
                sum += v[j][e];
            }
        sum = row_reduce<TPR>(sum, red_sum[g], p.bar_id, OpSum(), fail);
        const float inv = safe_inverse(sum);
        T* yr = y + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < nvec) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[j][e] * inv;
                st_stream16(yr + size_t(k) * V, E::pack(o));
            }
        }
    }
}

// w, b staged as fp32 in a thread-major order: float4 slot (j * (V/4) + h) * TPR + t
// holds columns 4h .. 4h+3 of vector k = t + j * TPR, so each LDS.128 of a warp
// reads 512 contiguous bytes. Shared by all row groups of the CTA.
template <typename T, int TPR, int VPT>
__device__ __forceinline__ void stage_affine_thread_major(const T* w, const T* b, int nvec, float4* sw4,
                                                          float4* sb4) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    for (int q = threadIdx.x; q < VPT * H * TPR; q += blockDim.x) {
        const int tt = q % TPR, rest = q / TPR, h = rest % H, j = rest / H;
        const int k = tt + j * TPR;
        float4 ww = make_float4(1.f, 1.f, 1.f, 1.f), bb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nvec) {
            const int c = k * V + 4 * h;
            if (w) ww = make_float4(E::load(w + c), E::load(w + c + 1), E::load(w + c + 2), E::load(w + c + 3));
            if (b) bb = make_float4(E::load(b + c), E::load(b + c + 1), E::load(b + c + 2), E::load(b + c + 3));
        }
        sw4[q] = ww;
        sb4[q] = bb;
    }
}

template <typename T, int TPR, int VPT>
__host__ __device__ constexpr uint32_t tma_affine_bytes() {
    return uint32_t(2) * VPT * TPR * Elem<T>::kVec * 4;
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL>
__global__ void __launch_bounds__(TPR * ROWS)
    ln_gelu_tma_kernel(const T* x, T* y, const T* w, const T* b, float eps, int64_t M, int N, int64_t ld,
                       int nbuf, unsigned* err, unsigned long long wait_ns, int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_a[ROWS][TPR / 32];
    __shared__ float red_b[ROWS][2 * TPR / 32];
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    float4* sw4 = reinterpret_cast<float4*>(smem + kRingHeader + size_t(ROWS) * nbuf * p.ring.row_bytes);
    float4* sb4 = sw4 + VPT * H * TPR;
    const uint32_t bytes = uint32_t(N) * E::kBytes;
    const int nvec = N / V;
    const float fN = float(N);
    start_pipes<ROWS>(smem, p, x, M, ld, E::kBytes, bytes, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, nvec, sw4, sb4);
    __syncthreads();

    for (int64_t i = 0;; ++i) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = int(i % nbuf);
        int fail = !mbar_wait(p.ring.bar + s, uint32_t((i / nbuf) & 1), wait_ns);
        const char* sb = p.ring.slot(s);

        float v[VPT][V];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < nvec) {
                E::unpack(lds16(sb + size_t(k) * 16), v[j]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[j][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) sum += v[j][e];
        }
        sum = row_reduce<TPR>(sum, red_a[g], p.bar_id, OpSum(), fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            return;
        }
        refill(p, s, row, x, M, ld, E::kBytes, bytes, stall_row);
        const float mean = sum / fN;
        // centred values, their squares and the residual of the fp32 mean
        float q = 0.f, r = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const bool ok = FULL || (t + j * TPR) < nvec;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = ok ? v[j][e] - mean : 0.f;
                q = fmaf(v[j][e], v[j][e], q);
                r += v[j][e];
            }
        }
        row_reduce_sum2<TPR>(q, r, red_b[g], p.bar_id, fail);
        const float delta = r / fN;
        const float rstd = rsqrtf(fmaxf(q / fN - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;
        T* yr = y + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < nvec) {
                float o[V];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float4 ww = sw4[(j * H + h) * TPR + t];
                    const float4 bb = sb4[(j * H + h) * TPR + t];
                    o[4 * h + 0] = gelu_tanh_approx(fmaf(fmaf(v[j][4 * h + 0], rstd, shift), ww.x, bb.x));
                    o[4 * h + 1] = gelu_tanh_approx(fmaf(fmaf(v[j][4 * h + 1], rstd, shift), ww.y, bb.y));
                    o[4 * h + 2] = gelu_tanh_approx(fmaf(fmaf(v[j][4 * h + 2], rstd, shift), ww.z, bb.z));
                    o[4 * h + 3] = gelu_tanh_approx(fmaf(fmaf(v[j][4 * h + 3], rstd, shift), ww.w, bb.w));
                }
                st_stream16(yr + size_t(k) * V, E::pack(o));
            }
        }
    }
}

}  // namespace rowops
