// Softmax and LayerNorm+GELU on the TMA-fed row pipeline (row_pipeline.cuh).
//
// A CTA holds ROWS independent row groups of TPR threads. Group g works on
// rows gg, gg + GG, gg + 2 GG, ... (gg = blockIdx.x * ROWS + g, GG = gridDim.x *
// ROWS; with phase classes, below, the same within the CTA's class of rows)
// with its own ring of nbuf row buffers, its own producer thread (the
// group's first thread) and its own named barrier, so groups never wait for
// each other; they share only the staged w, b of LayerNorm+GELU, which is what
// lets one CTA keep many rows in flight without a copy of w, b per row. Each
// thread owns vectors k = t + j * TPR (j < VPT) of its row, so a warp's reads
// of a row buffer are contiguous and free of bank conflicts. FULL: rows start
// on 16-byte boundaries and are exactly TPR * VPT vectors (no per-element
// predicates). Otherwise rows may start anywhere (x and y at the same offset
// modulo 16 bytes): each row's 16-byte-aligned body comes by bulk copy and its
// unaligned head and tail (< 16 bytes each) by plain loads, issued before the
// wait so their latency overlaps it.
//
// Phase classes (LayerNorm+GELU on general rows): with row stride ld, row r
// starts at offset r * ld * sizeof(T) modulo 16 bytes, which repeats with period
// P = 16 / gcd(16, ld * sizeof(T)). The grid is a multiple of P and its P
// equal blocks of CTAs take one class r mod P each, so all rows of a CTA have
// the same head, body and tail, and w,
// b are staged once in the thread-major order of that split: the loop body is
// then that of full rows plus predicates and the head/tail elements.
//
// The arithmetic is that of the register-resident kernels (softmax_kernels.cuh,
// ln_gelu_kernels.cuh): stable softmax [Triton Kernel 实现练习 §2.4]; LayerNorm
// with the variance of the centred row and the residual correction of the fp32
// mean, then z / (1 + exp(-2u)) GELU [PyTorch 自定义 CUDA 算子与 Triton 编程 §三].
#pragma once

#include "ln_gelu_kernels.cuh"
#include "row_pipeline.cuh"
#include "rowops_launch.h"
#include "softmax_kernels.cuh"

namespace rowops {

// Per-group view of the pipeline state.
struct GroupPipe {
    RowRing ring;
    int64_t first, stride;  // rows first + i * stride, i = 0, 1, ...
    int cls;                // phase class of the CTA's rows
    int bar_id;             // named barrier of the group
    bool producer;          // the group's first thread issues its copies
};

// `period`: number of phase classes (1: every CTA takes every kind of row);
// `streams`: rows of that many inputs share each ring slot.
template <int TPR, int ROWS>
__device__ __forceinline__ GroupPipe make_group(char* smem, int64_t N, int es, int nbuf, int period = 1,
                                                int streams = 1) {
    const int g = threadIdx.x / TPR;
    const uint32_t rb = uint32_t(streams) * ring_row_bytes(N, es);
    GroupPipe p;
    p.ring = RowRing{reinterpret_cast<uint64_t*>(smem) + g * nbuf, smem + kRingHeader + size_t(g) * nbuf * rb, rb,
                     nbuf};
    // CTAs [cls * ctas, (cls + 1) * ctas) take class cls (the grid is a multiple of period)
    const int ctas = period == 1 ? int(gridDim.x) : int(gridDim.x) / period;
    const int cls = period == 1 ? 0 : int(blockIdx.x) / ctas;
    const int local = period == 1 ? int(blockIdx.x) : int(blockIdx.x) % ctas;
    p.cls = cls;
    p.first = cls + int64_t(period) * (int64_t(local) * ROWS + g);
    p.stride = int64_t(period) * ctas * ROWS;
    p.bar_id = 1 + g;
    p.producer = (threadIdx.x % TPR) == 0;
    return p;
}

// The part of a row the bulk copy brings: `body` 16-byte vectors starting
// `head` elements in; `tail` elements follow them.
struct RowSpan {
    int head, body, tail;
};

template <typename T, bool FULL>
__device__ __forceinline__ RowSpan row_span(const T* row, int N) {
    if constexpr (FULL) {
        return RowSpan{0, N / Elem<T>::kVec, 0};
    } else {
        const RowGeom g = row_geometry<T>(row, N);
        return RowSpan{g.head, int(g.nvec), g.tail};
    }
}

// Test hook: the copy of row `stall_row` is expected to bring 16 bytes more than
// it does, so the wait on it runs out (-1: no such row).
__device__ __forceinline__ uint32_t stall_extra(int64_t row, int64_t stall_row) { return row == stall_row ? 16u : 0u; }

// Producer: copy the body of `row` into buffer s.
template <typename T, bool FULL>
__device__ __forceinline__ void issue_row(const GroupPipe& p, int s, int64_t row, const T* x, int N, int64_t ld,
                                          int64_t stall_row) {
    const T* xr = x + row * ld;
    const RowSpan sp = row_span<T, FULL>(xr, N);
    tma_load_row(p.ring.slot(s), xr + sp.head, uint32_t(sp.body) * 16u, p.ring.bar + s, stall_extra(row, stall_row));
}

// CTA start: thread 0 initialises every group's barriers; then each group's
// producer issues the copies of its first nbuf rows.
template <typename T, bool FULL, int ROWS>
__device__ __forceinline__ void start_pipes(char* smem, const GroupPipe& p, const T* x, int64_t M, int N, int64_t ld,
                                            int64_t stall_row) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROWS * p.ring.nbuf; ++s) mbar_init(reinterpret_cast<uint64_t*>(smem) + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (p.producer)
        for (int s = 0; s < p.ring.nbuf; ++s) {
            const int64_t row = p.first + s * p.stride;
            if (row < M) issue_row<T, FULL>(p, s, row, x, N, ld, stall_row);
        }
}

// After the group's first reduction: refill buffer s with the row nbuf
// iterations ahead (every thread of the group has its data in registers).
template <typename T, bool FULL>
__device__ __forceinline__ void refill(const GroupPipe& p, int s, int64_t row, const T* x, int64_t M, int N,
                                       int64_t ld, int64_t stall_row) {
    if (!p.producer) return;
    const int64_t nxt = row + int64_t(p.ring.nbuf) * p.stride;
    if (nxt < M) {
        fence_proxy_async_smem();
        issue_row<T, FULL>(p, s, nxt, x, N, ld, stall_row);
    }
}

// Column of unaligned element e (head first, then tail) of a row.
__device__ __forceinline__ int span_extra_col(const RowSpan& sp, int e, int V) {
    return e < sp.head ? e : sp.head + sp.body * V + (e - sp.head);
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
    start_pipes<T, FULL, ROWS>(smem, p, x, M, N, ld, stall_row);

    for (int64_t i = 0;; ++i) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = int(i % nbuf);
        const T* xr = x + row * ld;
        const RowSpan sp = row_span<T, FULL>(xr, N);
        // unaligned head / tail elements: plain loads, in flight during the wait
        const bool has_ex = !FULL && t < sp.head + sp.tail;
        const int ecol = has_ex ? span_extra_col(sp, t, V) : 0;
        float ex = has_ex ? E::load(xr + ecol) : -INFINITY;
        int fail = !mbar_wait(p.ring.bar + s, uint32_t((i / nbuf) & 1), wait_ns);
        const char* sb = p.ring.slot(s);

        float v[VPT][V];
        float mx = ex;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
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
        refill<T, FULL>(p, s, row, x, M, N, ld, stall_row);
        if (mx == -INFINITY) mx = 0.f;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = exp_shifted(v[j][e], mx);
                sum += v[j][e];
            }
        ex = exp_shifted(ex, mx);
        sum += ex;
        sum = row_reduce<TPR>(sum, red_sum[g], p.bar_id, OpSum(), fail);
        const float inv = safe_inverse(sum);
        T* yr = y + row * ld;
        T* yb = yr + sp.head;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[j][e] * inv;
                st_stream16(yb + size_t(k) * V, E::pack(o));
            }
        }
        if (has_ex) E::store(yr + ecol, ex * inv);
    }
}

// w, b staged as fp32 in a thread-major order: float4 slot (j * (V/4) + h) * TPR + t
// holds columns c0 + 4h .. c0 + 4h + 3 of vector k = t + j * TPR (column c0 =
// head + k * V), so each LDS.128 of a warp reads 512 contiguous bytes. Vectors
// k >= nvec get w = 1, b = 0. Shared by all row groups of the CTA.
template <typename T, int TPR, int VPT>
__device__ __forceinline__ void stage_affine_thread_major(const T* w, const T* b, int head, int nvec, float4* sw4,
                                                          float4* sb4) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    for (int q = threadIdx.x; q < VPT * H * TPR; q += blockDim.x) {
        const int tt = q % TPR, rest = q / TPR, h = rest % H, j = rest / H;
        const int k = tt + j * TPR;
        float4 ww = make_float4(1.f, 1.f, 1.f, 1.f), bb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nvec) {
            const int c = head + k * V + 4 * h;
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

// General rows add the (w, b) pairs of the class's head and tail columns
// (fewer than 2V of them), in the order span_extra_col numbers them.
constexpr uint32_t kAffineExtraBytes = 256;

template <typename T, int TPR, int VPT, bool FULL>
__host__ __device__ constexpr uint32_t affine_stage_bytes() {
    return tma_affine_bytes<T, TPR, VPT>() + (FULL ? 0u : kAffineExtraBytes);
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
    const int period = FULL ? 1 : row_phase_period(ld * E::kBytes);
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf, period);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    char* affine = smem + kRingHeader + size_t(ROWS) * nbuf * p.ring.row_bytes;
    float4* sw4 = reinterpret_cast<float4*>(affine);
    float4* sb4 = sw4 + VPT * H * TPR;
    float2* sxb = reinterpret_cast<float2*>(affine + tma_affine_bytes<T, TPR, VPT>());
    const float fN = float(N);
    // the split shared by every row of this CTA's phase class
    const RowSpan sp = row_span<T, FULL>(x + int64_t(p.cls) * ld, N);
    start_pipes<T, FULL, ROWS>(smem, p, x, M, N, ld, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, sp.head, sp.body, sw4, sb4);
    if constexpr (!FULL) {
        for (int e = threadIdx.x; e < sp.head + sp.tail; e += blockDim.x) {
            const int c = span_extra_col(sp, e, V);
            sxb[e] = make_float2(w ? E::load(w + c) : 1.f, b ? E::load(b + c) : 0.f);
        }
    }
    __syncthreads();
    const bool has_ex = !FULL && t < sp.head + sp.tail;
    const int ecol = has_ex ? span_extra_col(sp, t, V) : 0;

    for (int64_t i = 0;; ++i) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = int(i % nbuf);
        const T* xr = x + row * ld;
        float ex = has_ex ? E::load(xr + ecol) : 0.f;
        int fail = !mbar_wait(p.ring.bar + s, uint32_t((i / nbuf) & 1), wait_ns);
        const char* sbuf = p.ring.slot(s);

        float v[VPT][V];
        float sum = ex;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
                E::unpack(lds16(sbuf + size_t(k) * 16), v[j]);
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
        refill<T, FULL>(p, s, row, x, M, N, ld, stall_row);
        const float mean = sum / fN;
        // centred values, their squares and the residual of the fp32 mean
        float q = 0.f, r = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const bool ok = FULL || (t + j * TPR) < sp.body;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = ok ? v[j][e] - mean : 0.f;
                q = fmaf(v[j][e], v[j][e], q);
                r += v[j][e];
            }
        }
        if constexpr (!FULL) {
            ex = has_ex ? ex - mean : 0.f;
            q = fmaf(ex, ex, q);
            r += ex;
        }
        row_reduce_sum2<TPR>(q, r, red_b[g], p.bar_id, fail);
        const float delta = r / fN;
        const float rstd = rsqrtf(fmaxf(q / fN - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;
        T* yr = y + row * ld;
        T* yb = yr + sp.head;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
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
                st_stream16(yb + size_t(k) * V, E::pack(o));
            }
        }
        if (has_ex) {
            const float2 wb = sxb[t];
            E::store(yr + ecol, gelu_tanh_approx(fmaf(fmaf(ex, rstd, shift), wb.x, wb.y)));
        }
    }
}

}  // namespace rowops
