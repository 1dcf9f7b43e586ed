// Softmax and LayerNorm+GELU on the TMA-fed row pipeline (row_pipeline.cuh):
// one row per CTA iteration, BLOCK threads per row, VPT 16-byte vectors per
// thread. Thread t owns vectors k = t + i * BLOCK (i < VPT), so a warp's reads
// of a row buffer are contiguous and free of bank conflicts. FULL: the row is
// exactly BLOCK * VPT vectors (no per-element predicates).
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

template <typename T, int BLOCK, int VPT, bool FULL>
__global__ void __launch_bounds__(BLOCK)
    softmax_tma_kernel(const T* x, T* y, int64_t M, int N, int64_t ld, int nbuf, unsigned* err) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    static_assert(BLOCK % 64 == 0, "one row per CTA of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_max[BLOCK / 32];
    __shared__ float red_sum[BLOCK / 32];
    const RowRing ring{reinterpret_cast<uint64_t*>(smem), smem + kRingHeader,
                       ring_row_bytes(N, E::kBytes), nbuf};
    const int t = threadIdx.x;
    const int64_t G = gridDim.x, r0 = blockIdx.x;
    const uint32_t bytes = uint32_t(N) * E::kBytes;
    const int nvec = N / V;

    if (t == 0) {
        for (int s = 0; s < nbuf; ++s) mbar_init(ring.bar + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (t == 0)
        for (int s = 0; s < nbuf; ++s) {
            const int64_t row = r0 + s * G;
            if (row < M) tma_load_row(ring.slot(s), x + row * ld, bytes, ring.bar + s);
        }

    for (int64_t i = 0;; ++i) {
        const int64_t row = r0 + i * G;
        if (row >= M) break;
        const int s = int(i % nbuf);
        int fail = !mbar_wait(ring.bar + s, uint32_t((i / nbuf) & 1));
        const char* sb = ring.slot(s);

        float v[VPT][V];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * BLOCK;
            if (FULL || k < nvec) {
                E::unpack(lds16(sb + size_t(k) * 16), v[j]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[j][e] = -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) mx = fmaxf(mx, v[j][e]);
        }
        mx = cta_reduce<BLOCK>(mx, red_max, OpMax(), fail);
        if (fail) {
            if (t == 0) {
                drain_ring(ring, i, r0, G, M);
                atomicExch(err, kDeviceErrTimeout);
            }
            return;
        }
        // every thread now holds its part of the row: refill this buffer
        if (t == 0) {
            const int64_t nxt = row + int64_t(nbuf) * G;
            if (nxt < M) {
                fence_proxy_async_smem();
                tma_load_row(ring.slot(s), x + nxt * ld, bytes, ring.bar + s);
            }
        }
        if (mx == -INFINITY) mx = 0.f;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = exp_shifted(v[j][e], mx);
                sum += v[j][e];
            }
        sum = cta_reduce<BLOCK>(sum, red_sum, OpSum(), fail);
        const float inv = safe_inverse(sum);
        T* yr = y + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * BLOCK;
            if (FULL || k < nvec) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[j][e] * inv;
                st_stream16(yr + size_t(k) * V, E::pack(o));
            }
        }
    }
}

// w, b staged as fp32 in a thread-major order: float4 slot (j * (V/4) + h) * BLOCK + t
// holds columns 4h .. 4h+3 of vector k = t + j * BLOCK, so each LDS.128 of a warp
// reads 512 contiguous bytes.
template <typename T, int BLOCK, int VPT>
__device__ __forceinline__ void stage_affine_thread_major(const T* w, const T* b, int nvec, float4* sw4,
                                                          float4* sb4) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    for (int q = threadIdx.x; q < VPT * H * BLOCK; q += BLOCK) {
        const int tt = q % BLOCK, rest = q / BLOCK, h = rest % H, j = rest / H;
        const int k = tt + j * BLOCK;
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

template <typename T, int BLOCK, int VPT>
__host__ __device__ constexpr uint32_t tma_affine_bytes() {
    return uint32_t(2) * VPT * BLOCK * Elem<T>::kVec * 4;
}

template <typename T, int BLOCK, int VPT, bool FULL>
__global__ void __launch_bounds__(BLOCK)
    ln_gelu_tma_kernel(const T* x, T* y, const T* w, const T* b, float eps, int64_t M, int N, int64_t ld,
                       int nbuf, unsigned* err) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    static_assert(BLOCK % 64 == 0, "one row per CTA of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_a[BLOCK / 32];
    __shared__ float red_b[2 * BLOCK / 32];
    const uint32_t row_bytes = ring_row_bytes(N, E::kBytes);
    const RowRing ring{reinterpret_cast<uint64_t*>(smem), smem + kRingHeader, row_bytes, nbuf};
    float4* sw4 = reinterpret_cast<float4*>(smem + kRingHeader + size_t(nbuf) * row_bytes);
    float4* sb4 = sw4 + VPT * H * BLOCK;
    const int t = threadIdx.x;
    const int64_t G = gridDim.x, r0 = blockIdx.x;
    const uint32_t bytes = uint32_t(N) * E::kBytes;
    const int nvec = N / V;
    const float fN = float(N);

    if (t == 0) {
        for (int s = 0; s < nbuf; ++s) mbar_init(ring.bar + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (t == 0)
        for (int s = 0; s < nbuf; ++s) {
            const int64_t row = r0 + s * G;
            if (row < M) tma_load_row(ring.slot(s), x + row * ld, bytes, ring.bar + s);
        }
    stage_affine_thread_major<T, BLOCK, VPT>(w, b, nvec, sw4, sb4);
    __syncthreads();

    for (int64_t i = 0;; ++i) {
        const int64_t row = r0 + i * G;
        if (row >= M) break;
        const int s = int(i % nbuf);
        int fail = !mbar_wait(ring.bar + s, uint32_t((i / nbuf) & 1));
        const char* sb = ring.slot(s);

        float v[VPT][V];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * BLOCK;
            if (FULL || k < nvec) {
                E::unpack(lds16(sb + size_t(k) * 16), v[j]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[j][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) sum += v[j][e];
        }
        sum = cta_reduce<BLOCK>(sum, red_a, OpSum(), fail);
        if (fail) {
            if (t == 0) {
                drain_ring(ring, i, r0, G, M);
                atomicExch(err, kDeviceErrTimeout);
            }
            return;
        }
        if (t == 0) {
            const int64_t nxt = row + int64_t(nbuf) * G;
            if (nxt < M) {
                fence_proxy_async_smem();
                tma_load_row(ring.slot(s), x + nxt * ld, bytes, ring.bar + s);
            }
        }
        const float mean = sum / fN;
        // centred values, their squares and the residual of the fp32 mean
        float q = 0.f, r = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const bool ok = FULL || (t + j * BLOCK) < nvec;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = ok ? v[j][e] - mean : 0.f;
                q = fmaf(v[j][e], v[j][e], q);
                r += v[j][e];
            }
        }
        cta_reduce_sum2<BLOCK>(q, r, red_b, fail);
        const float delta = r / fN;
        const float rstd = rsqrtf(fmaxf(q / fN - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;
        T* yr = y + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * BLOCK;
            if (FULL || k < nvec) {
                float o[V];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float4 ww = sw4[(j * H + h) * BLOCK + t];
                    const float4 bb = sb4[(j * H + h) * BLOCK + t];
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
