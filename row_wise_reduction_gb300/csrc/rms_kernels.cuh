// RMSNorm and fused residual + RMSNorm kernels (register-resident row groups
// and a looped any-layout form; the row-pipeline form is in
// tma_rms_kernels.cuh).
//
// Definition ["Triton Kernel 实现练习" §4.2 RMSNorm, §4.3 Fused Residual
// RMSNorm]: inv_rms = rsqrt(mean(s^2) + eps), y = s * inv_rms * w, with s = x
// (RMSNorm) or s = x + residual (fused form, which also writes s out as
// residual_out). Accumulation is fp32 and results are cast back to the I/O
// type. The fused form normalises s as it is stored (rounded to the I/O type),
// so its y equals RMSNorm applied to its own residual_out.
#pragma once

#include "rowops_device.cuh"

namespace rowops {

// w staged as fp32 with one unused slot after every V columns: column c at
// c + c / V. Thread v of a warp reads column c0 + V*v + j of its own vector,
// slot (V + 1) v + const, and V + 1 (5 or 9) is odd, so the 32 threads hit 32
// different banks whatever c0 (the row's head) is.
__host__ __device__ constexpr int weight_slot(int c, int V) { return c + c / V; }

__host__ __device__ constexpr size_t rms_weight_smem_bytes(int64_t N, int V) {
    return size_t(4) * size_t((N + N / V + 4) & ~int64_t(3));
}

template <typename T>
__device__ __forceinline__ void stage_weight_padded(const T* w, int N, float* sw) {
    using E = Elem<T>;
    for (int c = threadIdx.x; c < N; c += blockDim.x) sw[weight_slot(c, E::kVec)] = w ? E::load(w + c) : 1.f;
}

// s of one 16-byte vector: x, or x + residual as the I/O type stores it (the
// packed words are also the residual_out vector).
template <typename T, bool RES>
__device__ __forceinline__ uint4 residual_sum(const uint4& xa, const uint4& ra, float* s) {
    using E = Elem<T>;
    if constexpr (RES) {
        float a[E::kVec], b[E::kVec];
        E::unpack(xa, a);
        E::unpack(ra, b);
#pragma unroll
        for (int e = 0; e < E::kVec; ++e) a[e] += b[e];
        const uint4 packed = E::pack(a);
        E::unpack(packed, s);
        return packed;
    } else {
        E::unpack(xa, s);
        return xa;
    }
}

// TPR threads per row, VPT 16-byte vectors per thread held in registers; all
// of x, residual, y, residual_out share their offset modulo 16 bytes.
template <typename T, int TPR, int VPT, int BLOCK, bool RES>
__global__ void __launch_bounds__(BLOCK)
    rms_reg_kernel(const T* x, const T* res, T* y, T* res_out, const T* w, float eps, int64_t M, int N,
                   int64_t ld) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int ROWS = BLOCK / TPR;
    static_assert(BLOCK % TPR == 0 && TPR >= 16, "row group must be at least a half warp");
    extern __shared__ float4 smem_weight[];
    float* sw = reinterpret_cast<float*>(smem_weight);
    // one reduction per row: two buffers used alternately, so that a buffer is
    // rewritten only after the other one's barrier
    __shared__ float red[2][BLOCK / 32 > 0 ? BLOCK / 32 : 1];

    stage_weight_padded(w, N, sw);
    __syncthreads();

    const int t = threadIdx.x % TPR;
    const int slot = threadIdx.x / TPR;
    const int64_t ngroups = (M + ROWS - 1) / ROWS;
    // 1/N once; arithmetic on packed fp32 pairs
    const float inv_n = 1.f / float(N);

    for (int64_t g = blockIdx.x; g < ngroups; g += gridDim.x) {
        const int64_t row = g * ROWS + slot;
        const bool live = row < M;
        const int64_t off = (live ? row : 0) * ld;
        RowGeom geo = row_geometry<T>(x + off, N);
        if (!live) geo = RowGeom{0, 0, 0};

        uint4 xa[VPT], ra[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                xa[i] = ld_stream16(x + off + geo.head + k * V);
                if constexpr (RES) ra[i] = ld_stream16(res + off + geo.head + k * V);
            }
        }
        const bool has_ex = t < geo.extras();
        const int ecol = has_ex ? int(extra_col(geo, t, V)) : 0;
        float ex = 0.f;
        if (has_ex) {
            ex = E::load(x + off + ecol);
            if constexpr (RES) ex = E::round(ex + E::load(res + off + ecol));
        }

        float v[VPT][V];
        float2 q2 = make_float2(ex * ex, 0.f);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                const uint4 packed = residual_sum<T, RES>(xa[i], ra[i], v[i]);
                if constexpr (RES) st_stream16(res_out + off + geo.head + k * V, packed);
            } else {
#pragma unroll
                for (int j = 0; j < V; ++j) v[i][j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < V; j += 2) {
                const float2 p2 = make_float2(v[i][j], v[i][j + 1]);
                q2 = f2_fma(p2, p2, q2);
            }
        }
        const float q = group_reduce<TPR>(q2.x + q2.y, red[(g / gridDim.x) & 1], OpSum());
        const float inv = rsqrtf(q * inv_n + eps);

#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t k = t + int64_t(i) * TPR;
            if (k < geo.nvec) {
                const int c0 = geo.head + int(k) * V;
                float o[V];
#pragma unroll
                for (int j = 0; j < V; j += 2) {
                    const float2 p2 = f2_mul(f2_mul(make_float2(v[i][j], v[i][j + 1]), f2(inv)),
                                             make_float2(sw[weight_slot(c0 + j, V)], sw[weight_slot(c0 + j + 1, V)]));
                    o[j] = p2.x;
                    o[j + 1] = p2.y;
                }
                st_stream16(y + off + c0, E::pack(o));
            }
        }
        if (has_ex) {
            E::store(y + off + ecol, ex * inv * sw[weight_slot(ecol, V)]);
            if constexpr (RES) E::store(res_out + off + ecol, ex);
        }
    }
}

// One CTA per row, any layout (the four row pointers may sit at different
// offsets modulo 16 bytes): element-wise coalesced loops. Pass 1 forms s
// (writing residual_out in the fused form) and the sum of squares; pass 2
// reads s back (from residual_out, or x) and writes y. Each thread reads back
// only what it wrote itself.
template <typename T, int BLOCK, bool RES>
__global__ void __launch_bounds__(BLOCK)
    rms_looped_kernel(const T* x, const T* res, T* y, T* res_out, const T* w, float eps, int64_t M, int64_t N,
                      int64_t ld) {
    using E = Elem<T>;
    __shared__ float red[2][BLOCK / 32];  // alternate per row, as in rms_reg_kernel
    const float fN = float(N);
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const int64_t off = row * ld;
        float q = 0.f;
        for (int64_t c = threadIdx.x; c < N; c += BLOCK) {
            float s = E::load(x + off + c);
            if constexpr (RES) {
                s = E::round(s + E::load(res + off + c));
                E::store(res_out + off + c, s);
            }
            q = fmaf(s, s, q);
        }
        q = group_reduce<BLOCK>(q, red[(row / gridDim.x) & 1], OpSum());
        const float inv = rsqrtf(q / fN + eps);
        const T* src = RES ? res_out : x;
        for (int64_t c = threadIdx.x; c < N; c += BLOCK) {
            const float s = E::load(src + off + c);
            E::store(y + off + c, s * inv * (w ? E::load(w + c) : 1.f));
        }
    }
}

}  // namespace rowops
