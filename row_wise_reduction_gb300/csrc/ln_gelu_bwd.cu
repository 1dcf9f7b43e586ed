// Backward of LayerNorm -> affine -> tanh-GELU ["PyTorch 自定义 CUDA 算子与 Triton
// 编程" §三 FusedLayerNormGELU: the exact gradient of that forward; the page's own
// backward is a stated shortcut]. Per row, xh = (x - mean) rstd, z = xh w + b:
//   dz = dy g'(z);  dxh = dz w
//   dx = rstd (dxh - mean(dxh) - xh mean(dxh xh))
//   dw = sum over rows of dz xh,  db = sum over rows of dz
// The row statistics are recomputed from x (nothing is saved by the forward).
//
// Full rows: the row pipeline with the x and dy rows in each ring slot, three
// group reductions per row, and dw, db partials of each thread's columns kept in
// registers across the CTA's rows; other layouts: a looped CTA-per-row kernel
// that accumulates its partials in the workspace. A last kernel adds the
// per-CTA partials in a fixed order (deterministic dw, db).
#include "rowops_launch.h"
#include "tma_inst.cuh"
#include "tma_rms_kernels.cuh"

namespace rowops {

// d/dz of gelu_tanh_approx. With e = 2^a = exp(-2u) (a as in the forward) and
// s = 1 / (1 + e) = 0.5 (1 + tanh u): 1 - tanh(u)^2 = 4 s (1 - s) and
// s (1 - s) = e s^2 (no cancellation), so
//   g'(z) = s + 2 z e s^2 du/dz,   du/dz = k0 (1 + 3 k1 z^2).
__device__ __forceinline__ float gelu_tanh_grad(float z) {
    constexpr float k0 = 0.79788456f, k1 = 0.044715f;
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    const float z2 = z * z;
    const float e = ex2_approx(fmaf(c1, z2, c0) * z);
    const float s = rcp_approx(1.f + e);
    const float du = k0 * fmaf(3.f * k1, z2, 1.f);
    return fmaf(2.f * z * e * s * s, du, s);
}

// Full rows, one row group (TPR threads) per CTA; VPT vectors per thread, so a
// thread owns the columns of vectors k = t + j * TPR in every row.
template <typename T, int TPR, int VPT>
__global__ void __launch_bounds__(TPR)
    ln_gelu_bwd_tma_kernel(const T* x, const T* dy, const T* w, const T* b, float eps, T* dx, float* part,
                           int64_t M, int N, int64_t ld, int nbuf, unsigned* err, unsigned long long wait_ns,
                           int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_a[TPR / 32];
    __shared__ float red_b[2 * TPR / 32];
    __shared__ float red_c[2 * TPR / 32];
    const GroupPipe p = make_group<TPR, 1>(smem, N, E::kBytes, nbuf, 1, 2);
    const int t = threadIdx.x;
    char* affine = smem + kRingHeader + size_t(nbuf) * p.ring.row_bytes;
    float4* sw4 = reinterpret_cast<float4*>(affine);
    float4* sb4 = sw4 + VPT * H * TPR;
    const T* const src[2] = {x, dy};
    start_rows<T, true, 1, 2>(smem, p, src, M, N, ld, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, 0, N / V, sw4, sb4);
    __syncthreads();
    const uint32_t gstride = p.ring.row_bytes / 2;  // the dy row's place in a slot
    const float fN = float(N);
    float aw[VPT][V], ab[VPT][V];  // dw, db partials of this thread's columns
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int e = 0; e < V; ++e) aw[j][e] = ab[j][e] = 0.f;

    for (int64_t i = 0;; ++i) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = int(i % nbuf);
        int fail = !mbar_wait(p.ring.bar + s, uint32_t((i / nbuf) & 1), wait_ns);
        const char* sbuf = p.ring.slot(s);
        float v[VPT][V], g[VPT][V];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            E::unpack(lds16(sbuf + size_t(k) * 16), v[j]);
            E::unpack(lds16(sbuf + gstride + size_t(k) * 16), g[j]);
#pragma unroll
            for (int e = 0; e < V; ++e) sum += v[j][e];
        }
        sum = row_reduce<TPR>(sum, red_a, p.bar_id, OpSum(), fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            return;
        }
        refill_rows<T, true, 2>(p, s, row, src, M, N, ld, stall_row);
        // statistics as in the forward: variance of the centred row with the
        // residual correction of the fp32 mean
        const float mean = sum / fN;
        float q = 0.f, r = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] -= mean;
                q = fmaf(v[j][e], v[j][e], q);
                r += v[j][e];
            }
        row_reduce_sum2<TPR>(q, r, red_b, p.bar_id, fail);
        const float delta = r / fN;
        const float rstd = rsqrtf(fmaxf(q / fN - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;
        // xh into v, dxh into g; sums of dxh and dxh xh
        float a1 = 0.f, a2 = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float4 ww = sw4[(j * H + h) * TPR + t];
                const float4 bb = sb4[(j * H + h) * TPR + t];
                const float wv[4] = {ww.x, ww.y, ww.z, ww.w}, bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = 4 * h + c;
                    const float xh = fmaf(v[j][e], rstd, shift);
                    const float dz = g[j][e] * gelu_tanh_grad(fmaf(xh, wv[c], bv[c]));
                    aw[j][e] = fmaf(dz, xh, aw[j][e]);
                    ab[j][e] += dz;
                    const float dxh = dz * wv[c];
                    a1 += dxh;
                    a2 = fmaf(dxh, xh, a2);
                    v[j][e] = xh;
                    g[j][e] = dxh;
                }
            }
        row_reduce_sum2<TPR>(a1, a2, red_c, p.bar_id, fail);
        const float m1 = a1 / fN, m2 = a2 / fN;
        T* dxr = dx + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = rstd * (g[j][e] - fmaf(v[j][e], m2, m1));
            st_stream16(dxr + size_t(t + j * TPR) * V, E::pack(o));
        }
    }
    // this CTA's partials: part[blockIdx.x] holds dw then db, N floats each
    float* pw = part + size_t(blockIdx.x) * 2 * N;
    float* pb = pw + N;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int c0 = (t + j * TPR) * V;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            *reinterpret_cast<float4*>(pw + c0 + 4 * h) =
                make_float4(aw[j][4 * h], aw[j][4 * h + 1], aw[j][4 * h + 2], aw[j][4 * h + 3]);
            *reinterpret_cast<float4*>(pb + c0 + 4 * h) =
                make_float4(ab[j][4 * h], ab[j][4 * h + 1], ab[j][4 * h + 2], ab[j][4 * h + 3]);
        }
    }
}

// Any layout: one CTA per row (grid-stride), element-wise coalesced passes.
// Pass 1: shifted sums around x0 (mean, variance without cancellation); pass 2:
// dz, dxh, the row sums of dxh and dxh xh, and this CTA's dw, db partials (the
// column c is only ever touched by thread c mod BLOCK of the CTA, in row order,
// so the sums are deterministic); pass 3 recomputes dxh and writes dx.
template <typename T, int BLOCK>
__global__ void __launch_bounds__(BLOCK)
    ln_gelu_bwd_looped_kernel(const T* x, const T* dy, const T* w, const T* b, float eps, T* dx, float* part,
                              int64_t M, int64_t N, int64_t ld) {
    using E = Elem<T>;
    __shared__ float red[2][2 * BLOCK / 32];
    float* pw = part + size_t(blockIdx.x) * 2 * N;
    float* pb = pw + N;
    const float fN = float(N);
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const T* xr = x + row * ld;
        const T* gr = dy + row * ld;
        const float x0 = E::load(xr);
        float s1 = 0.f, s2 = 0.f;
        for (int64_t c = threadIdx.x; c < N; c += BLOCK) {
            const float d = E::load(xr + c) - x0;
            s1 += d;
            s2 = fmaf(d, d, s2);
        }
        group_reduce_sum2<BLOCK>(s1, s2, red[0]);
        const float m = s1 / fN;
        const float mean = x0 + m;
        const float rstd = rsqrtf(fmaxf(s2 / fN - m * m, 0.f) + eps);
        float a1 = 0.f, a2 = 0.f;
        for (int64_t c = threadIdx.x; c < N; c += BLOCK) {
            const float xh = (E::load(xr + c) - mean) * rstd;
            const float wc = w ? E::load(w + c) : 1.f, bc = b ? E::load(b + c) : 0.f;
            const float dz = E::load(gr + c) * gelu_tanh_grad(fmaf(xh, wc, bc));
            pw[c] = fmaf(dz, xh, pw[c]);
            pb[c] += dz;
            const float dxh = dz * wc;
            a1 += dxh;
            a2 = fmaf(dxh, xh, a2);
        }
        group_reduce_sum2<BLOCK>(a1, a2, red[1]);
        const float m1 = a1 / fN, m2 = a2 / fN;
        T* dxr = dx + row * ld;
        for (int64_t c = threadIdx.x; c < N; c += BLOCK) {
            const float xh = (E::load(xr + c) - mean) * rstd;
            const float wc = w ? E::load(w + c) : 1.f, bc = b ? E::load(b + c) : 0.f;
            const float dxh = E::load(gr + c) * gelu_tanh_grad(fmaf(xh, wc, bc)) * wc;
            E::store(dxr + c, rstd * (dxh - fmaf(xh, m2, m1)));
        }
        // red[0] is next written after red[1]'s barrier above (every thread has
        // read it by then), red[1] after the next row's red[0] barrier
    }
}

// dw[c], db[c]: the sum over the P partials, in order p = 0, 1, ...
__global__ void ln_gelu_bwd_reduce_kernel(const float* part, int P, int N, float* dw, float* db) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= N) return;
    float sw = 0.f, sb = 0.f;
    for (int p = 0; p < P; ++p) {
        sw += part[size_t(p) * 2 * N + c];
        sb += part[size_t(p) * 2 * N + N + c];
    }
    dw[c] = sw;
    db[c] = sb;
}

namespace {

template <typename T, int TPR, int VPT>
cudaError_t launch_bwd_tma(const void* x, const void* dy, const void* w, const void* b, float eps, void* dx,
                           float* part, int64_t M, int64_t N, int64_t ld, int nbuf, int* grid_out,
                           const LaunchCfg& cfg) {
    auto kern = ln_gelu_bwd_tma_kernel<T, TPR, VPT>;
    const size_t smem = kRingHeader + size_t(nbuf) * 2 * ring_row_bytes(N, Elem<T>::kBytes) +
                        tma_affine_bytes<T, TPR, VPT>();
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    int grid = grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg);
    if (grid > kBwdMaxPartials) grid = kBwdMaxPartials;
    *grid_out = grid;
    kern<<<grid, TPR, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy),
                                          static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                          static_cast<T*>(dx), part, M, int(N), ld, nbuf, cfg.dev_error,
                                          cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_looped(const void* x, const void* dy, const void* w, const void* b, float eps, void* dx,
                              float* part, int64_t M, int64_t N, int64_t ld, int* grid_out, const LaunchCfg& cfg) {
    constexpr int BLOCK = 512;
    auto kern = ln_gelu_bwd_looped_kernel<T, BLOCK>;
    int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, 0, M, cfg);
    if (grid > kBwdMaxPartials) grid = kBwdMaxPartials;
    *grid_out = grid;
    cudaError_t e = cudaMemsetAsync(part, 0, size_t(grid) * 2 * N * sizeof(float), cfg.stream);
    if (e != cudaSuccess) return e;
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy),
                                         static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                         static_cast<T*>(dx), part, M, N, ld);
    return cudaGetLastError();
}

// tiles of the row pipeline: TPR in {64, 128, 256, 512}, VPT in {1, 2, 3, 4} with
// at most 16 columns per thread (the dw, db partials live in registers)
template <typename T, int TPR, int VPT>
constexpr TmaBwdLaunch bwd_entry() {
    if constexpr (VPT * Elem<T>::kVec <= 16) return launch_bwd_tma<T, TPR, VPT>;
    else return nullptr;
}
#define ROWOPS_BWD_ROW(T, P) {bwd_entry<T, P, 1>(), bwd_entry<T, P, 2>(), bwd_entry<T, P, 3>(), bwd_entry<T, P, 4>()}

template <typename T>
TmaBwdLaunch bwd_tma_table(int tpr_index, int vpt) {
    static const TmaBwdLaunch t[4][4] = {ROWOPS_BWD_ROW(T, 64), ROWOPS_BWD_ROW(T, 128), ROWOPS_BWD_ROW(T, 256),
                                         ROWOPS_BWD_ROW(T, 512)};
    if (tpr_index < 0 || tpr_index >= 4 || vpt < 1 || vpt > 4) return nullptr;
    return t[tpr_index][vpt - 1];
}
#undef ROWOPS_BWD_ROW

}  // namespace

TmaBwdLaunch ln_gelu_bwd_tma_f32(int tpr_index, int vpt) { return bwd_tma_table<float>(tpr_index, vpt); }
TmaBwdLaunch ln_gelu_bwd_tma_bf16(int tpr_index, int vpt) { return bwd_tma_table<bf16_t>(tpr_index, vpt); }
BwdLaunch ln_gelu_bwd_looped_f32() { return launch_bwd_looped<float>; }
BwdLaunch ln_gelu_bwd_looped_bf16() { return launch_bwd_looped<bf16_t>; }

cudaError_t ln_gelu_bwd_reduce(const float* part, int P, int64_t N, float* dw, float* db, const LaunchCfg& cfg) {
    const int block = 256;
    const int grid = int((N + block - 1) / block);
    ln_gelu_bwd_reduce_kernel<<<grid, block, 0, cfg.stream>>>(part, P, int(N), dw, db);
    return cudaGetLastError();
}

}  // namespace rowops
