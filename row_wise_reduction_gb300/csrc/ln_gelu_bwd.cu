// Backward of LayerNorm -> affine -> tanh-GELU ["PyTorch 自定义 CUDA 算子与 Triton
// 编程" §三 FusedLayerNormGELU: the exact gradient of that forward; the page's own
// backward is a stated shortcut]. Per row, xh = (x - mean) rstd, z = xh w + b:
//   dz = dy g'(z);  dxh = dz w
//   dx = rstd (dxh - mean(dxh) - xh mean(dxh xh))
//   dw = sum over rows of dz xh,  db = sum over rows of dz
// The row statistics are recomputed from x (nothing is saved by the forward).
//
// Full rows: the row pipeline with the x and dy rows in each ring slot and the
// dw, db partials of each thread's columns kept in registers across the CTA's
// rows; where the ring holds at least four slots, three rows at different
// stages share one group reduction per row (ln_gelu_bwd_pipe_kernel), else one
// row at a time with three reductions (ln_gelu_bwd_tma_kernel). Other layouts:
// a looped CTA-per-row kernel that accumulates its partials in the workspace.
// A last kernel adds the per-CTA partials in a fixed order (deterministic dw, db).
#include "rowops_launch.h"
#include "tma_inst.cuh"
#include "tma_rms_kernels.cuh"
#include "tmem.cuh"

namespace rowops {

// d/dz of gelu_tanh_approx. With e = 2^a = exp(-2u) (a as in the forward) and
// s = 1 / (1 + e) = 0.5 (1 + tanh u): 1 - tanh(u)^2 = 4 s (1 - s) and
// s (1 - s) = e s^2 (no cancellation), so
//   g'(z) = s + (e s) s (2 z du/dz),   du/dz = k0 (1 + 3 k1 z^2).
// a is clamped at 126: below z ~ -10 e would overflow and (e s) s turn into
// inf * 0; with the clamp g' comes out ~1e-36 there, the true value being smaller.
__device__ __forceinline__ float gelu_tanh_grad(float z) {
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    constexpr float d0 = float(2.0 * 0.79788456), d1 = float(2.0 * 3.0 * 0.79788456 * 0.044715);
    const float z2 = z * z;
    const float e = ex2_approx(fminf(fmaf(c1, z2, c0) * z, 126.f));
    const float s = rcp_approx(1.f + e);
    return fmaf((e * s) * s, z * fmaf(d1, z2, d0), s);
}

// Sums over the TPR threads of a row group of s and of v[0..3], with one named
// barrier. In a warp s is added by a butterfly and v by a reduce-scatter: the
// offsets 16 and 8 split the four values between the lane halves and quarters,
// 4, 2 and 1 finish, so lane l holds the warp's sum of v[l / 8]. Lanes 0, 8,
// 16 and 24 store those (lane 0 also s); after the barrier lane l loads the
// sums of warp l mod W and a butterfly over W lanes adds the warps.
template <int TPR>
__device__ __forceinline__ void row_reduce_sum5(float& s, float (&v)[4], float (*red)[8], int bar_id, int& fail) {
    constexpr int W = TPR / 32;
    const int lane = threadIdx.x & 31;
    const bool h16 = lane & 16, h8 = lane & 8;
    float k0 = h16 ? v[2] : v[0], k1 = h16 ? v[3] : v[1];
    k0 += __shfl_xor_sync(0xffffffffu, h16 ? v[0] : v[2], 16);
    k1 += __shfl_xor_sync(0xffffffffu, h16 ? v[1] : v[3], 16);
    float k = h8 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) k += __shfl_xor_sync(0xffffffffu, k, o);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int w = (threadIdx.x % TPR) >> 5;
    if ((lane & 7) == 0) red[w][lane >> 3] = k;
    if (lane == 0) red[w][4] = s;
    fail = group_bar_or(bar_id, TPR, fail);
    const float4 r = *reinterpret_cast<const float4*>(red[lane % W]);
    float o5[5] = {r.x, r.y, r.z, r.w, red[lane % W][4]};
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1)
#pragma unroll
        for (int q = 0; q < 5; ++q) o5[q] += __shfl_xor_sync(0xffffffffu, o5[q], o);
    v[0] = o5[0];
    v[1] = o5[1];
    v[2] = o5[2];
    v[3] = o5[3];
    s = o5[4];
}

// gelu_tanh_grad of two values with packed fp32 pairs.
__device__ __forceinline__ float2 gelu_tanh_grad2(float2 z) {
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    constexpr float d0 = float(2.0 * 0.79788456), d1 = float(2.0 * 3.0 * 0.79788456 * 0.044715);
    const float2 z2 = f2_mul(z, z);
    const float2 a = f2_mul(f2_fma(f2(c1), z2, f2(c0)), z);
    float2 e = make_float2(ex2_approx(fminf(a.x, 126.f)), ex2_approx(fminf(a.y, 126.f)));
    const float2 e1 = f2_add(e, f2(1.f));
    const float2 sg = make_float2(rcp_approx(e1.x), rcp_approx(e1.y));
    e = f2_mul(f2_mul(e, sg), sg);
    return f2_fma(e, f2_mul(f2_fma(f2(d1), z2, f2(d0)), z), sg);
}

// -gelu_tanh_grad of two values, with fewer instructions: n = -s comes from
// the reciprocal of -(1 + e), and s (1 - s) = -(n + n^2) is one fused
// multiply-add with an exact product, so
//   -g'(z) = n + (n + n^2) (2 z du/dz).
// Below z ~ -10 e overflows to +inf and n = -0: -g' = -0, with no clamp (no
// inf * 0 arises). For large z, 1 + e carries the rounding of 1 (2^-24
// absolute), which the small 1 - s takes in relative terms: the slope is then
// off by at most ~1.2e-6 relative (z ~ 4, where e reaches 2^-24; the clamped
// form above is exact there up to the approximate exp2 and reciprocal).
__device__ __forceinline__ float2 gelu_tanh_grad2_neg(float2 z) {
    constexpr float c0 = float(-2.0 * 0.79788456 * kLog2e);
    constexpr float c1 = float(-2.0 * 0.79788456 * 0.044715 * kLog2e);
    constexpr float d0 = float(2.0 * 0.79788456), d1 = float(2.0 * 3.0 * 0.79788456 * 0.044715);
    const float2 z2 = f2_mul(z, z);
    const float2 a = f2_mul(f2_fma(f2(c1), z2, f2(c0)), z);
    const float2 nd = f2_fma(make_float2(ex2_approx(a.x), ex2_approx(a.y)), f2(-1.f), f2(-1.f));
    const float2 n = make_float2(rcp_approx(nd.x), rcp_approx(nd.y));
    return f2_fma(f2_fma(n, n, n), f2_mul(f2_fma(f2(d1), z2, f2(d0)), z), n);
}

// Full rows on a row pipeline of four stages, one row group (TPR threads) per
// CTA, one barrier per row. At step k the group
//   C: writes dx of row k-3 (xh, dxh kept in registers from its stage A),
//   A: reads x, dy of row k-2 and forms xh, dz, dxh, the dw, db partials and
//      the sums of dxh and dxh xh,
//   Q: turns its own shifted sums of row k-1 into sum (x - mean)^2 and
//      sum (x - mean) over its columns (no element is read again),
//   S: waits for row k and sums x - c and (x - c)^2 over its n_t columns,
//      c the first of them (so the terms of Q cancel at most ~2 n_t-fold:
//      c itself contributes (c - mean)^2 to Q),
// and one reduction adds sum x, the two sums of Q and the two of A over the
// group. The variance of the centred row then gets the residual correction of
// the fp32 mean, as in the forward. Rows k-2 .. k stay in the ring, the slot of
// row k-2 is refilled after the barrier: nbuf - 3 rows are in flight beyond the
// ones being worked on. Elementwise arithmetic runs on packed fp32 pairs.
template <typename T, int TPR, int VPT>
__global__ void __launch_bounds__(TPR)
    ln_gelu_bwd_pipe_kernel(const T* x, const T* dy, const T* w, const T* b, float eps, T* dx, float* part,
                            int64_t M, int N, int64_t ld, int nbuf, unsigned* err, unsigned long long wait_ns,
                            int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4, P = V / 2;
    constexpr float kNt = float(VPT * V);  // columns of a thread
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    __shared__ __align__(16) float red[2][TPR / 32][8];
    const GroupPipe p = make_group<TPR, 1>(smem, N, E::kBytes, nbuf, 1, 2);
    const int t = threadIdx.x;
    char* affine = smem + kRingHeader + size_t(nbuf) * p.ring.row_bytes;
    const float4* sw4 = reinterpret_cast<const float4*>(affine);
    const float4* sb4 = sw4 + VPT * H * TPR;
    const T* const src[2] = {x, dy};
    start_rows<T, true, 1, 2>(smem, p, src, M, N, ld, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, 0, N / V, reinterpret_cast<float4*>(affine),
                                           reinterpret_cast<float4*>(affine) + VPT * H * TPR);
    __syncthreads();
    const uint32_t gstride = p.ring.row_bytes / 2;  // the dy row's place in a slot
    const float fN = float(N);
    const int64_t n = p.first < M ? (M - 1 - p.first) / p.stride + 1 : 0;  // rows of this CTA
    float2 aw[VPT][P], ab[VPT][P];   // dw, db partials of this thread's columns
    float2 xh[VPT][P], dxh[VPT][P];  // of the row between its stages A and C
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int q = 0; q < P; ++q) aw[j][q] = ab[j][q] = xh[j][q] = dxh[j][q] = f2(0.f);
    float c_q = 0.f, s_q = 0.f, q_q = 0.f, mean_q = 0.f;  // stage Q's row: shift, shifted sums, mean
    float mean_a = 0.f, rstd_a = 0.f, shift_a = 0.f;      // stage A's row
    float rstd_c = 0.f, m1_c = 0.f, m2_c = 0.f;           // stage C's row (-m1, -m2 times rstd)

    RingCursor rk;  // ring slot and phase parity of row k
    for (int64_t k = 0;; ++k, rk.next(nbuf)) {
        const int sa = rk.slot >= 2 ? rk.slot - 2 : rk.slot - 2 + nbuf;  // slot of row k-2 (nbuf >= 4)
        if (k >= 3) {  // C: dx of row k-3
            T* dxr = dx + (p.first + (k - 3) * p.stride) * ld;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                float o[V];
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    const float2 r = f2_fma(f2(rstd_c), dxh[j][q], f2_fma(xh[j][q], f2(m2_c), f2(m1_c)));
                    o[2 * q] = r.x;
                    o[2 * q + 1] = r.y;
                }
                st_stream16(dxr + size_t(t + j * TPR) * V, E::pack(o));
            }
        }
        if (k == n + 2) break;
        float sv[4] = {0.f, 0.f, 0.f, 0.f};  // Q: sum (x - mean)^2, sum (x - mean); A: sum dxh, sum dxh xh
        float s1 = 0.f;                      // S: sum x
        if (k >= 2 && k - 2 < n) {           // A: row k-2
            const char* sb = p.ring.slot(sa);
            float2 a1 = f2(0.f), a2 = f2(0.f);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                float xv[V], gv[V];
                E::unpack(lds16(sb + size_t(t + j * TPR) * 16), xv);
                E::unpack(lds16(sb + gstride + size_t(t + j * TPR) * 16), gv);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float4 ww = sw4[(j * H + h) * TPR + t];
                    const float4 bb = sb4[(j * H + h) * TPR + t];
                    const float2 wv[2] = {make_float2(ww.x, ww.y), make_float2(ww.z, ww.w)};
                    const float2 bv[2] = {make_float2(bb.x, bb.y), make_float2(bb.z, bb.w)};
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int q = 2 * h + c;
                        const float2 xq = make_float2(xv[2 * q], xv[2 * q + 1]);
                        const float2 gq = make_float2(gv[2 * q], gv[2 * q + 1]);
                        const float2 xhv = f2_fma(f2_add(xq, f2(-mean_a)), f2(rstd_a), f2(shift_a));
                        const float2 dz = f2_mul(gq, gelu_tanh_grad2(f2_fma(xhv, wv[c], bv[c])));
                        aw[j][q] = f2_fma(dz, xhv, aw[j][q]);
                        ab[j][q] = f2_add(ab[j][q], dz);
                        const float2 d = f2_mul(dz, wv[c]);
                        a1 = f2_add(a1, d);
                        a2 = f2_fma(d, xhv, a2);
                        xh[j][q] = xhv;
                        dxh[j][q] = d;
                    }
                }
            }
            sv[2] = a1.x + a1.y;
            sv[3] = a2.x + a2.y;
        }
        if (k >= 1 && k - 1 < n) {  // Q: row k-1, from this thread's sums around c
            const float d = c_q - mean_q;
            sv[0] = fmaf(d, fmaf(kNt, d, 2.f * s_q), q_q);  // sum (x - c + d)^2
            sv[1] = fmaf(kNt, d, s_q);                      // sum (x - c + d)
        }
        int fail = 0;
        if (k < n) {  // S: row k
            fail = !mbar_wait(p.ring.bar + rk.slot, rk.parity, wait_ns);
            const char* ss = p.ring.slot(rk.slot);
            float2 s2 = f2(0.f), q2 = f2(0.f);
            float xv[V];
            E::unpack(lds16(ss + size_t(t) * 16), xv);
            c_q = xv[0];
            const float2 nc = f2(-c_q);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                if (j > 0) E::unpack(lds16(ss + size_t(t + j * TPR) * 16), xv);
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    const float2 e = f2_add(make_float2(xv[2 * q], xv[2 * q + 1]), nc);
                    s2 = f2_add(s2, e);
                    q2 = f2_fma(e, e, q2);
                }
            }
            s_q = s2.x + s2.y;
            q_q = q2.x + q2.y;
            s1 = fmaf(kNt, c_q, s_q);
        }
        row_reduce_sum5<TPR>(s1, sv, red[k & 1], p.bar_id, fail);
        if (fail) {  // row k's copy never completed: wait (bounded) for the copies issued
            if (p.producer) {
                // issued: rows 0 .. nbuf - 1 at the start, row j - 2 + nbuf after step j >= 2
                int64_t last = k >= 3 ? k - 3 + nbuf : int64_t(nbuf) - 1;
                if (last > n - 1) last = n - 1;
                for (int64_t i = k; i <= last; ++i)
                    mbar_wait(p.ring.bar + (i % nbuf), uint32_t((i / nbuf) & 1), wait_ns);
                atomicExch(err, kDeviceErrTimeout);
            }
            return;
        }
        if (k >= 2 && k - 2 < n)  // stage A is done with row k-2's slot
            refill_rows<T, true, 2>(p, sa, p.first + (k - 2) * p.stride, src, M, N, ld, stall_row);
        rstd_c = rstd_a;
        m1_c = -rstd_a * (sv[2] / fN);
        m2_c = -rstd_a * (sv[3] / fN);
        const float delta = sv[1] / fN;
        mean_a = mean_q;
        rstd_a = rsqrtf(fmaxf(sv[0] / fN - delta * delta, 0.f) + eps);
        shift_a = -delta * rstd_a;
        mean_q = s1 / fN;
    }
    float* pw = part + size_t(blockIdx.x) * 2 * N;
    float* pb = pw + N;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int c0 = (t + j * TPR) * V;
#pragma unroll
        for (int h = 0; h < H; ++h) {
            *reinterpret_cast<float4*>(pw + c0 + 4 * h) =
                make_float4(aw[j][2 * h].x, aw[j][2 * h].y, aw[j][2 * h + 1].x, aw[j][2 * h + 1].y);
            *reinterpret_cast<float4*>(pb + c0 + 4 * h) =
                make_float4(ab[j][2 * h].x, ab[j][2 * h].y, ab[j][2 * h + 1].x, ab[j][2 * h + 1].y);
        }
    }
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

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = rc.slot;
        int fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
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

// TMEM columns of the TMEM-partials kernel: 2 VPT V per warp (the dw and db
// partials of its threads' columns), warps w and w + 4 in the same lane
// quarter, rounded up to a power of two >= 32 (the allocation unit).
template <typename T, int TPR, int VPT, int ROWS>
__host__ __device__ constexpr uint32_t bwd_tmem_cols() {
    const uint32_t need = uint32_t(TPR * ROWS / 128) * 2u * uint32_t(VPT * Elem<T>::kVec);
    uint32_t c = 32;
    while (c < need) c <<= 1;
    return c;
}

// Full rows, ROWS row groups of TPR threads per CTA, each group one row at a
// time with three group reductions per row (as ln_gelu_bwd_tma_kernel), and
// the dw, db partials of each thread's columns kept in tensor memory (TMEM)
// across the CTA's rows instead of in registers. Registers then hold one row
// (x and dy, later xh and dxh) and no partials, so a CTA of 512 threads runs
// two or four independent row groups: while one group waits at a reduction's
// barrier, the others compute, where the register-partial kernels have one
// group of 512 threads per SM and idle during each of its reductions. Per row
// and vector of a thread, the partials of its V columns come in with one TMEM
// load issued before that vector's arithmetic, and go back with one store.
// Each group's partials go to their own slot of `part` (blockIdx.x * ROWS + g).
// Every thread reaches the final CTA barrier (a group whose wait gave up
// leaves its row loop, it does not return), after which warp 0 frees TMEM.
template <typename T, int TPR, int VPT, int ROWS>
__global__ void __launch_bounds__(TPR * ROWS, 1)
    ln_gelu_bwd_tmem_kernel(const T* x, const T* dy, const T* w, const T* b, float eps, T* dx, float* part,
                            int64_t M, int N, int64_t ld, int nbuf, unsigned* err, unsigned long long wait_ns,
                            int64_t stall_row) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4, P = V / 2, NE = VPT * V;
    constexpr uint32_t kCols = bwd_tmem_cols<T, TPR, VPT, ROWS>();
    static_assert(TPR % 128 == 0, "a row group spans the four TMEM lane quarters");
    static_assert(kCols <= 256, "at most half of TMEM, so two CTAs on one SM never wait for each other");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_a[ROWS][TPR / 32];
    __shared__ __align__(16) float2 red_b[ROWS][TPR / 32];
    __shared__ __align__(16) float2 red_c[ROWS][TPR / 32];
    __shared__ uint32_t tmem_base;
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf, 1, 2);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR, warp = threadIdx.x >> 5;
    char* affine = smem + kRingHeader + size_t(ROWS) * nbuf * p.ring.row_bytes;
    const float4* sw4 = reinterpret_cast<const float4*>(affine);
    const float4* sb4 = sw4 + VPT * H * TPR;
    const T* const src[2] = {x, dy};
    if (warp == 0) tmem_alloc(&tmem_base, kCols);
    start_rows<T, true, ROWS, 2>(smem, p, src, M, N, ld, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, 0, N / V, reinterpret_cast<float4*>(affine),
                                           reinterpret_cast<float4*>(affine) + VPT * H * TPR);
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    // this thread's lane and its 2 NE columns: per vector j, the dw then the db
    // partials of the vector's V columns
    const uint32_t tm = tmem_base + ((32u * uint32_t(warp & 3)) << 16) + uint32_t(warp >> 2) * (2u * NE);
    {
        float zero[2 * V];
#pragma unroll
        for (int e = 0; e < 2 * V; ++e) zero[e] = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) tmem_st<2 * V>(tm + 2u * V * j, zero);
        tmem_wait_st();
    }
    const uint32_t gstride = p.ring.row_bytes / 2;  // the dy row's place in a slot
    const float fN = float(N);
    bool ok = true;
    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = rc.slot;
        int fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
        const char* sbuf = p.ring.slot(s);
        float2 v[VPT][P], gd[VPT][P];  // x then xh; dy then dxh
        float2 s2 = f2(0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            float xv[V], gv[V];
            E::unpack(lds16(sbuf + size_t(k) * 16), xv);
            E::unpack(lds16(sbuf + gstride + size_t(k) * 16), gv);
#pragma unroll
            for (int q = 0; q < P; ++q) {
                v[j][q] = make_float2(xv[2 * q], xv[2 * q + 1]);
                gd[j][q] = make_float2(gv[2 * q], gv[2 * q + 1]);
                s2 = f2_add(s2, v[j][q]);
            }
        }
        const float sum = row_reduce<TPR>(s2.x + s2.y, red_a[g], p.bar_id, OpSum(), fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            ok = false;
            break;
        }
        refill_rows<T, true, 2>(p, s, row, src, M, N, ld, stall_row);
        // statistics as in the forward: variance of the centred row with the
        // residual correction of the fp32 mean
        const float mean = sum / fN;
        float2 q2 = f2(0.f), r2 = f2(0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j)
#pragma unroll
            for (int q = 0; q < P; ++q) {
                v[j][q] = f2_add(v[j][q], f2(-mean));
                q2 = f2_fma(v[j][q], v[j][q], q2);
                r2 = f2_add(r2, v[j][q]);
            }
        float qs = q2.x + q2.y, rs = r2.x + r2.y;
        row_reduce_sum2_packed<TPR>(qs, rs, red_b[g], p.bar_id, fail);
        const float delta = rs / fN;
        const float rstd = rsqrtf(fmaxf(qs / fN - delta * delta, 0.f) + eps);
        const float shift = -delta * rstd;
        // xh into v, -dxh into gd; the sums of -dxh and -dxh xh; the partials,
        // negated (from -dz = dy (-g'), gelu_tanh_grad2_neg: every sign flip is
        // exact, so dx and the sums are those of the positive form)
        float2 a1 = f2(0.f), a2 = f2(0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float acc[2 * V];
            tmem_ld<2 * V>(tm + 2u * V * j, acc);
            float2 dz[P];
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float4 ww = sw4[(j * H + h) * TPR + t];
                const float4 bb = sb4[(j * H + h) * TPR + t];
                const float2 wv[2] = {make_float2(ww.x, ww.y), make_float2(ww.z, ww.w)};
                const float2 bv[2] = {make_float2(bb.x, bb.y), make_float2(bb.z, bb.w)};
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int q = 2 * h + c;
                    const float2 xhv = f2_fma(v[j][q], f2(rstd), f2(shift));
                    dz[q] = f2_mul(gd[j][q], gelu_tanh_grad2_neg(f2_fma(xhv, wv[c], bv[c])));
                    const float2 d = f2_mul(dz[q], wv[c]);
                    a1 = f2_add(a1, d);
                    a2 = f2_fma(d, xhv, a2);
                    v[j][q] = xhv;
                    gd[j][q] = d;
                }
            }
            tmem_wait_ld(acc);
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const float2 aw = f2_fma(dz[q], v[j][q], make_float2(acc[2 * q], acc[2 * q + 1]));
                const float2 ab = f2_add(dz[q], make_float2(acc[V + 2 * q], acc[V + 2 * q + 1]));
                acc[2 * q] = aw.x;
                acc[2 * q + 1] = aw.y;
                acc[V + 2 * q] = ab.x;
                acc[V + 2 * q + 1] = ab.y;
            }
            tmem_st<2 * V>(tm + 2u * V * j, acc);
        }
        float s1 = a1.x + a1.y, s2b = a2.x + a2.y;  // -sum dxh, -sum dxh xh
        row_reduce_sum2_packed<TPR>(s1, s2b, red_c[g], p.bar_id, fail);
        // dx = rstd (dxh - mean(dxh) - xh mean(dxh xh)) from the negated terms
        const float nm1 = rstd * (s1 / fN), nm2 = rstd * (s2b / fN);
        T* dxr = dx + row * ld;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float o[V];
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const float2 r = f2_fma(f2(-rstd), gd[j][q], f2_fma(v[j][q], f2(nm2), f2(nm1)));
                o[2 * q] = r.x;
                o[2 * q + 1] = r.y;
            }
            st_stream16(dxr + size_t(t + j * TPR) * V, E::pack(o));
        }
        tmem_wait_st();  // the next row's loads read these columns
    }
    if (ok) {  // this group's partials: part[blockIdx.x * ROWS + g] holds dw then db, N floats each
        float* pw = part + (size_t(blockIdx.x) * ROWS + g) * 2 * N;
        float* pb = pw + N;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float acc[2 * V];
            tmem_ld<2 * V>(tm + 2u * V * j, acc);
            tmem_wait_ld(acc);
            const int c0 = (t + j * TPR) * V;
#pragma unroll
            for (int h = 0; h < H; ++h) {  // the partials were kept negated
                *reinterpret_cast<float4*>(pw + c0 + 4 * h) =
                    make_float4(-acc[4 * h], -acc[4 * h + 1], -acc[4 * h + 2], -acc[4 * h + 3]);
                *reinterpret_cast<float4*>(pb + c0 + 4 * h) =
                    make_float4(-acc[V + 4 * h], -acc[V + 4 * h + 1], -acc[V + 4 * h + 2], -acc[V + 4 * h + 3]);
            }
        }
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 0) {
        tmem_fence_after();
        tmem_free(tmem_base, kCols);
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

// dw[c], db[c]: the sums over the P partials. A CTA takes 32 columns of dw or
// db; thread (x, y) adds the partials p = y, y + 32, ... of column x in order,
// then the 32 sums are added in order of y: a fixed order, so the result does
// not depend on scheduling.
__global__ void __launch_bounds__(1024) ln_gelu_bwd_reduce_kernel(const float* part, int P, int N, float* dw,
                                                                  float* db) {
    __shared__ float acc[32][33];
    const int c = blockIdx.x * 32 + threadIdx.x;
    const int which = blockIdx.y;  // 0: dw, 1: db
    float s = 0.f;
    if (c < N)
        for (int p = threadIdx.y; p < P; p += 32) s += part[size_t(p) * 2 * N + size_t(which) * N + c];
    acc[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < N) {
        float t = 0.f;
#pragma unroll 8
        for (int y = 0; y < 32; ++y) t += acc[y][threadIdx.x];
        (which ? db : dw)[c] = t;
    }
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
    int grid = cap_ctas(grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg), 4, cfg);  // as before
    if (grid > bwd_max_partials(N)) grid = bwd_max_partials(N);
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
    if (grid > bwd_max_partials(N)) grid = bwd_max_partials(N);
    *grid_out = grid;
    cudaError_t e = cudaMemsetAsync(part, 0, size_t(grid) * 2 * N * sizeof(float), cfg.stream);
    if (e != cudaSuccess) return e;
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy),
                                         static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                         static_cast<T*>(dx), part, M, N, ld);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT>
cudaError_t launch_bwd_pipe(const void* x, const void* dy, const void* w, const void* b, float eps, void* dx,
                            float* part, int64_t M, int64_t N, int64_t ld, int nbuf, int* grid_out,
                            const LaunchCfg& cfg) {
    auto kern = ln_gelu_bwd_pipe_kernel<T, TPR, VPT>;
    const size_t smem = kRingHeader + size_t(nbuf) * 2 * ring_row_bytes(N, Elem<T>::kBytes) +
                        tma_affine_bytes<T, TPR, VPT>();
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    int grid = cap_ctas(grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg), 4, cfg);  // as before
    if (grid > bwd_max_partials(N)) grid = bwd_max_partials(N);
    *grid_out = grid;
    kern<<<grid, TPR, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy),
                                          static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                          static_cast<T*>(dx), part, M, int(N), ld, nbuf, cfg.dev_error,
                                          cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, int ROWS>
cudaError_t launch_bwd_tmem(const void* x, const void* dy, const void* w, const void* b, float eps, void* dx,
                            float* part, int64_t M, int64_t N, int64_t ld, int nbuf, int* grid_out,
                            const LaunchCfg& cfg) {
    auto kern = ln_gelu_bwd_tmem_kernel<T, TPR, VPT, ROWS>;
    const size_t smem = kRingHeader + size_t(ROWS) * nbuf * 2 * ring_row_bytes(N, Elem<T>::kBytes) +
                        tma_affine_bytes<T, TPR, VPT>();
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    int grid = grid_for(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, (M + ROWS - 1) / ROWS, cfg);
    const int cap = bwd_max_partials(N) / ROWS;  // each group leaves its own partials
    if (grid > cap) grid = cap;
    *grid_out = grid * ROWS;
    kern<<<grid, TPR * ROWS, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(dy),
                                                 static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                                 static_cast<T*>(dx), part, M, int(N), ld, nbuf, cfg.dev_error,
                                                 cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

// TMEM-partials tiles: 512 threads per CTA as two groups of 256 or four of
// 128, VPT in {1, 2, 4} with at most 32 columns per thread
template <typename T, int TPR, int VPT>
constexpr TmaBwdLaunch bwd_tmem_entry() {
    if constexpr (VPT * Elem<T>::kVec > 32) return nullptr;
    else return launch_bwd_tmem<T, TPR, VPT, 512 / TPR>;
}

template <typename T>
TmaBwdLaunch bwd_tmem_table(int tpr, int vpt) {
    static const TmaBwdLaunch t[2][3] = {
        {bwd_tmem_entry<T, 128, 1>(), bwd_tmem_entry<T, 128, 2>(), bwd_tmem_entry<T, 128, 4>()},
        {bwd_tmem_entry<T, 256, 1>(), bwd_tmem_entry<T, 256, 2>(), bwd_tmem_entry<T, 256, 4>()}};
    const int i = tpr == 128 ? 0 : (tpr == 256 ? 1 : -1);
    const int j = vpt == 1 ? 0 : (vpt == 2 ? 1 : (vpt == 4 ? 2 : -1));
    return i < 0 || j < 0 ? nullptr : t[i][j];
}

// tiles of the row pipeline: TPR in {64, 128, 256, 512}, VPT in {1, 2, 3, 4} with
// at most 16 columns per thread (the dw, db partials live in registers); TPR
// 1024 with at most 8 columns per thread for the three-stage kernel (64
// registers a thread)
template <typename T, int TPR, int VPT, bool PIPE>
constexpr TmaBwdLaunch bwd_entry() {
    if constexpr (VPT * Elem<T>::kVec > 16 || (TPR > 512 && (!PIPE || VPT * Elem<T>::kVec > 8))) return nullptr;
    else if constexpr (PIPE) return launch_bwd_pipe<T, TPR, VPT>;
    else return launch_bwd_tma<T, TPR, VPT>;
}
#define ROWOPS_BWD_ROW(T, P, PIPE) \
    {bwd_entry<T, P, 1, PIPE>(), bwd_entry<T, P, 2, PIPE>(), bwd_entry<T, P, 3, PIPE>(), bwd_entry<T, P, 4, PIPE>()}

template <typename T>
TmaBwdLaunch bwd_tma_table(int tpr_index, int vpt, bool pipe) {
    static const TmaBwdLaunch t[2][5][4] = {
        {ROWOPS_BWD_ROW(T, 64, false), ROWOPS_BWD_ROW(T, 128, false), ROWOPS_BWD_ROW(T, 256, false),
         ROWOPS_BWD_ROW(T, 512, false), ROWOPS_BWD_ROW(T, 1024, false)},
        {ROWOPS_BWD_ROW(T, 64, true), ROWOPS_BWD_ROW(T, 128, true), ROWOPS_BWD_ROW(T, 256, true),
         ROWOPS_BWD_ROW(T, 512, true), ROWOPS_BWD_ROW(T, 1024, true)}};
    if (tpr_index < 0 || tpr_index >= 5 || vpt < 1 || vpt > 4) return nullptr;
    return t[pipe ? 1 : 0][tpr_index][vpt - 1];
}
#undef ROWOPS_BWD_ROW

}  // namespace

TmaBwdLaunch ln_gelu_bwd_tma_f32(int tpr_index, int vpt, bool pipe) {
    return bwd_tma_table<float>(tpr_index, vpt, pipe);
}
TmaBwdLaunch ln_gelu_bwd_tma_bf16(int tpr_index, int vpt, bool pipe) {
    return bwd_tma_table<bf16_t>(tpr_index, vpt, pipe);
}
TmaBwdLaunch ln_gelu_bwd_tmem_f32(int tpr, int vpt) { return bwd_tmem_table<float>(tpr, vpt); }
TmaBwdLaunch ln_gelu_bwd_tmem_bf16(int tpr, int vpt) { return bwd_tmem_table<bf16_t>(tpr, vpt); }
BwdLaunch ln_gelu_bwd_looped_f32() { return launch_bwd_looped<float>; }
BwdLaunch ln_gelu_bwd_looped_bf16() { return launch_bwd_looped<bf16_t>; }

cudaError_t ln_gelu_bwd_reduce(const float* part, int P, int64_t N, float* dw, float* db, const LaunchCfg& cfg) {
    const dim3 grid(unsigned((N + 31) / 32), 2);
    ln_gelu_bwd_reduce_kernel<<<grid, dim3(32, 32), 0, cfg.stream>>>(part, P, int(N), dw, db);
    return cudaGetLastError();
}

}  // namespace rowops
