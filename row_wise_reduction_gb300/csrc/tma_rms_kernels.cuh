// RMSNorm and fused residual + RMSNorm on the TMA-fed row pipeline
// (tma_row_kernels.cuh): ROWS row groups of TPR threads per CTA, each with its
// own ring of nbuf slots. In the fused form (RES) a slot holds the x row and
// the residual row; the producer issues both bulk copies on the slot's one
// mbarrier, which expects their total bytes. Full rows and general rows (phase
// classes: every row of a CTA has the same head / body / tail split) as for
// LayerNorm+GELU; w is staged once per CTA as fp32 in the thread-major order of
// that split.
//
// Per row: s = x or x + residual (rounded to the I/O type, and written out as
// residual_out), one group reduction of sum(s^2), inv_rms = rsqrt(sum / N +
// eps), y = s * inv_rms * w ["Triton Kernel 实现练习" §4.2, §4.3].
#pragma once

#include "rms_kernels.cuh"
#include "tma_row_kernels.cuh"

namespace rowops {

// w in thread-major fp32 order: float4 slot (j * (V/4) + h) * TPR + t holds
// columns c0 + 4h .. c0 + 4h + 3 of vector k = t + j * TPR (c0 = head + k V);
// vectors k >= nvec get 1.
template <typename T, int TPR, int VPT>
__device__ __forceinline__ void stage_weight_thread_major(const T* w, int head, int nvec, float4* sw4) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4;
    for (int q = threadIdx.x; q < VPT * H * TPR; q += blockDim.x) {
        const int tt = q % TPR, rest = q / TPR, h = rest % H, j = rest / H;
        const int k = tt + j * TPR;
        float4 ww = make_float4(1.f, 1.f, 1.f, 1.f);
        if (k < nvec && w) {
            const int c = head + k * V + 4 * h;
            ww = make_float4(E::load(w + c), E::load(w + c + 1), E::load(w + c + 2), E::load(w + c + 3));
        }
        sw4[q] = ww;
    }
}

// Shared memory after the rings: the thread-major w, then (general rows) the
// weights of the class's head and tail columns (fewer than 2V floats).
template <typename T, int TPR, int VPT>
__host__ __device__ constexpr uint32_t rms_weight_bytes() {
    return uint32_t(VPT) * TPR * Elem<T>::kVec * 4;
}
constexpr uint32_t kRmsExtraBytes = 64;

template <typename T, int TPR, int VPT, bool FULL>
__host__ __device__ constexpr uint32_t rms_stage_bytes() {
    return rms_weight_bytes<T, TPR, VPT>() + (FULL ? 0u : kRmsExtraBytes);
}

// Producer: copy the bodies of row `row` of each of the S inputs into slot s.
template <typename T, bool FULL, int S>
__device__ __forceinline__ void issue_rows(const GroupPipe& p, int s, int64_t row, const T* const* src, int N,
                                           int64_t ld, int64_t stall_row) {
    const RowSpan sp = row_span<T, FULL>(src[0] + row * ld, N);
    const uint32_t bytes = uint32_t(sp.body) * 16u;
    const uint32_t stride = p.ring.row_bytes / S;
    mbar_expect_tx(p.ring.bar + s, S * bytes + stall_extra(row, stall_row));
#pragma unroll
    for (int k = 0; k < S; ++k)
        tma_copy_row(p.ring.slot(s) + k * stride, src[k] + row * ld + sp.head, bytes, p.ring.bar + s);
}

template <typename T, bool FULL, int ROWS, int S>
__device__ __forceinline__ void start_rows(char* smem, const GroupPipe& p, const T* const* src, int64_t M, int N,
                                           int64_t ld, int64_t stall_row) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROWS * p.ring.nbuf; ++s) mbar_init(reinterpret_cast<uint64_t*>(smem) + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (p.producer)
        for (int s = 0; s < p.ring.nbuf; ++s) {
            const int64_t row = p.first + s * p.stride;
            if (row < M) issue_rows<T, FULL, S>(p, s, row, src, N, ld, stall_row);
        }
}

template <typename T, bool FULL, int S>
__device__ __forceinline__ void refill_rows(const GroupPipe& p, int s, int64_t row, const T* const* src, int64_t M,
                                            int N, int64_t ld, int64_t stall_row) {
    if (!p.producer) return;
    const int64_t nxt = row + int64_t(p.ring.nbuf) * p.stride;
    if (nxt < M) {
        fence_proxy_async_smem();
        issue_rows<T, FULL, S>(p, s, nxt, src, N, ld, stall_row);
    }
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool RES>
__global__ void __launch_bounds__(TPR * ROWS)
    rms_tma_kernel(const T* x, const T* res, T* y, T* res_out, const T* w, float eps, int64_t M, int N, int64_t ld,
                   int nbuf, unsigned* err, unsigned long long wait_ns, int64_t stall_row, int unit_rows) {
    using E = Elem<T>;
    constexpr int V = E::kVec, H = V / 4, S = RES ? 2 : 1;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    extern __shared__ __align__(128) char smem[];
    // one reduction per row: two buffers per group used alternately
    __shared__ float red[ROWS][2][TPR / 32];
    __shared__ ClcShared cs;
    const int period = FULL ? 1 : row_phase_period(ld * E::kBytes);
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf, period, S);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    char* staged = smem + kRingHeader + size_t(ROWS) * nbuf * p.ring.row_bytes;
    float4* sw4 = reinterpret_cast<float4*>(staged);
    float* sxw = reinterpret_cast<float*>(staged + rms_weight_bytes<T, TPR, VPT>());
    const uint32_t rstride = p.ring.row_bytes / S;  // the residual row's place in a slot
    const float fN = float(N);
    // the split shared by every row of this CTA's phase class
    const RowSpan sp = row_span<T, FULL>(x + int64_t(p.cls) * ld, N);
    const T* const src[2] = {x, res};
    const bool dynamic = FULL && unit_rows > 0;  // unit_rows 0: static schedule
    DynFeed f{};
    if (dynamic) f = dyn_start<T, ROWS, S>(smem, p, cs, g, src, N, ld, M, stall_row, wait_ns, err, unit_rows);
    else start_rows<T, FULL, ROWS, S>(smem, p, src, M, N, ld, stall_row);
    stage_weight_thread_major<T, TPR, VPT>(w, sp.head, sp.body, sw4);
    if constexpr (!FULL) {
        for (int e = threadIdx.x; e < sp.head + sp.tail; e += blockDim.x)
            sxw[e] = w ? E::load(w + span_extra_col(sp, e, V)) : 1.f;
    }
    __syncthreads();
    const bool has_ex = !FULL && t < sp.head + sp.tail;
    const int ecol = has_ex ? span_extra_col(sp, t, V) : 0;

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int s = rc.slot;
        int64_t row;
        int fail = 0;
        if (dynamic) {
            row = dyn_row(p, cs, g, rc, wait_ns, fail);
            if (row < 0) {  // the end of the work (a failed wait goes on to the reduction below)
                dyn_finish(f, cs, wait_ns);
                return;
            }
        } else {
            row = p.first + i * p.stride;
            if (row >= M) break;
        }
        const int64_t off = row * ld;
        float ex = 0.f;
        if (has_ex) {
            ex = E::load(x + off + ecol);
            if constexpr (RES) ex = E::round(ex + E::load(res + off + ecol));
        }
        if (!dynamic) fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
        const char* sbuf = p.ring.slot(s);

        float v[VPT][V];
        float q = ex * ex;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
                const uint4 xa = lds16(sbuf + size_t(k) * 16);
                uint4 ra = xa;
                if constexpr (RES) ra = lds16(sbuf + rstride + size_t(k) * 16);
                const uint4 packed = residual_sum<T, RES>(xa, ra, v[j]);
                if constexpr (RES) st_stream16(res_out + off + sp.head + size_t(k) * V, packed);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) v[j][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) q = fmaf(v[j][e], v[j][e], q);
        }
        q = row_reduce<TPR>(q, red[g][i & 1], p.bar_id, OpSum(), fail);
        if (fail) {
            if (dynamic) dyn_abandon(p, f, cs, g, i, err, wait_ns);
            else abandon(p, i, M, err, wait_ns);
            return;
        }
        if (dynamic) {
            if (p.producer) dyn_issue<T, ROWS, S>(p, cs, f, g, s, src, N, ld, M, stall_row, wait_ns, err);
        } else {
            refill_rows<T, FULL, S>(p, s, row, src, M, N, ld, stall_row);
        }
        const float inv = rsqrtf(q / fN + eps);
        T* yb = y + off + sp.head;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (FULL || k < sp.body) {
                float o[V];
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float4 ww = sw4[(j * H + h) * TPR + t];
                    o[4 * h + 0] = v[j][4 * h + 0] * inv * ww.x;
                    o[4 * h + 1] = v[j][4 * h + 1] * inv * ww.y;
                    o[4 * h + 2] = v[j][4 * h + 2] * inv * ww.z;
                    o[4 * h + 3] = v[j][4 * h + 3] * inv * ww.w;
                }
                st_stream16(yb + size_t(k) * V, E::pack(o));
            }
        }
        if (has_ex) {
            E::store(y + off + ecol, ex * inv * sxw[t]);
            if constexpr (RES) E::store(res_out + off + ecol, ex);
        }
    }
}

}  // namespace rowops
