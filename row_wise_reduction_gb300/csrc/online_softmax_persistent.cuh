// Single-read split-row online softmax for very long rows [Triton Kernel 实现练习
// §2.5 split_online_softmax; 第 6 讲 §7.2 Online Softmax].
//
// The two-launch form (online_softmax_kernels.cuh) reads x twice: once for the
// chunk partials, once more to normalise. The forms here keep every chunk on
// chip between the two passes, so x is read once and y written once:
//   - split_grouped_kernel (below; the default for large batches of long
//     rows): each row spread over a group of CTAs;
//   - split_persistent_kernel / split_l2_kernel (on request): every CTA holds
//     a column slice of every row, staged in shared memory or in L2.
//
// Column slices: a cooperative grid of G CTAs (all resident at once). CTA c owns the column
// slice [c nvec / G, (c + 1) nvec / G) (16-byte vectors) of every row, and warp
// w of the CTA the w-th sixteenth of that slice. The CTA keeps its slices of NS
// consecutive rows in a ring of shared-memory stages, filled by bulk copies,
// and runs a software pipeline over steps s = 0, 1, ...:
//   partial   row s      : each warp folds its part of the slice into a partial
//                          (m, d) = (max, sum exp(x - m)) and stores it in the
//                          row's slot c * 16 + w;
//   merge     row s - L/2: if c owns that row (row mod G), wait (bounded) until
//                          all G * 16 slots of the row are set, merge them in
//                          slot order (m = max m_i, d = sum d_i exp(m_i - m),
//                          d_i = 0 skipped) and store the row's (m, d);
//   normalise row s - L  : with the row's (m, d) (fetched before the step's one
//                          barrier), write y = exp(x - m) / d from the stage;
//                          the stage then takes row s - L + NS.
// Every wait is for data that other CTAs produced L/2 steps earlier, so it
// normally succeeds on its first look. Each slot and each row result is one
// 64-bit word written by a single relaxed 64-bit store over a sentinel (all
// one bits) that the host fills in before the launch: the data is its own flag
// and needs no fence. A CTA never waits on work of a later step, and all CTAs
// are resident, so every wait ends. A wait that runs past its limit records
// ROWOPS_ERR_TIMEOUT and raises the abort word, which makes every other wait
// give up at once; each CTA then drains its copies in flight and returns.
//
// Workspace: [0, 256) header (word 0 status, word 1 abort), then M row results
// (64-bit, padded to 256 bytes), then 64-bit warp partials [M][G * 16].
#pragma once

#include <cooperative_groups.h>

#include "grouped_plan.h"
#include "reduce_kernels.cuh"
#include "row_pipeline.cuh"
#include "softmax_kernels.cuh"

namespace rowops {

constexpr unsigned long long kSlotEmpty = ~0ull;
constexpr int kPersistBlock = 512;
constexpr int kPersistWarps = kPersistBlock / 32;
constexpr int kPersistMaxSlots = 4096;  // G * 16 partials per row, at most

// (m, d) as one 64-bit word, m in the low half; computed NaNs become the
// canonical quiet NaN, so a stored pair is never the all-ones sentinel.
__device__ __forceinline__ unsigned long long pack_md(float m, float d) {
    if (m != m) m = __uint_as_float(0x7fc00000u);
    if (d != d) d = __uint_as_float(0x7fc00000u);
    return (static_cast<unsigned long long>(__float_as_uint(d)) << 32) | __float_as_uint(m);
}

__device__ __forceinline__ MD unpack_md(unsigned long long v) {
    return MD{__uint_as_float(unsigned(v)), __uint_as_float(unsigned(v >> 32))};
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

struct PersistentArgs {
    int64_t M, N, ld;
    int nstages;                   // NS: stages of the ring
    int lookahead;                 // L: steps from a row's partial to its normalise (even, 2 <= L < NS)
    int stage_vecs;                // vectors of one stage (>= the widest CTA slice)
    unsigned* header;              // [0] status, [1] abort
    unsigned long long* rowstat;   // M row results (sentinel-filled)
    unsigned long long* partials;  // M * G * 16 warp partials (sentinel-filled)
    unsigned long long wait_ns;    // limit of every wait
    int64_t stall_row;             // test hook: CTA 0 withholds its partials of this row (-1: none)
};

// Bounded wait until *p is not the sentinel. Gives up (false) after
// `limit_ns`, recording the timeout and raising the abort word, or at once
// once another CTA raised it.
__device__ __forceinline__ bool wait_slot(const unsigned long long* p, unsigned* header, unsigned long long* out,
                                          unsigned long long limit_ns) {
    unsigned long long v = ld_relaxed_u64(p);
    if (v != kSlotEmpty) {
        *out = v;
        return true;
    }
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        v = ld_relaxed_u64(p);
        if (v != kSlotEmpty) {
            *out = v;
            return true;
        }
        if ((it & 31u) == 31u) {
            if (ld_acquire_u32(header + 1) != 0u) return false;
            if (global_ns() - t0 > limit_ns) {
                atomicExch(header + 0, kDeviceErrTimeout);
                atomicExch(header + 1, 1u);
                return false;
            }
        }
    }
    return false;
}

template <typename T>
__global__ void __launch_bounds__(kPersistBlock, 1) split_persistent_kernel(const T* x, T* y, PersistentArgs a) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int kLoc = kPersistMaxSlots / kPersistBlock;
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_m[kPersistWarps];
    __shared__ float red_d[kPersistWarps];
    __shared__ unsigned long long row_result[2];  // (m, d) of the rows being normalised, by parity
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    char* ring = smem + kRingHeader;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t nvec = a.N / V;
    const int NS = a.nstages, L = a.lookahead;
    const size_t stage_bytes = size_t(a.stage_vecs) * 16;
    // this CTA's slice of every row and this warp's part of it (in vectors)
    const int64_t s_lo = c * nvec / G, s_hi = (c + 1) * nvec / G;
    const int width = int(s_hi - s_lo);
    const int w_lo = width * warp / kPersistWarps, w_hi = width * (warp + 1) / kPersistWarps;
    const uint32_t bytes = uint32_t(width) * 16;
    const int64_t slots = G * kPersistWarps;
    int64_t issued = 0;   // rows 0 .. issued - 1 have been copied in or are on their way (thread 0)
    int64_t refill = -1;  // stage freed by the last normalise, refilled after the next barrier

    if (t == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(bar + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (t == 0)
        for (; issued < NS && issued < a.M; ++issued)
            tma_load_row(ring + issued * stage_bytes, x + issued * a.ld + s_lo * V, bytes, bar + issued);

    // error exit: thread 0 waits (bounded) for the copies of rows from..issued-1
    auto drain = [&](int64_t from) {
        if (t == 0)
            for (int64_t q = from; q < issued; ++q) mbar_wait(bar + (q % NS), uint32_t((q / NS) & 1), a.wait_ns);
    };

    unsigned long long next_stat = kSlotEmpty;  // thread 0: row result loaded one step early
    for (int64_t s = 0; s < a.M + L; ++s) {
        const int64_t q3 = s - L;  // row normalised in this step
        // ---- one barrier per step: row s has landed, row q3's (m, d) is known ----
        int fail = 0;
        if (s < a.M) fail = !mbar_wait(bar + int(s % NS), uint32_t((s / NS) & 1), a.wait_ns);
        if (t == 0 && q3 >= 0) {
            unsigned long long v = next_stat;
            if (v == kSlotEmpty && !wait_slot(a.rowstat + q3, a.header, &v, a.wait_ns)) fail = 1;
            row_result[q3 & 1] = v;
        }
        if (__syncthreads_or(fail)) {
            if (t == 0) {
                atomicExch(a.header + 0, kDeviceErrTimeout);
                atomicExch(a.header + 1, 1u);
            }
            drain(s < a.M ? s : a.M);
            return;
        }
        // every thread finished the last normalise: its stage may be refilled
        if (t == 0 && refill >= 0 && issued < a.M) {
            fence_proxy_async_smem();
            tma_load_row(ring + refill * stage_bytes, x + issued * a.ld + s_lo * V, bytes, bar + refill);
            ++issued;
        }
        refill = -1;
        // start loading the next step's row result now; its latency overlaps this step
        if (t == 0) next_stat = (q3 + 1 >= 0 && q3 + 1 < a.M) ? ld_relaxed_u64(a.rowstat + q3 + 1) : kSlotEmpty;

        // ---- partial of row s, one per warp ----
        if (s < a.M) {
            const char* sp = ring + int(s % NS) * stage_bytes;
            float m = -INFINITY, dv[V];
#pragma unroll
            for (int j = 0; j < V; ++j) dv[j] = 0.f;
            for (int v = w_lo + lane; v < w_hi; v += 32) {
                float f[V];
                E::unpack(lds16(sp + v * 16), f);
                float vm = f[0];
#pragma unroll
                for (int j = 1; j < V; ++j) vm = fmaxf(vm, f[j]);
                if (vm == -INFINITY) continue;  // all masked (m may still be -inf)
                if (vm > m) {
                    const float sc = ex2_approx((m - vm) * kLog2eF);
#pragma unroll
                    for (int j = 0; j < V; ++j) dv[j] *= sc;
                    m = vm;
                }
#pragma unroll
                for (int j = 0; j < V; ++j) dv[j] += exp_shifted(f[j], m);
            }
            float d = 0.f;
#pragma unroll
            for (int j = 0; j < V; ++j) d += dv[j];
            // warp merge: max, rescale, sum (fixed order)
            float wm = m;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
            d = d == 0.f ? 0.f : d * ex2_approx((m - wm) * kLog2eF);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0 && !(c == 0 && s == a.stall_row))
                st_relaxed_u64(a.partials + s * slots + c * kPersistWarps + warp, pack_md(wm, d));
        }

        // ---- merge of row s - L/2 by its owner ----
        const int64_t q2 = s - L / 2;
        if (q2 >= 0 && q2 < a.M && q2 % G == c) {
            // load this thread's slots t, t + BLOCK, ... all at once, then wait
            // (bounded) only for any still holding the sentinel
            unsigned long long raw[kLoc];
            const int n = int((slots - t + kPersistBlock - 1) / kPersistBlock);
#pragma unroll
            for (int k = 0; k < kLoc; ++k)
                raw[k] = k < n ? ld_relaxed_u64(a.partials + q2 * slots + t + k * kPersistBlock) : 0ull;
            MD loc[kLoc];
            int mfail = 0;
            float lm = -INFINITY;
#pragma unroll
            for (int k = 0; k < kLoc; ++k) {
                if (k >= n) break;
                if (raw[k] == kSlotEmpty && !wait_slot(a.partials + q2 * slots + t + k * kPersistBlock, a.header, &raw[k], a.wait_ns)) {
                    mfail = 1;
                    break;
                }
                loc[k] = unpack_md(raw[k]);
                if (loc[k].d != 0.f) lm = fmaxf(lm, loc[k].m);
            }
            if (__syncthreads_or(mfail)) {
                drain(s + 1);
                return;
            }
            const float Mx = group_reduce<kPersistBlock>(lm, red_m, OpMax());
            float d = 0.f;
#pragma unroll
            for (int k = 0; k < kLoc; ++k)
                if (k < n && loc[k].d != 0.f) d += loc[k].d * ex2_approx((loc[k].m - Mx) * kLog2eF);
            d = group_reduce<kPersistBlock>(d, red_d, OpSum());
            if (t == 0) st_relaxed_u64(a.rowstat + q2, pack_md(Mx, d));
        }

        // ---- normalise row q3; its stage is refilled after the next barrier ----
        if (q3 >= 0) {
            const MD md = unpack_md(row_result[q3 & 1]);
            const float m = md.d > 0.f ? md.m : 0.f;
            const float inv = safe_inverse(md.d);
            const int st = int(q3 % NS);
            const char* sp = ring + st * stage_bytes;
            T* yr = y + q3 * a.ld + s_lo * V;
            for (int v = t; v < width; v += kPersistBlock) {
                float f[V];
                E::unpack(lds16(sp + v * 16), f);
#pragma unroll
                for (int j = 0; j < V; ++j) f[j] = exp_shifted(f[j], m) * inv;
                st_stream16(yr + size_t(v) * V, E::pack(f));
            }
            refill = st;
        }
    }
}

// ---------------------------------------------------------------------------
// The same pipeline with L2 as the staging memory. Row slices are pulled into
// L2 `prefetch` steps ahead by bulk L2 prefetches (no shared memory, no
// registers held), the partial pass reads its slice from L2 with an
// evict-last policy, and the normalise pass re-reads it from L2 L steps later
// with an evict-first policy. HBM sees each x byte once while the on-chip
// window is the 129 MB L2 instead of the 225 KB of shared memory per SM.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_l2_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kPersistBlock, 1) split_l2_kernel(const T* x, T* y, PersistentArgs a, int prefetch) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int kLoc = kPersistMaxSlots / kPersistBlock;
    __shared__ float red_m[kPersistWarps];
    __shared__ float red_d[kPersistWarps];
    __shared__ unsigned long long row_result[2];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t nvec = a.N / V;
    const int L = a.lookahead;
    const int64_t s_lo = c * nvec / G, s_hi = (c + 1) * nvec / G;
    const int width = int(s_hi - s_lo);
    const int w_lo = width * warp / kPersistWarps, w_hi = width * (warp + 1) / kPersistWarps;
    const uint32_t bytes = uint32_t(width) * 16;
    const int64_t slots = G * kPersistWarps;
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    // this thread's vectors of the slice in the two passes
    constexpr int kMaxPer = 8;  // dispatcher: width <= 32 * kMaxPer per warp part, BLOCK * kMaxPer per slice

    if (t == 0)
        for (int64_t q = 0; q < prefetch && q < a.M; ++q) prefetch_l2_bulk(x + q * a.ld + s_lo * V, bytes);

    unsigned long long next_stat = kSlotEmpty;
    for (int64_t s = 0; s < a.M + L; ++s) {
        const int64_t q3 = s - L;
        // issue both passes' loads first: one L2 latency per step
        uint4 rp[kMaxPer], rn[kMaxPer];
        const T* xs = x + s * a.ld + s_lo * V;
        const T* xq = x + q3 * a.ld + s_lo * V;
        if (s < a.M) {
#pragma unroll
            for (int k = 0; k < kMaxPer; ++k) {
                const int v = w_lo + lane + 32 * k;
                if (v < w_hi) rp[k] = ld_l2_hint(xs + size_t(v) * V, keep);
            }
        }
        if (q3 >= 0) {
#pragma unroll
            for (int k = 0; k < kMaxPer; ++k) {
                const int v = t + kPersistBlock * k;
                if (v < width) rn[k] = ld_l2_hint(xq + size_t(v) * V, drop);
            }
        }
        int fail = 0;
        if (t == 0) {
            if (s + prefetch < a.M) prefetch_l2_bulk(x + (s + prefetch) * a.ld + s_lo * V, bytes);
            if (q3 >= 0) {
                unsigned long long v = next_stat;
                if (v == kSlotEmpty && !wait_slot(a.rowstat + q3, a.header, &v, a.wait_ns)) fail = 1;
                row_result[q3 & 1] = v;
            }
        }
        if (__syncthreads_or(fail)) return;
        if (t == 0) next_stat = (q3 + 1 >= 0 && q3 + 1 < a.M) ? ld_relaxed_u64(a.rowstat + q3 + 1) : kSlotEmpty;

        if (s < a.M) {
            float m = -INFINITY, dv[V];
#pragma unroll
            for (int j = 0; j < V; ++j) dv[j] = 0.f;
#pragma unroll
            for (int k = 0; k < kMaxPer; ++k) {
                const int v = w_lo + lane + 32 * k;
                if (v >= w_hi) break;
                float f[V];
                E::unpack(rp[k], f);
                float vm = f[0];
#pragma unroll
                for (int j = 1; j < V; ++j) vm = fmaxf(vm, f[j]);
                if (vm == -INFINITY) continue;
                if (vm > m) {
                    const float sc = ex2_approx((m - vm) * kLog2eF);
#pragma unroll
                    for (int j = 0; j < V; ++j) dv[j] *= sc;
                    m = vm;
                }
#pragma unroll
                for (int j = 0; j < V; ++j) dv[j] += exp_shifted(f[j], m);
            }
            float d = 0.f;
#pragma unroll
            for (int j = 0; j < V; ++j) d += dv[j];
            float wm = m;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
            d = d == 0.f ? 0.f : d * ex2_approx((m - wm) * kLog2eF);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0 && !(c == 0 && s == a.stall_row))
                st_relaxed_u64(a.partials + s * slots + c * kPersistWarps + warp, pack_md(wm, d));
        }

        const int64_t q2 = s - L / 2;
        if (q2 >= 0 && q2 < a.M && q2 % G == c) {
            unsigned long long raw[kLoc];
            const int n = int((slots - t + kPersistBlock - 1) / kPersistBlock);
#pragma unroll
            for (int k = 0; k < kLoc; ++k)
                raw[k] = k < n ? ld_relaxed_u64(a.partials + q2 * slots + t + k * kPersistBlock) : 0ull;
            MD loc[kLoc];
            int mfail = 0;
            float lm = -INFINITY;
#pragma unroll
            for (int k = 0; k < kLoc; ++k) {
                if (k >= n) break;
                if (raw[k] == kSlotEmpty && !wait_slot(a.partials + q2 * slots + t + k * kPersistBlock, a.header, &raw[k], a.wait_ns)) {
                    mfail = 1;
                    break;
                }
                loc[k] = unpack_md(raw[k]);
                if (loc[k].d != 0.f) lm = fmaxf(lm, loc[k].m);
            }
            if (__syncthreads_or(mfail)) return;
            const float Mx = group_reduce<kPersistBlock>(lm, red_m, OpMax());
            float d = 0.f;
#pragma unroll
            for (int k = 0; k < kLoc; ++k)
                if (k < n && loc[k].d != 0.f) d += loc[k].d * ex2_approx((loc[k].m - Mx) * kLog2eF);
            d = group_reduce<kPersistBlock>(d, red_d, OpSum());
            if (t == 0) st_relaxed_u64(a.rowstat + q2, pack_md(Mx, d));
        }

        if (q3 >= 0) {
            const MD md = unpack_md(row_result[q3 & 1]);
            const float m = md.d > 0.f ? md.m : 0.f;
            const float inv = safe_inverse(md.d);
            T* yr = y + q3 * a.ld + s_lo * V;
#pragma unroll
            for (int k = 0; k < kMaxPer; ++k) {
                const int v = t + kPersistBlock * k;
                if (v >= width) break;
                float f[V];
                E::unpack(rn[k], f);
#pragma unroll
                for (int j = 0; j < V; ++j) f[j] = exp_shifted(f[j], m) * inv;
                st_stream16(yr + size_t(v) * V, E::pack(f));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Row groups: the single-read form with each row spread over n CTAs instead
// of all of them. The grid is R row groups of n CTAs (gridDim.x = R * n); CTA
// c = g * n + q holds column slice q, [q nvec / n, (q + 1) nvec / n) vectors,
// of rows g, g + R, g + 2R, ... in turn, so the n CTAs of a group always work
// on the same row and a wave of the grid covers R whole rows. A CTA's ring
// holds nbuf slices in shared memory (bulk copies, one mbarrier each); step j
// of a CTA:
//   1. every thread moves its vectors of slice j from the ring into registers
//      (the buffer then takes slice j + nbuf at once); each warp takes the
//      maximum of its entries, then the sum of exp(x - max) relative to it;
//      after the step's one CTA barrier warp 1 merges the warp partials into
//      the slice's (m_q, d_q) and stores it in the row's slot q;
//   2. meanwhile the row of slice j - L is merged from its n slots, loaded in
//      the last step (waiting, bounded, only for any still empty), by
//      U = ceil(n / 32) warps at one slot per lane: the highest-numbered warp
//      takes slots 0..31, the next 32..63, and so on; each forms its chunk's
//      m_u = max m_q over d_q > 0 and d_u = sum d_q exp(m_q - m_u) and leaves
//      it in shared memory for the barrier;
//   3. after the barrier every thread combines the U chunk states in chunk
//      order (m = max m_u over d_u > 0, d = sum d_u exp(m_u - m)), so every
//      CTA of the group gets the same (m, d), and writes y = exp(x - m) / d
//      for slice j - L from its registers.
// Spreading step 2 over U warps keeps it off the barrier's critical path: one
// warp merging all n slots (three per lane at n = 76) held every other warp
// at the barrier for ~0.4 us per step (64 x 2^20 fp32: 99.0 -> 91.0 us; 512 x
// 2^19 fp32: 351 -> 321 us, the measured copy bandwidth).
// Step 2 waits only on the other CTAs of the group finishing step 1 of a row
// L steps earlier, which never waits on anything but their own copies and
// earlier steps: with all CTAs resident (a cooperative launch) every wait
// ends, and the lag L lets the slots' round trip through L2 overlap the next
// slices' work.
// Slots are self-flagging 64-bit words over a zero sentinel (a stored pair is
// never zero: a finite m comes with d >= 1, the maximal entry's own term, and
// an all -inf slice stores (-inf, 0)). Nothing needs to be zeroed before the
// launch: each CTA first zeroes its own slots (the ones it will fill) and CTA
// 0 the header's status and abort words, then the grid meets once at the
// cooperative launch's grid barrier, arrived at before the first copies are
// issued and waited for (bounded, by thread 0) before the first slot access,
// so its latency hides under the first slices' loads. A previous call's
// leftovers in the workspace, of any shape, are therefore never mistaken for
// this call's partials.
// Workspace: [0, 256) header (word 0 status, word 1 abort), then M * n slots.
// ---------------------------------------------------------------------------
constexpr int kGroupedLag = 2;  // steps from a slice's partial to its normalise

struct GroupedArgs {
    int64_t M, N, ld;
    int n;                         // CTAs per row group (gridDim.x is a multiple)
    int nbuf;                      // ring buffers per CTA
    int slot_vecs;                 // 16-byte vectors per buffer (>= the widest slice, multiple of 8)
    unsigned* header;              // [0] status, [1] abort
    unsigned long long* partials;  // M * n slice partials
    unsigned long long wait_ns;    // limit of every wait
    int64_t stall_row;             // test hook: the slice-0 CTA withholds its partial of this row (-1: none)
};

// Bounded wait until *p is nonzero (the zero-sentinel form of wait_slot).
__device__ __forceinline__ bool wait_filled(const unsigned long long* p, unsigned* header, unsigned long long* out,
                                            unsigned long long limit_ns) {
    unsigned long long v = ld_relaxed_u64(p);
    if (v != 0ull) {
        *out = v;
        return true;
    }
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        v = ld_relaxed_u64(p);
        if (v != 0ull) {
            *out = v;
            return true;
        }
        if ((it & 31u) == 31u) {
            if (ld_acquire_u32(header + 1) != 0u) return false;
            if (global_ns() - t0 > limit_ns) {
                atomicExch(header + 0, kDeviceErrTimeout);
                atomicExch(header + 1, 1u);
                return false;
            }
        }
    }
    return false;
}

// Thread 0 of a CTA, after the CTA arrived at the cooperative launch's grid
// barrier with `token`: bounded wait until every CTA has arrived (the
// barrier's top bit flips once all arrivals are in).
__device__ __forceinline__ bool grid_barrier_wait(const unsigned* bar, unsigned token, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if ((ld_acquire_u32(bar) ^ token) & 0x80000000u) return true;
        if ((it & 63u) == 63u && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Warp-wide max and sum by xor butterflies: every lane ends with the same bits
// (each step combines the same two values in either order).
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Merge of the partial states (m_i, d_i) that the lanes of a warp hold, one
// per lane: m = max m_i over d_i != 0, d = sum d_i exp(m_i - m). Every lane
// gets the result.
__device__ __forceinline__ MD warp_merge_states(MD p) {
    const float m = warp_max(p.d != 0.f ? p.m : -INFINITY);
    return MD{m, warp_sum(p.d != 0.f ? p.d * ex2_approx((p.m - m) * kLog2eF) : 0.f)};
}

// Each slice moves from its ring buffer into registers (a thread's vectors
// t, t + BLOCK, ...: at most MAXV of them) as soon as it has landed, and the
// buffer takes the slice nbuf steps ahead at once. A thread therefore holds
// L + 1 slices in registers: the one of the current step and the L waiting
// for their rows' merge. The step loop is unrolled L + 1 times so that every
// register array keeps a fixed role.
template <typename T, int BLOCK, int MAXV, int L>
__global__ void __launch_bounds__(BLOCK, 512 / BLOCK) split_grouped_kernel(const T* x, T* y, GroupedArgs a) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    constexpr int W = BLOCK / 32;
    constexpr int kChunks = (kGroupedMaxSlots + 31) / 32;  // slot chunks of 32, at most
    static_assert(BLOCK % 64 == 0 && BLOCK <= 1024 && L >= 2, "two warps or more; a lag of two steps or more");
    static_assert(kChunks <= W - 2, "the chunk-merging warps must leave warps 0 and 1 free");
    extern __shared__ __align__(128) char smem[];
    __shared__ MD warp_md[2][W];          // warp partials of a slice, by step parity
    __shared__ MD row_part[2][kChunks];   // chunk states of the row being normalised, by step parity
    const RowRing ring{reinterpret_cast<uint64_t*>(smem), smem + kRingHeader, uint32_t(a.slot_vecs) * 16u, a.nbuf};
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int n = a.n;
    const int U = (n + 31) / 32;             // chunks of the row's slots
    const int chunk = W - 1 - warp;          // this warp merges chunk `chunk` when 0 <= chunk < U
    const bool merger = chunk < U;           // (chunk >= 0 always: warp < W)
    const int my_slot = 32 * chunk + lane;   // this lane's slot when merger (none when >= n)
    const int q = int(blockIdx.x % unsigned(n));
    const int64_t R = gridDim.x / unsigned(n), r0 = blockIdx.x / unsigned(n);
    const int64_t nvec = a.N / V;
    const int64_t lo = q * nvec / n;
    const int width = int((q + 1) * nvec / n - lo);
    const uint32_t bytes = uint32_t(width) * 16u;
    const int64_t iters = a.M > r0 ? (a.M - r0 + R - 1) / R : 0;
    int64_t issued = 0;  // thread 0: slices 0 .. issued - 1 have been copied in or are on their way
    auto issue = [&](int64_t item) {  // thread 0: copy slice `item` into its buffer
        tma_load_row(ring.slot(int(item % ring.nbuf)), x + (r0 + item * R) * a.ld + lo * V, bytes,
                     ring.bar + int(item % ring.nbuf));
        issued = item + 1;
    };

    // the grid barrier of the cooperative launch (its memory is the driver's)
    const cooperative_groups::grid_group grid = cooperative_groups::this_grid();
    if (!grid.is_valid()) {  // not a cooperative launch: nothing here may run
        if (blockIdx.x == 0 && t == 0) atomicExch(a.header + 0, 1u);
        return;
    }
    // this call's own slots start empty, the status and abort words at zero
    if (blockIdx.x == 0 && t < 2) a.header[t] = 0u;
    for (int64_t i = t; i < iters; i += BLOCK) a.partials[(r0 + i * R) * n + q] = 0ull;
    if (t == 0) {
        for (int s = 0; s < ring.nbuf; ++s) mbar_init(ring.bar + s, 1);
        mbar_init_fence();
    }
    const unsigned token = grid.barrier_arrive();  // (a CTA barrier first, then thread 0 arrives)
    int fail0 = 0;
    if (t == 0) {
        for (int64_t s = 0; s < ring.nbuf && s < iters; ++s) issue(s);
        if (!grid_barrier_wait(&cooperative_groups::details::get_grid_workspace()->barrier, token, a.wait_ns)) {
            atomicExch(a.header + 0, kDeviceErrTimeout);
            atomicExch(a.header + 1, 1u);
            fail0 = 1;
        }
    }

    // merging warps: this lane's slot of the next row to merge, loaded one step early
    unsigned long long slot = 0ull;
    auto load_slot = [&](int64_t k) {
        if (merger && k >= 0 && k < iters)
            slot = my_slot < n ? ld_relaxed_u64(a.partials + (r0 + k * R) * n + my_slot) : 0ull;
    };

    // Step j: the merging warps fold their chunks of the row of slice k = j - L
    // (waiting, bounded, only for slots that were still empty) while every
    // warp takes slice j from its buffer into registers (`cur`) and folds its
    // part of the slice's partial; one barrier; the buffer takes slice
    // j + nbuf, warp 1 merges the warp partials and stores the slice's slot,
    // and every thread combines the chunk states and normalises slice k
    // (`old`). Returns false on an error exit.
    auto step = [&](int64_t j, uint4 (&cur)[MAXV], const uint4 (&old)[MAXV]) -> bool {
        const int64_t k = j - L;
        int fail = j == 0 ? fail0 : 0;
        if (merger && k >= 0) {
            const int64_t r = r0 + k * R;
            if (my_slot < n && slot == 0ull && !wait_filled(a.partials + r * n + my_slot, a.header, &slot, a.wait_ns))
                fail = 1;
            // (a lane past n holds (-inf, 0), which the merge skips)
            const MD c = warp_merge_states(my_slot < n ? unpack_md(slot) : MD{-INFINITY, 0.f});
            if (lane == 0) row_part[k & 1][chunk] = c;
        }
        if (j < iters) {
            const char* sb = ring.slot(int(j % ring.nbuf));
            if (!mbar_wait(ring.bar + int(j % ring.nbuf), uint32_t((j / ring.nbuf) & 1), a.wait_ns)) {
                if (t == 0) {
                    atomicExch(a.header + 0, kDeviceErrTimeout);
                    atomicExch(a.header + 1, 1u);
                }
                fail = 1;
            }
#pragma unroll
            for (int u = 0; u < MAXV; ++u)
                if (t + u * BLOCK < width) cur[u] = lds16(sb + size_t(t + u * BLOCK) * 16);
            // the warp's (max, sum exp(x - max)) over its vectors: the max
            // first (NaN-propagating), then the sum relative to it
            float m = -INFINITY, d = 0.f;
#pragma unroll
            for (int u = 0; u < MAXV; ++u)
                if (t + u * BLOCK < width) {
                    float f[V];
                    E::unpack(cur[u], f);
#pragma unroll
                    for (int e = 0; e < V; ++e) m = fmax_nan(m, f[e]);
                }
            m = warp_max_nan(m);
            if (m != -INFINITY) {
#pragma unroll
                for (int u = 0; u < MAXV; ++u)
                    if (t + u * BLOCK < width) {
                        float f[V];
                        E::unpack(cur[u], f);
#pragma unroll
                        for (int e = 0; e < V; ++e) d += exp_shifted(f[e], m);
                    }
            }
            d = warp_sum(d);
            if (lane == 0) warp_md[j & 1][warp] = MD{m, d};
        }
        if (group_bar_or(1, BLOCK, fail)) return false;
        if (j < iters) {
            // every thread has slice j in registers: its buffer takes slice j + nbuf
            if (t == 0 && j + ring.nbuf < iters) {
                fence_proxy_async_smem();
                issue(j + ring.nbuf);
            }
            if (warp == 1) {
                const MD c = warp_merge_states(lane < W ? warp_md[j & 1][lane] : MD{-INFINITY, 0.f});
                const int64_t r = r0 + j * R;
                if (lane == 0 && !(q == 0 && r == a.stall_row)) st_relaxed_u64(a.partials + r * n + q, pack_md(c.m, c.d));
            }
        }
        load_slot(k + 1);
        if (k < 0) return true;
        // the row's (m, d) from the chunk states, in chunk order
        float rm = -INFINITY;
        for (int u = 0; u < U; ++u) {
            const MD p = row_part[k & 1][u];
            if (p.d != 0.f) rm = fmaxf(rm, p.m);
        }
        float rd = 0.f;
        for (int u = 0; u < U; ++u) {
            const MD p = row_part[k & 1][u];
            if (p.d != 0.f) rd += p.d * ex2_approx((p.m - rm) * kLog2eF);
        }
        const float mm = rd > 0.f ? rm : 0.f;
        const float inv = safe_inverse(rd);
        T* yr = y + (r0 + k * R) * a.ld + lo * V;
#pragma unroll
        for (int u = 0; u < MAXV; ++u)
            if (t + u * BLOCK < width) {
                float f[V];
                E::unpack(old[u], f);
#pragma unroll
                for (int e = 0; e < V; ++e) f[e] = exp_shifted(f[e], mm) * inv;
                st_stream16(yr + size_t(t + u * BLOCK) * V, E::pack(f));
            }
        return true;
    };

    uint4 xs[L + 1][MAXV];
    int64_t j = 0;
    bool ok = true;
    while (ok && j < iters + L) {
        // j is a multiple of L + 1 here: step j + i fills xs[i] and normalises
        // xs[(i + 1) % (L + 1)], which holds slice j + i - L
#pragma unroll
        for (int i = 0; i <= L; ++i) {
            if (j >= iters + L) break;
            ok = step(j, xs[i], xs[(i + 1) % (L + 1)]);
            if (!ok) break;
            ++j;
        }
    }
    // error exit: thread 0 waits (bounded) for the copies in flight, slices j .. issued - 1
    if (!ok && t == 0)
        for (int64_t it = j < issued ? j : issued; it < issued; ++it)
            mbar_wait(ring.bar + int(it % ring.nbuf), uint32_t((it / ring.nbuf) & 1), a.wait_ns);
}

}  // namespace rowops
