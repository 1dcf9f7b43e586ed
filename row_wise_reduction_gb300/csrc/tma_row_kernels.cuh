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
// `streams`: rows of that many inputs share each ring slot; `min_row_bytes`:
// a floor on the slot size (a multiple of 128).
template <int TPR, int ROWS>
__device__ __forceinline__ GroupPipe make_group(char* smem, int64_t N, int es, int nbuf, int period = 1,
                                                int streams = 1, uint32_t min_row_bytes = 0) {
    const int g = threadIdx.x / TPR;
    const uint32_t rb = uint32_t(streams) * max(ring_row_bytes(N, es), min_row_bytes);
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
    p.bar_id = ROWS == 1 ? 1 : 1 + g;  // a constant id lets a one-group CTA reserve two barriers, not 16
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

// Causal mask of the causal softmax ["Triton Kernel 实现练习" §5.1: query m
// sees keys n <= m]: row r is query r mod period and keeps the columns
// c <= (r mod period) + offset; the masked columns are never read.
struct CausalMask {
    int64_t period, offset;
    // columns kept by a row whose index mod period is rm
    __device__ __forceinline__ int kept_at(int64_t rm, int N) const {
        const int64_t k = rm + offset + 1;
        return int(k < 0 ? 0 : (k > N ? int64_t(N) : k));
    }
    // (rm + step) mod period for rm, step in [0, period): no division per row
    __device__ __forceinline__ int64_t advance(int64_t rm, int64_t step) const {
        rm += step;
        return rm >= period ? rm - period : rm;
    }
};

// Test hook: the copy of row `stall_row` is expected to bring 16 bytes more than
// it does, so the wait on it runs out (-1: no such row).
__device__ __forceinline__ uint32_t stall_extra(int64_t row, int64_t stall_row) { return row == stall_row ? 16u : 0u; }

// Causal rows (full rows): copy the 16-byte vectors that hold the kept
// prefix; a row that keeps nothing completes its phase with a plain arrival
// (the test hook instead expects bytes that never come).
template <typename T>
__device__ __forceinline__ void issue_prefix(const GroupPipe& p, int s, int64_t row, const T* x, int64_t ld,
                                             int64_t stall_row, int kept) {
    const int kv = (kept + Elem<T>::kVec - 1) / Elem<T>::kVec;
    const uint32_t extra = stall_extra(row, stall_row);
    if (kv > 0) tma_load_row(p.ring.slot(s), x + row * ld, uint32_t(kv) * 16u, p.ring.bar + s, extra);
    else if (extra) mbar_expect_tx(p.ring.bar + s, extra);
    else mbar_arrive(p.ring.bar + s);
}

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
// `cm` (CAUSAL): the first nbuf rows copy only their kept prefixes.
template <typename T, bool FULL, int ROWS, bool CAUSAL = false>
__device__ __forceinline__ void start_pipes(char* smem, const GroupPipe& p, const T* x, int64_t M, int N, int64_t ld,
                                            int64_t stall_row, const CausalMask& cm = CausalMask{1, 0}) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROWS * p.ring.nbuf; ++s) mbar_init(reinterpret_cast<uint64_t*>(smem) + s, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (p.producer)
        for (int s = 0; s < p.ring.nbuf; ++s) {
            const int64_t row = p.first + s * p.stride;
            if (row >= M) continue;
            if constexpr (CAUSAL) issue_prefix<T>(p, s, row, x, ld, stall_row, cm.kept_at(row % cm.period, N));
            else issue_row<T, FULL>(p, s, row, x, N, ld, stall_row);
        }
}

// After the group's first reduction: refill buffer s with the row nbuf
// iterations ahead (every thread of the group has its data in registers).
// `next_kept` (CAUSAL): the kept columns of the row nbuf iterations ahead.
template <typename T, bool FULL, bool CAUSAL = false>
__device__ __forceinline__ void refill(const GroupPipe& p, int s, int64_t row, const T* x, int64_t M, int N,
                                       int64_t ld, int64_t stall_row, int next_kept = 0) {
    if (!p.producer) return;
    const int64_t nxt = row + int64_t(p.ring.nbuf) * p.stride;
    if (nxt < M) {
        fence_proxy_async_smem();
        if constexpr (CAUSAL) issue_prefix<T>(p, s, nxt, x, ld, stall_row, next_kept);
        else issue_row<T, FULL>(p, s, nxt, x, N, ld, stall_row);
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

// ---------------------------------------------------------------------------
// Dynamic row schedule (full rows). A static schedule gives every row group the
// same number of rows, and the kernel ends with its slowest SM: on GB300 the
// busiest SM is active ~6% longer than the average one. Instead the grid is one
// CTA per work unit of rows; the resident CTAs take the units
// of CTAs that have not started yet with cluster launch control (a CTA cancels
// a pending CTA and processes its unit), so fast SMs take more rows and
// nothing but the last unit waits. A unit holds `unit_rows` rows of each group.
// Used by the RMSNorm kernels (tma_rms_kernels.cuh): on GB300 it made them
// ~10% faster, while softmax and LayerNorm+GELU, which issue more
// instructions per row, ran 5-10% slower with it and keep the static schedule. Thread 0 keeps one steal request in flight,
// its 16-byte response double-buffered in shared memory (`full` completes when
// a response lands, `empty` when every group's producer has read it), and
// issues the next request only after a successful one. Each group's producer
// takes the rows of the units in order, writes the row of every ring slot next
// to the slot, and marks the end of the work by a plain arrival on the slot.
// ---------------------------------------------------------------------------
struct __align__(16) ClcShared {
    uint4 resp[2];
    uint64_t full[2];
    uint64_t empty[2];
    int64_t slot_row[kMaxRingBuffers];  // row of ring slot s of group g at g * nbuf + s; -1: end
};

// Producer-side state of the dynamic schedule (in each group's producer thread).
struct DynFeed {
    int64_t unit;  // work unit whose rows are being taken
    int c;         // next row of the unit, 0 .. rows
    int rows;      // rows of each group in a work unit
    int k;         // responses read: unit k came with response k - 1
    bool end, requester, pending;
};

__device__ __forceinline__ void clc_init(ClcShared& cs, int rows) {
    mbar_init(&cs.full[0], 1);
    mbar_init(&cs.full[1], 1);
    mbar_init(&cs.empty[0], unsigned(rows));
    mbar_init(&cs.empty[1], unsigned(rows));
}

// Request r: cancel a CTA that has not started; the response lands in entry r & 1.
__device__ __forceinline__ void clc_request(ClcShared& cs, int r) {
    fence_proxy_async_smem();  // the entry's last response was read through the generic proxy
    mbar_expect_tx(&cs.full[r & 1], 16u);
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
            smem_addr(&cs.resp[r & 1])),
        "r"(smem_addr(&cs.full[r & 1]))
        : "memory");
}

// true and the cancelled CTA's x index (its work unit), or false: no CTA was left.
__device__ __forceinline__ bool clc_taken(const uint4* resp, int64_t& unit) {
    uint32_t ok, cx = 0;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "+r"(cx)
        : "r"(smem_addr(resp))
        : "memory");
    unit = int64_t(cx);
    return ok != 0;
}

// The producer's next row (-1: no more work). `fail` is set if a wait on the
// schedule gave up; the caller then ends the group's work like a finished one.
template <int ROWS>
__device__ __forceinline__ int64_t dyn_next_row(DynFeed& f, ClcShared& cs, int g, int64_t M,
                                                unsigned long long wait_ns, int& fail) {
    for (;;) {
        if (f.end) return -1;
        if (f.c == f.rows) {
            const int r = f.k;  // response r carries unit r + 1
            if (!mbar_wait(&cs.full[r & 1], uint32_t((r >> 1) & 1), wait_ns)) {
                fail = 1;
                f.end = true;
                return -1;
            }
            int64_t unit;
            const bool taken = clc_taken(&cs.resp[r & 1], unit);
            mbar_arrive(&cs.empty[r & 1]);
            if (f.requester) f.pending = false;
            f.k = r + 1;
            if (!taken) {
                f.end = true;
                return -1;
            }
            if (f.requester) {
                // request r + 1 reuses the entry of response r - 1: every group must have read it
                if (r >= 1 && !mbar_wait(&cs.empty[(r + 1) & 1], uint32_t(((r - 1) >> 1) & 1), wait_ns)) {
                    fail = 1;
                    f.end = true;
                    return -1;
                }
                clc_request(cs, r + 1);
                f.pending = true;
            }
            f.unit = unit;
            f.c = 0;
        }
        const int64_t row = f.unit * (ROWS * f.rows) + int64_t(f.c) * ROWS + g;
        ++f.c;
        if (row < M) return row;
    }
}

// Producer: fill ring slot s with the next row of each of the S inputs (or the
// end mark). A schedule wait that gave up records the timeout and ends the work.
template <typename T, int ROWS, int S>
__device__ __forceinline__ void dyn_issue(const GroupPipe& p, ClcShared& cs, DynFeed& f, int g, int s,
                                          const T* const* src, int N, int64_t ld, int64_t M, int64_t stall_row,
                                          unsigned long long wait_ns, unsigned* err) {
    int fail = 0;
    const int64_t row = dyn_next_row<ROWS>(f, cs, g, M, wait_ns, fail);
    if (fail) atomicExch(err, kDeviceErrTimeout);
    cs.slot_row[g * p.ring.nbuf + s] = row;
    if (row >= 0) {
        const uint32_t bytes = uint32_t(N / Elem<T>::kVec) * 16u;  // full rows: the whole row
        const uint32_t stride = p.ring.row_bytes / S;
        fence_proxy_async_smem();  // the slot was last read through the generic proxy
        mbar_expect_tx(p.ring.bar + s, S * bytes + stall_extra(row, stall_row));
#pragma unroll
        for (int k = 0; k < S; ++k) tma_copy_row(p.ring.slot(s) + k * stride, src[k] + row * ld, bytes, p.ring.bar + s);
    } else {
        mbar_arrive(p.ring.bar + s);
    }
}

// CTA start of the dynamic schedule: barriers, the first steal request, and
// each group's first nbuf rows. A work unit holds `unit_rows` rows of each group.
template <typename T, int ROWS, int S>
__device__ __forceinline__ DynFeed dyn_start(char* smem, const GroupPipe& p, ClcShared& cs, int g,
                                             const T* const* src, int N, int64_t ld, int64_t M, int64_t stall_row,
                                             unsigned long long wait_ns, unsigned* err, int unit_rows) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < ROWS * p.ring.nbuf; ++s) mbar_init(reinterpret_cast<uint64_t*>(smem) + s, 1);
        clc_init(cs, ROWS);
        mbar_init_fence();
    }
    __syncthreads();
    DynFeed f{int64_t(blockIdx.x), 0, unit_rows, 0, false, threadIdx.x == 0, false};
    if (f.requester) {
        clc_request(cs, 0);
        f.pending = true;
    }
    if (p.producer)
        for (int s = 0; s < p.ring.nbuf; ++s) dyn_issue<T, ROWS, S>(p, cs, f, g, s, src, N, ld, M, stall_row, wait_ns, err);
    return f;
}

// Consumer side, iteration i (at cursor rc): wait for the slot and read its row; -1: the
// work has ended (every thread of the group sees it: an end mark completes its
// slot's phase when it is written). A wait that gave up sets `fail` and hands
// back the slot's row as written, so the thread goes on to the group's first
// reduction, whose barrier tells the whole group to stop.
__device__ __forceinline__ int64_t dyn_row(const GroupPipe& p, const ClcShared& cs, int g, const RingCursor& rc,
                                           unsigned long long wait_ns, int& fail) {
    const int s = rc.slot;
    fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
    const int64_t row = cs.slot_row[g * p.ring.nbuf + s];
    return fail && row < 0 ? 0 : row;
}

// End of a group's work: the steal requester waits (bounded) for a request it
// still has in flight, so that no response lands after the CTA is gone.
__device__ __forceinline__ void dyn_finish(const DynFeed& f, ClcShared& cs, unsigned long long wait_ns) {
    if (f.requester && f.pending) mbar_wait(&cs.full[f.k & 1], uint32_t((f.k >> 1) & 1), wait_ns);
}

// Error exit (a wait of iteration i gave up): the producer waits (bounded) for
// the copies of the slots it filled, then records the timeout.
__device__ __forceinline__ void dyn_abandon(const GroupPipe& p, const DynFeed& f, ClcShared& cs, int g, int64_t i,
                                            unsigned* err, unsigned long long wait_ns) {
    if (!p.producer) return;
    const int nbuf = p.ring.nbuf;
    for (int d = 0; d < nbuf; ++d) {
        const int64_t it = i + d;
        const int s = int(it % nbuf);
        if (cs.slot_row[g * nbuf + s] >= 0) mbar_wait(p.ring.bar + s, uint32_t((it / nbuf) & 1), wait_ns);
    }
    dyn_finish(f, cs, wait_ns);
    atomicExch(err, kDeviceErrTimeout);
}

// CAUSAL (full rows only): the causal softmax; row `row` keeps cm.kept(row, N)
// columns, only the 16-byte vectors holding them are copied, and the masked
// columns come out as exactly 0 (their exponentials of -inf).
template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool CAUSAL = false>
__global__ void __launch_bounds__(TPR * ROWS)
    softmax_tma_kernel(const T* x, T* y, int64_t M, int N, int64_t ld, int nbuf, unsigned* err,
                       unsigned long long wait_ns, int64_t stall_row, CausalMask cm) {
    using E = Elem<T>;
    constexpr int V = E::kVec;
    static_assert(TPR % 64 == 0, "row groups of at least two warps");
    static_assert(FULL || !CAUSAL, "the causal form runs on full rows");
    extern __shared__ __align__(128) char smem[];
    __shared__ float red_max[ROWS][TPR / 32];
    __shared__ float red_sum[ROWS][TPR / 32];
    const GroupPipe p = make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf);
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    start_pipes<T, FULL, ROWS, CAUSAL>(smem, p, x, M, N, ld, stall_row, cm);
    // causal: row mod period of iteration i, its step per iteration and per ring turn
    int64_t rm = CAUSAL ? p.first % cm.period : 0;
    const int64_t step = CAUSAL ? p.stride % cm.period : 0;
    const int64_t ring_step = CAUSAL ? (int64_t(nbuf) * step) % cm.period : 0;

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = rc.slot;
        const T* xr = x + row * ld;
        const RowSpan sp = row_span<T, FULL>(xr, N);
        // unaligned head / tail elements: plain loads, in flight during the wait
        const bool has_ex = !FULL && t < sp.head + sp.tail;
        const int ecol = has_ex ? span_extra_col(sp, t, V) : 0;
        float ex = has_ex ? E::load(xr + ecol) : -INFINITY;
        int fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
        const char* sb = p.ring.slot(s);
        const int kept = CAUSAL ? cm.kept_at(rm, N) : N;

        float v[VPT][V];
        float mx = ex;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = t + j * TPR;
            if (CAUSAL) {
                // vectors wholly past the kept prefix were not copied and take
                // no arithmetic (their outputs are stored as zeros below); only
                // the vector that straddles the boundary is masked per element
                if (k * V < kept) {
                    E::unpack(lds16(sb + size_t(k) * 16), v[j]);
                    if (k * V + V > kept) {
#pragma unroll
                        for (int e = 0; e < V; ++e)
                            if (k * V + e >= kept) v[j][e] = -INFINITY;
                    }
#pragma unroll
                    for (int e = 0; e < V; ++e) mx = fmaxf(mx, v[j][e]);
                }
                continue;
            } else if (FULL || k < sp.body) {
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
        refill<T, FULL, CAUSAL>(p, s, row, x, M, N, ld, stall_row, CAUSAL ? cm.kept_at(cm.advance(rm, ring_step), N) : 0);
        if (CAUSAL) rm = cm.advance(rm, step);
        if (mx == -INFINITY) mx = 0.f;
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (CAUSAL && (t + j * TPR) * V >= kept) continue;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] = exp_shifted(v[j][e], mx);
                sum += v[j][e];
            }
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
            if (CAUSAL && k * V >= kept) {
                st_stream16(yb + size_t(k) * V, make_uint4(0u, 0u, 0u, 0u));
            } else if (FULL || k < sp.body) {
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

// Ring slot of LayerNorm+GELU: general rows reserve the whole tile (TPR * VPT
// vectors) so that the vectors past the body can stay zero in every slot.
template <typename T, int TPR, int VPT, bool FULL>
__host__ __device__ constexpr uint32_t ln_slot_bytes(int64_t N) {
    return FULL ? ring_row_bytes(N, Elem<T>::kBytes)
                : (ring_row_bytes(N, Elem<T>::kBytes) > uint32_t(TPR * VPT * 16) ? ring_row_bytes(N, Elem<T>::kBytes)
                                                                                  : uint32_t(TPR * VPT * 16));
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool ERF = false>
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
    const GroupPipe p =
        make_group<TPR, ROWS>(smem, N, E::kBytes, nbuf, period, 1, ln_slot_bytes<T, TPR, VPT, FULL>(N));
    const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
    char* affine = smem + kRingHeader + size_t(ROWS) * nbuf * p.ring.row_bytes;
    float4* sw4 = reinterpret_cast<float4*>(affine);
    float4* sb4 = sw4 + VPT * H * TPR;
    float2* sxb = reinterpret_cast<float2*>(affine + tma_affine_bytes<T, TPR, VPT>());
    // General rows use 1/N once instead of three IEEE divisions per row and
    // thread (bf16 65536 x 4097: 200 -> 192 us together with the body
    // predicates below; the mean's rounding is taken up by the residual
    // correction either way). Full rows keep the divisions: measured side by
    // side they were as fast at 8192 columns and 1.5% faster at 4096.
    const float fN = float(N), inv_n = 1.f / fN;
    // the split shared by every row of this CTA's phase class
    const RowSpan sp = row_span<T, FULL>(x + int64_t(p.cls) * ld, N);
    // vectors j < jf lie inside the body for every thread of the group
    const int jf = FULL ? VPT : sp.body / TPR;
    start_pipes<T, FULL, ROWS>(smem, p, x, M, N, ld, stall_row);
    stage_affine_thread_major<T, TPR, VPT>(w, b, sp.head, sp.body, sw4, sb4);
    if constexpr (!FULL) {
        for (int e = threadIdx.x; e < sp.head + sp.tail; e += blockDim.x) {
            const int c = span_extra_col(sp, e, V);
            sxb[e] = make_float2(w ? E::load(w + c) : 1.f, b ? E::load(b + c) : 0.f);
        }
        // the vectors past the body read as zeros in every slot: the copies
        // (the body only) never write them, so the load pass needs no predicate
        for (int s = 0; s < nbuf; ++s)
            for (int k = sp.body + t; k < TPR * VPT; k += TPR)
                *reinterpret_cast<uint4*>(p.ring.slot(s) + size_t(k) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    const bool has_ex = !FULL && t < sp.head + sp.tail;
    const int ecol = has_ex ? span_extra_col(sp, t, V) : 0;

    RingCursor rc;
    for (int64_t i = 0;; ++i, rc.next(nbuf)) {
        const int64_t row = p.first + i * p.stride;
        if (row >= M) break;
        const int s = rc.slot;
        const T* xr = x + row * ld;
        float ex = has_ex ? E::load(xr + ecol) : 0.f;
        int fail = !mbar_wait(p.ring.bar + s, rc.parity, wait_ns);
        const char* sbuf = p.ring.slot(s);

        // elementwise arithmetic on packed fp32 pairs
        float2 v[VPT][V / 2];
        float2 s2 = make_float2(ex, 0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float u[V];
            E::unpack(lds16(sbuf + size_t(t + j * TPR) * 16), u);
#pragma unroll
            for (int e = 0; e < V / 2; ++e) {
                v[j][e] = make_float2(u[2 * e], u[2 * e + 1]);
                s2 = f2_add(s2, v[j][e]);
            }
        }
        float sum = row_reduce<TPR>(s2.x + s2.y, red_a[g], p.bar_id, OpSum(), fail);
        if (fail) {
            abandon(p, i, M, err, wait_ns);
            return;
        }
        refill<T, FULL>(p, s, row, x, M, N, ld, stall_row);
        const float mean = FULL ? sum / fN : sum * inv_n;
        // centred values, their squares and the residual of the fp32 mean
        // (vectors past the body stay 0; only j >= jf can hold such vectors)
        float2 q2 = f2(0.f), r2 = f2(0.f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (FULL || j < jf) {
#pragma unroll
                for (int e = 0; e < V / 2; ++e) {
                    v[j][e] = f2_add(v[j][e], f2(-mean));
                    q2 = f2_fma(v[j][e], v[j][e], q2);
                    r2 = f2_add(r2, v[j][e]);
                }
            } else {
                const bool ok = (t + j * TPR) < sp.body;
#pragma unroll
                for (int e = 0; e < V / 2; ++e) {
                    v[j][e] = ok ? f2_add(v[j][e], f2(-mean)) : f2(0.f);
                    q2 = f2_fma(v[j][e], v[j][e], q2);
                    r2 = f2_add(r2, v[j][e]);
                }
            }
        }
        float q = q2.x + q2.y, r = r2.x + r2.y;
        if constexpr (!FULL) {
            ex = has_ex ? ex - mean : 0.f;
            q = fmaf(ex, ex, q);
            r += ex;
        }
        row_reduce_sum2<TPR>(q, r, red_b[g], p.bar_id, fail);
        const float delta = FULL ? r / fN : r * inv_n;
        const float rstd = rsqrtf(fmaxf((FULL ? q / fN : q * inv_n) - delta * delta, 0.f) + eps);
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
                    const float4 ww = ERF ? ldsf4(sw4 + (j * H + h) * TPR + t) : sw4[(j * H + h) * TPR + t];
                    const float4 bb = ERF ? ldsf4(sb4 + (j * H + h) * TPR + t) : sb4[(j * H + h) * TPR + t];
                    const float2 z0 = f2_fma(f2_fma(v[j][2 * h], f2(rstd), f2(shift)), make_float2(ww.x, ww.y),
                                             make_float2(bb.x, bb.y));
                    const float2 z1 = f2_fma(f2_fma(v[j][2 * h + 1], f2(rstd), f2(shift)), make_float2(ww.z, ww.w),
                                             make_float2(bb.z, bb.w));
                    const float2 g0 = gelu_of2<ERF>(z0), g1 = gelu_of2<ERF>(z1);
                    o[4 * h + 0] = g0.x;
                    o[4 * h + 1] = g0.y;
                    o[4 * h + 2] = g1.x;
                    o[4 * h + 3] = g1.y;
                }
                st_stream16(yb + size_t(k) * V, E::pack(o));
            }
        }
        if (has_ex) {
            const float2 wb = sxb[t];
            E::store(yr + ecol, gelu_of<ERF>(fmaf(fmaf(ex, rstd, shift), wb.x, wb.y)));
        }
    }
}

}  // namespace rowops
