// LayerNorm+GELU on short rows stored back to back (ld == N <= 256): rows
// whose length is not a whole number of 16-byte vectors (e.g. bf16 rows of 127
// elements), rows of at most 128 columns, and large batches of such rows.
//
// Row-by-row kernels meet unaligned rows at a different offset modulo 16 bytes
// each time, so every row costs a head and a tail of scalar accesses and a
// per-row split, and on short rows their per-row costs (group reductions,
// waits) outweigh the arithmetic. Here the unit of memory traffic is a chunk
// of R consecutive rows instead: R is a multiple of 16 / gcd(16, N * es), so
// every chunk starts on a 16-byte boundary and all but the matrix's last chunk
// are whole 16-byte vectors. A chunk moves global -> shared with one bulk copy and back with one
// bulk store; in shared memory, teams of L lanes normalise its rows in place
// (lane l takes the columns l, l + L, ...: consecutive lanes, consecutive
// elements), with w, b held in registers for the whole kernel.
//
// The statistics and the output follow the other LayerNorm+GELU kernels
// ["PyTorch 自定义 CUDA 算子与 Triton 编程" §三 (fused LayerNorm+GELU)]: the
// mean, the variance of the centred row with the fp32 mean's residual taken
// out, rstd = 1/sqrt(var + eps), then GELU(w (x - mean) rstd + b).
#pragma once

#include "ln_gelu_kernels.cuh"
#include "row_pipeline.cuh"

namespace rowops {

constexpr int kFlatBlock = 256;
constexpr uint32_t kFlatChunkTarget = 16384;  // bytes of x per chunk (about)

// bulk store shared -> global of `bytes` (a multiple of 16, both ends 16-byte
// aligned), as one bulk group
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// wait until every bulk store issued by this thread has read its source
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// wait until every bulk store issued by this thread has completed its writes
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// two outputs of one lane, each stored if its flag is set (bf16: one
// conversion for both)
template <typename T>
struct FlatOut;
template <>
struct FlatOut<float> {
    __device__ __forceinline__ static void store2(float* p0, bool s0, float* p1, bool s1, float2 g) {
        if (s0) *p0 = g.x;
        if (s1) *p1 = g.y;
    }
};
template <>
struct FlatOut<bf16_t> {
    __device__ __forceinline__ static void store2(bf16_t* p0, bool s0, bf16_t* p1, bool s1, float2 g) {
        const uint32_t r = pack_bf16x2(g.x, g.y);
        if (s0) p0->bits = uint16_t(r & 0xffffu);
        if (s1) p1->bits = uint16_t(r >> 16);
    }
};

// rows per chunk: a multiple of 16 / gcd(16, row bytes), about
// kFlatChunkTarget bytes
__host__ __device__ constexpr int64_t flat_chunk_rows(int64_t N, int es) {
    const int64_t rb = N * es;
    const int64_t unit = (rb & 15) == 0 ? 1 : 16 / (rb & -rb & 15);
    const int64_t r = int64_t(kFlatChunkTarget) / rb / unit * unit;
    return r > unit ? r : unit;
}

// chunk c of a matrix of M rows: its rows and bytes
struct FlatChunk {
    int rows;
    uint32_t bytes, bulk;  // all bytes; the part the bulk copies move (a multiple of 16)
};

__device__ __forceinline__ FlatChunk flat_chunk(int64_t c, int64_t R, int64_t M, int N, int es) {
    const int64_t left = M - c * R;
    const int rows = int(left < R ? left : R);
    const uint32_t bytes = uint32_t(rows) * uint32_t(N) * uint32_t(es);
    return FlatChunk{rows, bytes, bytes & ~15u};
}

// L lanes per row, EPL columns per lane (N <= L * EPL); kFlatBlock threads,
// two chunk buffers. `R`: rows per chunk (flat_chunk_rows). The wait for a
// chunk is bounded: past `wait_ns` the CTA sets *err = ROWOPS_ERR_TIMEOUT,
// waits (bounded) for its copies in flight and returns. `stall_row` (test hook):
// the copy of the chunk holding that row expects 16 bytes that never come.
template <typename T, int L, int EPL, bool ERF>
__global__ void __launch_bounds__(kFlatBlock)
    ln_gelu_flat_kernel(const T* x, T* y, const T* w, const T* b, float eps, int64_t M, int N, int64_t R,
                        unsigned* err, unsigned long long wait_ns, int64_t stall_row) {
    using E = Elem<T>;
    constexpr int TEAMS = kFlatBlock / L;
    static_assert(L == 8 || L == 16 || L == 32, "teams inside one warp");
    extern __shared__ __align__(128) char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    const uint32_t buf_bytes = uint32_t(R) * uint32_t(N) * uint32_t(E::kBytes);  // a multiple of 16
    auto buf = [&](int64_t i) { return reinterpret_cast<T*>(smem + kRingHeader + (i & 1) * buf_bytes); };
    const int64_t nchunks = (M + R - 1) / R;
    const int lane = threadIdx.x % L, team = threadIdx.x / L;
    const bool leader = threadIdx.x == 0;

    // the copy of local chunk i (global chunk blockIdx.x + i * gridDim.x) into buffer i & 1
    auto issue = [&](int64_t i) {
        const int64_t c = blockIdx.x + i * gridDim.x;
        const FlatChunk ch = flat_chunk(c, R, M, N, E::kBytes);
        const bool stall = stall_row >= c * R && stall_row < c * R + ch.rows;
        const uint32_t extra = stall ? 16u : 0u;
        if (ch.bulk > 0) tma_load_row(buf(i), x + c * R * N, ch.bulk, bar + (i & 1), extra);
        else if (extra) mbar_expect_tx(bar + (i & 1), extra);
        else mbar_arrive(bar + (i & 1));
    };
    auto live = [&](int64_t i) { return blockIdx.x + i * int64_t(gridDim.x) < nchunks; };

    if (leader) {
        mbar_init(bar, 1);
        mbar_init(bar + 1, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (leader) {
        if (live(0)) issue(0);
        if (live(1)) issue(1);
    }

    // w, b of this lane's columns (pairs of its columns k, k + 1), for every
    // row; the lane's columns k < nv lie inside the row
    static_assert(EPL % 2 == 0, "columns in pairs");
    constexpr int P = EPL / 2;
    const int nv = lane < N ? (N - 1 - lane) / L + 1 : 0;
    float2 w2[P], b2[P];
#pragma unroll
    for (int m = 0; m < P; ++m) {
        const int c0 = lane + 2 * m * L, c1 = c0 + L;
        w2[m] = make_float2((w && 2 * m < nv) ? E::load(w + c0) : 1.f, (w && 2 * m + 1 < nv) ? E::load(w + c1) : 1.f);
        b2[m] = make_float2((b && 2 * m < nv) ? E::load(b + c0) : 0.f, (b && 2 * m + 1 < nv) ? E::load(b + c1) : 0.f);
    }
    // 1/N once: the mean's rounding is taken out by the residual either way
    const float inv_n = 1.f / float(N);
    const int per_team = int((R + TEAMS - 1) / TEAMS);  // rows per team and chunk (uniform)

    for (int64_t i = 0; live(i); ++i) {
        const int64_t c = blockIdx.x + i * gridDim.x;
        const FlatChunk ch = flat_chunk(c, R, M, N, E::kBytes);
        T* const cb = buf(i);
        const int64_t base = c * R * N;  // first element of the chunk
        int fail = !mbar_wait(bar + (i & 1), uint32_t((i >> 1) & 1), wait_ns);
        // the last chunk's final bytes (< 16) come with plain loads
        const int tail = int(ch.bytes - ch.bulk) / E::kBytes;
        const int t0 = int(ch.bulk) / E::kBytes;
        if (int(threadIdx.x) < tail) cb[t0 + threadIdx.x] = x[base + t0 + threadIdx.x];
        if (__syncthreads_or(fail)) {
            if (leader) {
                // every copy issued and not yet waited for: this chunk's and the next one's
                mbar_wait(bar + (i & 1), uint32_t((i >> 1) & 1), wait_ns);
                if (live(i + 1)) mbar_wait(bar + ((i + 1) & 1), uint32_t(((i + 1) >> 1) & 1), wait_ns);
                bulk_wait_all();
                atomicExch(err, kDeviceErrTimeout);
            }
            return;
        }

        for (int j = 0; j < per_team; ++j) {
            const int r = team + j * TEAMS;
            const int lim = r < ch.rows ? nv : 0;  // this lane's columns in this row
            T* row = cb + (lim ? r : 0) * N;
            float2 v[P];
            float2 s2 = f2(0.f);
#pragma unroll
            for (int m = 0; m < P; ++m) {
                v[m] = make_float2(2 * m < lim ? E::load(row + lane + 2 * m * L) : 0.f,
                                   2 * m + 1 < lim ? E::load(row + lane + (2 * m + 1) * L) : 0.f);
                s2 = f2_add(s2, v[m]);
            }
            float s = s2.x + s2.y;
#pragma unroll
            for (int o = L / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const float mean = s * inv_n;
            // variance of the centred values; the residual r of the fp32 mean
            // gives x - true mean = (x - mean) - r / N
            float2 q2 = f2(0.f), r2 = f2(0.f);
#pragma unroll
            for (int m = 0; m < P; ++m) {
                v[m] = f2_add(v[m], f2(-mean));
                if (2 * m >= lim) v[m].x = 0.f;
                if (2 * m + 1 >= lim) v[m].y = 0.f;
                q2 = f2_fma(v[m], v[m], q2);
                r2 = f2_add(r2, v[m]);
            }
            float q = q2.x + q2.y, rs = r2.x + r2.y;
#pragma unroll
            for (int o = L / 2; o > 0; o >>= 1) {
                q += __shfl_xor_sync(0xffffffffu, q, o);
                rs += __shfl_xor_sync(0xffffffffu, rs, o);
            }
            const float delta = rs * inv_n;
            const float rstd = rsqrtf(fmaxf(q * inv_n - delta * delta, 0.f) + eps);
            const float shift = -delta * rstd;
#pragma unroll
            for (int m = 0; m < P; ++m) {
                const float2 g = gelu_of2<ERF>(f2_fma(f2_fma(v[m], f2(rstd), f2(shift)), w2[m], b2[m]));
                FlatOut<T>::store2(row + lane + 2 * m * L, 2 * m < lim, row + lane + (2 * m + 1) * L, 2 * m + 1 < lim,
                                   g);
            }
        }

        fence_proxy_async_smem();  // this thread's outputs, before the bulk store reads them
        __syncthreads();
        if (leader && ch.bulk > 0) bulk_store(y + base, cb, ch.bulk);
        if (int(threadIdx.x) < tail) y[base + t0 + threadIdx.x] = cb[t0 + threadIdx.x];
        // refill this buffer with local chunk i + 2 once the store has read it
        // (a chunk with a tail is the matrix's last: nothing follows it)
        if (leader && live(i + 2)) {
            bulk_wait_read();
            issue(i + 2);
        }
    }
    if (leader) bulk_wait_all();
}

}  // namespace rowops
