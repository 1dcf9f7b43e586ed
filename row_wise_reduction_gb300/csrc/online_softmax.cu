// Split-row online softmax: launch wrappers for both element types.
#include "online_softmax_kernels.cuh"
#include "online_softmax_persistent.cuh"
#include "online_softmax_tma.cuh"
#include "rowops_launch.h"

namespace rowops {

constexpr int kSplitBlock = 256;
constexpr int kSplitUnroll = 8;

int64_t split_step_cols(int elem_bytes) { return int64_t(kSplitBlock) * kSplitUnroll * (16 / elem_bytes); }

template <typename T>
static cudaError_t launch_split(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                                int64_t nchunks, void* workspace, const LaunchCfg& cfg) {
    unsigned* status = static_cast<unsigned*>(workspace);
    float2* partials = reinterpret_cast<float2*>(static_cast<char*>(workspace) + kWorkspaceHeader);
    const int64_t items = M * nchunks;
    const bool scalar = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) != 0;
    auto k1 = split_partial_kernel<T, kSplitBlock, kSplitUnroll>;
    auto k2 = split_normalise_kernel<T, kSplitBlock, kSplitUnroll>;
    const int g1 = grid_for(reinterpret_cast<const void*>(k1), kSplitBlock, 0, items, cfg);
    k1<<<g1, kSplitBlock, 0, cfg.stream>>>(static_cast<const T*>(x), M, N, ld, chunk, nchunks, scalar,
                                           status, partials);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int g2 = grid_for(reinterpret_cast<const void*>(k2), kSplitBlock, 0, items, cfg);
    k2<<<g2, kSplitBlock, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, N, ld, chunk,
                                           nchunks, scalar, partials);
    return cudaGetLastError();
}

SplitLaunch split_softmax_f32() { return launch_split<float>; }
SplitLaunch split_softmax_bf16() { return launch_split<bf16_t>; }

constexpr int kSplitTmaTpr = 256;

template <typename T, int VPT>
static cudaError_t launch_split_tma_v(const void* x, void* y, int64_t M, int64_t nchunks, int64_t ld, int nbuf,
                                     void* workspace, const LaunchCfg& cfg) {
    unsigned* status = static_cast<unsigned*>(workspace);
    float2* partials = reinterpret_cast<float2*>(static_cast<char*>(workspace) + kWorkspaceHeader);
    const int64_t items = M * nchunks;
    const size_t smem = kRingHeader + size_t(nbuf) * kSplitTmaTpr * VPT * 16;
    auto k1 = split_partial_tma_kernel<T, kSplitTmaTpr, VPT>;
    auto k2 = split_normalise_tma_kernel<T, kSplitTmaTpr, VPT>;
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(k1), smem, cfg);
    if (e == cudaSuccess) e = allow_smem(reinterpret_cast<const void*>(k2), smem, cfg);
    if (e != cudaSuccess) return e;
    const int g1 = grid_for(reinterpret_cast<const void*>(k1), kSplitTmaTpr, smem, items, cfg);
    k1<<<g1, kSplitTmaTpr, smem, cfg.stream>>>(static_cast<const T*>(x), items, nchunks, ld, status, partials, nbuf,
                                               cfg.wait_ns, cfg.stall_row);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // pass 2 as a programmatic dependent of pass 1 (it fills its ring while
    // pass 1 drains, and waits for pass 1 before its first partial)
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(unsigned(grid_for(reinterpret_cast<const void*>(k2), kSplitTmaTpr, smem, items, cfg)));
    lc.blockDim = dim3(kSplitTmaTpr);
    lc.dynamicSmemBytes = smem;
    lc.stream = cfg.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, k2, static_cast<const T*>(x), static_cast<T*>(y), items, nchunks, ld,
                              const_cast<const float2*>(partials), status, nbuf, cfg.wait_ns, cfg.stall_row);
}

template <typename T>
static cudaError_t launch_split_tma(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t chunk,
                                   int64_t nchunks, int nbuf, void* workspace, const LaunchCfg& cfg) {
    constexpr int64_t step = int64_t(kSplitTmaTpr) * Elem<T>::kVec;
    if (chunk % step != 0 || N % chunk != 0 || nbuf < 2 || nbuf > kMaxRingBuffers) return cudaErrorNotSupported;
    const size_t smem = kRingHeader + size_t(nbuf) * size_t(chunk) * sizeof(T);
    if (smem + 1024 > size_t(cfg.max_smem_optin)) return cudaErrorNotSupported;
    switch (chunk / step) {
        case 1: return launch_split_tma_v<T, 1>(x, y, M, nchunks, ld, nbuf, workspace, cfg);
        case 2: return launch_split_tma_v<T, 2>(x, y, M, nchunks, ld, nbuf, workspace, cfg);
        case 4: return launch_split_tma_v<T, 4>(x, y, M, nchunks, ld, nbuf, workspace, cfg);
        case 8: return launch_split_tma_v<T, 8>(x, y, M, nchunks, ld, nbuf, workspace, cfg);
        default: return cudaErrorNotSupported;
    }
}

SplitTmaLaunch split_softmax_tma_f32() { return launch_split_tma<float>; }
SplitTmaLaunch split_softmax_tma_bf16() { return launch_split_tma<bf16_t>; }

int64_t persistent_slots(int64_t N) { return (N + 255) / 256 + 2; }
size_t persistent_rowstat_bytes(int64_t M) { return size_t((M * 8 + 255) / 256 * 256); }

// The single-read form, when it applies: rows 16-byte aligned with a length
// that is a multiple of 16 bytes; every warp's part of a CTA slice at least 32
// vectors; at least 4 stages of one slice each in shared memory; G * 16 warp
// partials per row within the workspace's slots; a cooperative launch on the
// device. Returns cudaErrorNotSupported (and launches nothing) otherwise.
template <typename T>
static cudaError_t launch_persistent(const void* x, void* y, int64_t M, int64_t N, int64_t ld, void* workspace,
                                     const LaunchCfg& cfg) {
    constexpr int V = Elem<T>::kVec;
    if (!cfg.cooperative || N % V != 0) return cudaErrorNotSupported;
    const int64_t nvec = N / V;
    const int64_t G = cfg.num_sms;
    const int64_t slots = G * kPersistWarps;
    if (slots > kPersistMaxSlots || slots > persistent_slots(N)) return cudaErrorNotSupported;
    if (nvec / G < int64_t(kPersistWarps) * 32) return cudaErrorNotSupported;
    const int64_t stage_vecs = ((nvec + G - 1) / G + 7) / 8 * 8;  // widest slice, 128-byte multiple
    const int64_t avail = int64_t(cfg.max_smem_optin) - int64_t(kRingHeader) - 1024;
    int64_t ns = avail / (stage_vecs * 16);
    if (ns > kMaxRingBuffers) ns = kMaxRingBuffers;
    if (ns < 4) return cudaErrorNotSupported;
    // lookahead: 4 steps when the ring has room for two copies ahead, else 2
    int lookahead = ns >= 7 ? 4 : 2;
    if (cfg.persist_lookahead >= 2 && cfg.persist_lookahead % 2 == 0 && cfg.persist_lookahead + 2 <= ns)
        lookahead = cfg.persist_lookahead;
    if (cfg.persist_l2) {
        // L2-staged form: no shared-memory ring; each thread holds at most
        // 8 vectors of a pass in registers
        if ((stage_vecs + kPersistBlock * 8 - 1) / (kPersistBlock * 8) > 1 || stage_vecs / kPersistWarps + 1 > 32 * 8)
            return cudaErrorNotSupported;
        const int la = cfg.persist_lookahead >= 2 && cfg.persist_lookahead % 2 == 0 ? cfg.persist_lookahead : 4;
        const int pf = cfg.persist_prefetch > 0 ? cfg.persist_prefetch : 6;
        char* ws = static_cast<char*>(workspace);
        PersistentArgs a;
        a.M = M;
        a.N = N;
        a.ld = ld;
        a.nstages = 0;
        a.lookahead = la;
        a.stage_vecs = int(stage_vecs);
        a.wait_ns = cfg.wait_ns;
        a.stall_row = cfg.stall_row;
        a.header = reinterpret_cast<unsigned*>(ws);
        a.rowstat = reinterpret_cast<unsigned long long*>(ws + kWorkspaceHeader);
        a.partials = reinterpret_cast<unsigned long long*>(ws + kWorkspaceHeader + persistent_rowstat_bytes(M));
        cudaError_t e = cudaMemsetAsync(ws, 0, kWorkspaceHeader, cfg.stream);
        if (e == cudaSuccess)
            e = cudaMemsetAsync(a.rowstat, 0xff, persistent_rowstat_bytes(M) + size_t(M) * size_t(slots) * 8,
                                cfg.stream);
        if (e != cudaSuccess) return e;
        const T* xp = static_cast<const T*>(x);
        T* yp = static_cast<T*>(y);
        int pfv = pf;
        void* args[] = {&xp, &yp, &a, &pfv};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(split_l2_kernel<T>), dim3(unsigned(G)),
                                           dim3(kPersistBlock), args, 0, cfg.stream);
    }
    auto kern = split_persistent_kernel<T>;
    const size_t smem = kRingHeader + size_t(ns) * size_t(stage_vecs) * 16;
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kPersistBlock, smem) != cudaSuccess || occ < 1) {
        cudaGetLastError();
        return cudaErrorNotSupported;
    }

    char* ws = static_cast<char*>(workspace);
    PersistentArgs a;
    a.M = M;
    a.N = N;
    a.ld = ld;
    a.nstages = int(ns);
    a.lookahead = lookahead;
    a.stage_vecs = int(stage_vecs);
    a.wait_ns = cfg.wait_ns;
    a.stall_row = cfg.stall_row;
    a.header = reinterpret_cast<unsigned*>(ws);
    a.rowstat = reinterpret_cast<unsigned long long*>(ws + kWorkspaceHeader);
    a.partials = reinterpret_cast<unsigned long long*>(ws + kWorkspaceHeader + persistent_rowstat_bytes(M));
    e = cudaMemsetAsync(ws, 0, kWorkspaceHeader, cfg.stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(a.rowstat, 0xff, persistent_rowstat_bytes(M) + size_t(M) * size_t(slots) * 8, cfg.stream);
    if (e != cudaSuccess) return e;
    const T* xp = static_cast<const T*>(x);
    T* yp = static_cast<T*>(y);
    void* args[] = {&xp, &yp, &a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(unsigned(G)), dim3(kPersistBlock),
                                       args, smem, cfg.stream);
}

PersistLaunch split_persistent_f32() { return launch_persistent<float>; }
PersistLaunch split_persistent_bf16() { return launch_persistent<bf16_t>; }

// The row-group form (split_grouped_kernel) with BLOCK threads per CTA and
// 512 / BLOCK CTAs per SM, when it applies: rows 16-byte aligned with a
// length that is a multiple of 16 bytes, a cooperative launch on the device,
// and a plan (grouped_plan.h) for a CTA's share of shared memory. Returns
// cudaErrorNotSupported (and launches nothing) otherwise.
template <typename T, int BLOCK>
static cudaError_t launch_grouped_block(const void* x, void* y, int64_t M, int64_t N, int64_t ld, void* workspace,
                                        int min_buffers, const LaunchCfg& cfg) {
    constexpr int V = Elem<T>::kVec;
    constexpr int kPerSm = 512 / BLOCK;
    if (!cfg.cooperative || N % V != 0 || M < 1) return cudaErrorNotSupported;
    // a CTA's share of the SM's shared memory (1 KB per CTA is the system's),
    // minus the barriers and this kernel's static arrays
    const int64_t avail = (int64_t(cfg.max_smem_optin) + 1024) / kPerSm - 1024 - int64_t(kRingHeader) - 512;
    const GroupedLimits lim{BLOCK, kPerSm, kGroupedMaxVpt, kGroupedMaxSlots, kGroupedMaxBuffers, avail};
    const GroupedPlan plan = grouped_plan(M, N / V, cfg.num_sms, min_buffers, persistent_slots(N), lim);
    if (plan.n == 0) return cudaErrorNotSupported;
    const int n = plan.n;
    const int64_t slot_vecs = plan.slot_vecs, nbuf = plan.nbuf, G = plan.grid;

    auto kern = split_grouped_kernel<T, BLOCK, kGroupedMaxVpt, kGroupedLag>;
    const size_t smem = kRingHeader + size_t(nbuf) * size_t(slot_vecs) * 16;
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg, kPerSm > 1);
    if (e != cudaSuccess) return e;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, BLOCK, smem) != cudaSuccess || occ < kPerSm) {
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    char* ws = static_cast<char*>(workspace);
    GroupedArgs a;
    a.M = M;
    a.N = N;
    a.ld = ld;
    a.n = n;
    a.nbuf = int(nbuf);
    a.slot_vecs = int(slot_vecs);
    a.header = reinterpret_cast<unsigned*>(ws);
    a.partials = reinterpret_cast<unsigned long long*>(ws + kWorkspaceHeader);
    a.wait_ns = cfg.wait_ns;
    a.stall_row = cfg.stall_row;
    // no fill of the workspace: the kernel zeroes its own slots and the
    // header's status and abort words before the grid's first exchange
    const T* xp = static_cast<const T*>(x);
    T* yp = static_cast<T*>(y);
    void* args[] = {&xp, &yp, &a};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(unsigned(G)), dim3(BLOCK), args,
                                       smem, cfg.stream);
}

// One CTA of 512 threads per SM; two of 256 with ROWOPS_FORCE_TPR=256 where
// the shape allows (slower on GB300: 104.5 us against 101.2 for 64 x 2^20
// fp32).
template <typename T>
static cudaError_t launch_grouped(const void* x, void* y, int64_t M, int64_t N, int64_t ld, void* workspace,
                                  int min_buffers, const LaunchCfg& cfg) {
    if (cfg.grouped_block == 256) {
        const cudaError_t e = launch_grouped_block<T, 256>(x, y, M, N, ld, workspace, min_buffers, cfg);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch_grouped_block<T, 512>(x, y, M, N, ld, workspace, min_buffers, cfg);
}

GroupedLaunch split_grouped_f32() { return launch_grouped<float>; }
GroupedLaunch split_grouped_bf16() { return launch_grouped<bf16_t>; }

}  // namespace rowops
