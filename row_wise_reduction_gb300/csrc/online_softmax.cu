// Split-row online softmax: launch wrappers for both element types.
#include "online_softmax_kernels.cuh"
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

}  // namespace rowops
