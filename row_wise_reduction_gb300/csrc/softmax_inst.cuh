// Launch wrappers and dispatch tables of the softmax kernels for one element
// type. Included once per dtype by softmax_f32.cu / softmax_bf16.cu.
#pragma once

#include "rowops_launch.h"
#include "softmax_kernels.cuh"

namespace rowops {

template <int TPR>
constexpr int reg_block() {
    return TPR > 256 ? TPR : 256;
}

template <typename T, int TPR, int VPT>
cudaError_t launch_softmax_reg(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                               const LaunchCfg& cfg) {
    constexpr int BLOCK = reg_block<TPR>();
    constexpr int ROWS = BLOCK / TPR;
    auto kern = softmax_reg_kernel<T, TPR, VPT, BLOCK>;
    const int64_t groups = (M + ROWS - 1) / ROWS;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, 0, groups, cfg);
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, int(N),
                                         ld);
    return cudaGetLastError();
}

constexpr int kLoopedBlock = 512;
constexpr int kLoopedUnroll = 4;

template <typename T>
cudaError_t launch_softmax_looped(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                  const LaunchCfg& cfg) {
    auto kern = softmax_looped_kernel<T, kLoopedBlock, kLoopedUnroll>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kLoopedBlock, 0, M, cfg);
    const bool scalar = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) != 0;
    kern<<<grid, kLoopedBlock, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, N,
                                                ld, scalar);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_softmax_causal_looped(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t period,
                                         int64_t offset, const LaunchCfg& cfg) {
    auto kern = softmax_causal_looped_kernel<T, kLoopedBlock>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kLoopedBlock, 0, M, cfg);
    kern<<<grid, kLoopedBlock, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, N, ld, period,
                                                offset);
    return cudaGetLastError();
}

#define ROWOPS_SOFTMAX_ROW(T, TPR)                                                             \
    {                                                                                          \
        launch_softmax_reg<T, TPR, 1>, launch_softmax_reg<T, TPR, 2>,                          \
            launch_softmax_reg<T, TPR, 3>, launch_softmax_reg<T, TPR, 4>                       \
    }

template <typename T>
SoftmaxLaunch softmax_reg_table(int tpr_index, int vpt) {
    static const SoftmaxLaunch table[kNumTpr][kMaxVpt] = {
        ROWOPS_SOFTMAX_ROW(T, 16),  ROWOPS_SOFTMAX_ROW(T, 32),  ROWOPS_SOFTMAX_ROW(T, 64),
        ROWOPS_SOFTMAX_ROW(T, 128), ROWOPS_SOFTMAX_ROW(T, 256), ROWOPS_SOFTMAX_ROW(T, 512),
        ROWOPS_SOFTMAX_ROW(T, 1024),
    };
    if (tpr_index < 0 || tpr_index >= kNumTpr || vpt < 1 || vpt > kMaxVpt) return nullptr;
    return table[tpr_index][vpt - 1];
}
#undef ROWOPS_SOFTMAX_ROW

}  // namespace rowops
