// Launch wrappers and dispatch tables of the LayerNorm+GELU kernels for one
// element type. Included once per dtype by ln_gelu_f32.cu / ln_gelu_bf16.cu.
#pragma once

#include "ln_gelu_kernels.cuh"
#include "rowops_launch.h"
#include "softmax_inst.cuh"

namespace rowops {

template <typename T, int TPR, int VPT, bool ALIGNED, bool ERF = false>
cudaError_t launch_ln_gelu_reg(const void* x, void* y, const void* w, const void* b, float eps,
                               int64_t M, int64_t N, int64_t ld, const LaunchCfg& cfg) {
    constexpr int BLOCK = reg_block<TPR>();
    constexpr int ROWS = BLOCK / TPR;
    auto kern = ln_gelu_reg_kernel<T, TPR, VPT, BLOCK, ALIGNED, ERF>;
    const size_t smem = ln_gelu_smem_bytes(N);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int64_t groups = (M + ROWS - 1) / ROWS;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, smem, groups, cfg);
    const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };  // NULL passes
    if constexpr (ALIGNED) {
        // at most two row groups per CTA: w, b straight from global memory, no staging
        if (2 * int64_t(grid) >= groups && a16(w) && a16(b)) {
            auto direct = ln_gelu_reg_kernel<T, TPR, VPT, BLOCK, true, ERF, true>;
            direct<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                                   static_cast<const T*>(w), static_cast<const T*>(b), eps, M,
                                                   int(N), ld);
            return cudaGetLastError();
        }
    }
    kern<<<grid, BLOCK, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                            static_cast<const T*>(w), static_cast<const T*>(b), eps,
                                            M, int(N), ld);
    return cudaGetLastError();
}

template <typename T, bool ERF = false>
cudaError_t launch_ln_gelu_looped(const void* x, void* y, const void* w, const void* b, float eps,
                                  int64_t M, int64_t N, int64_t ld, const LaunchCfg& cfg) {
    auto kern = ln_gelu_looped_kernel<T, kLoopedBlock, kLoopedUnroll, ERF>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kLoopedBlock, 0, M, cfg);
    const bool scalar = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) != 0;
    kern<<<grid, kLoopedBlock, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                                static_cast<const T*>(w), static_cast<const T*>(b),
                                                eps, M, N, ld, scalar);
    return cudaGetLastError();
}

#define ROWOPS_LN_ROW(T, TPR, A, ERF)                                                           \
    {                                                                                           \
        launch_ln_gelu_reg<T, TPR, 1, A, ERF>, launch_ln_gelu_reg<T, TPR, 2, A, ERF>,           \
            launch_ln_gelu_reg<T, TPR, 3, A, ERF>, launch_ln_gelu_reg<T, TPR, 4, A, ERF>        \
    }
#define ROWOPS_LN_TABLE(T, A, ERF)                                                              \
    {                                                                                           \
        ROWOPS_LN_ROW(T, 16, A, ERF), ROWOPS_LN_ROW(T, 32, A, ERF), ROWOPS_LN_ROW(T, 64, A, ERF), \
            ROWOPS_LN_ROW(T, 128, A, ERF), ROWOPS_LN_ROW(T, 256, A, ERF),                      \
            ROWOPS_LN_ROW(T, 512, A, ERF), ROWOPS_LN_ROW(T, 1024, A, ERF)                      \
    }

// ERF: the exact GELU instead of the tanh approximation
template <typename T, bool ERF = false>
LnGeluLaunch ln_gelu_reg_table(int tpr_index, int vpt, bool aligned) {
    static const LnGeluLaunch table_aligned[kNumTpr][kMaxVpt] = ROWOPS_LN_TABLE(T, true, ERF);
    static const LnGeluLaunch table_any[kNumTpr][kMaxVpt] = ROWOPS_LN_TABLE(T, false, ERF);
    if (tpr_index < 0 || tpr_index >= kNumTpr || vpt < 1 || vpt > kMaxVpt) return nullptr;
    return aligned ? table_aligned[tpr_index][vpt - 1] : table_any[tpr_index][vpt - 1];
}
#undef ROWOPS_LN_TABLE
#undef ROWOPS_LN_ROW

}  // namespace rowops
