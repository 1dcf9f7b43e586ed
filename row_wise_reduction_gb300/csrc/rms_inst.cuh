// Launch wrappers and dispatch tables of the register-resident and looped
// RMSNorm kernels for one element type. Included once per dtype by
// rms_f32.cu / rms_bf16.cu.
#pragma once

#include "rms_kernels.cuh"
#include "rowops_launch.h"
#include "softmax_inst.cuh"

namespace rowops {

template <typename T, int TPR, int VPT, bool RES>
cudaError_t launch_rms_reg(const void* x, const void* r, void* y, void* ro, const void* w, float eps, int64_t M,
                           int64_t N, int64_t ld, const LaunchCfg& cfg) {
    constexpr int BLOCK = reg_block<TPR>();
    constexpr int ROWS = BLOCK / TPR;
    auto kern = rms_reg_kernel<T, TPR, VPT, BLOCK, RES>;
    const size_t smem = rms_weight_smem_bytes(N, Elem<T>::kVec);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int64_t groups = (M + ROWS - 1) / ROWS;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, smem, groups, cfg);
    kern<<<grid, BLOCK, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(r), static_cast<T*>(y),
                                            static_cast<T*>(ro), static_cast<const T*>(w), eps, M, int(N), ld);
    return cudaGetLastError();
}

template <typename T, bool RES>
cudaError_t launch_rms_looped(const void* x, const void* r, void* y, void* ro, const void* w, float eps, int64_t M,
                              int64_t N, int64_t ld, const LaunchCfg& cfg) {
    auto kern = rms_looped_kernel<T, kLoopedBlock, RES>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kLoopedBlock, 0, M, cfg);
    kern<<<grid, kLoopedBlock, 0, cfg.stream>>>(static_cast<const T*>(x), static_cast<const T*>(r),
                                                static_cast<T*>(y), static_cast<T*>(ro), static_cast<const T*>(w),
                                                eps, M, N, ld);
    return cudaGetLastError();
}

#define ROWOPS_RMS_ROW(T, TPR, R) \
    {launch_rms_reg<T, TPR, 1, R>, launch_rms_reg<T, TPR, 2, R>, launch_rms_reg<T, TPR, 3, R>, launch_rms_reg<T, TPR, 4, R>}
#define ROWOPS_RMS_TABLE(T, R)                                                                                  \
    {ROWOPS_RMS_ROW(T, 16, R), ROWOPS_RMS_ROW(T, 32, R), ROWOPS_RMS_ROW(T, 64, R), ROWOPS_RMS_ROW(T, 128, R), \
     ROWOPS_RMS_ROW(T, 256, R), ROWOPS_RMS_ROW(T, 512, R), ROWOPS_RMS_ROW(T, 1024, R)}

template <typename T>
RmsLaunch rms_reg_table(int tpr_index, int vpt, bool res) {
    static const RmsLaunch plain[kNumTpr][kMaxVpt] = ROWOPS_RMS_TABLE(T, false);
    static const RmsLaunch fused[kNumTpr][kMaxVpt] = ROWOPS_RMS_TABLE(T, true);
    if (tpr_index < 0 || tpr_index >= kNumTpr || vpt < 1 || vpt > kMaxVpt) return nullptr;
    return res ? fused[tpr_index][vpt - 1] : plain[tpr_index][vpt - 1];
}
#undef ROWOPS_RMS_TABLE
#undef ROWOPS_RMS_ROW

}  // namespace rowops
