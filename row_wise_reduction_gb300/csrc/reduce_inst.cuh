// Launch wrappers and dispatch tables of the row sum / row max kernels for one
// element type. Included once per dtype by reduce_f32.cu / reduce_bf16.cu.
#pragma once

#include "reduce_kernels.cuh"
#include "rowops_launch.h"
#include "softmax_inst.cuh"
#include "tma_inst.cuh"

namespace rowops {

template <typename T, int TPR, int VPT, bool FULL, class Op>
cudaError_t launch_reduce_tma(const void* x, float* out, int64_t M, int64_t N, int64_t ld, int nbuf,
                              const LaunchCfg& cfg) {
    auto kern = reduce_tma_kernel<T, TPR, VPT, FULL, Op>;
    const size_t smem = tma_ring_bytes<T>(N, nbuf);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    // 4 CTAs per SM: bf16 65536 x 8192 row sums 149.5 us against 152.4 with the occupancy limit
    const int grid = cap_ctas(grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg), 4, cfg);
    kern<<<grid, TPR, smem, cfg.stream>>>(static_cast<const T*>(x), out, M, int(N), ld, nbuf, cfg.dev_error,
                                          cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, class Op>
cudaError_t launch_reduce_reg(const void* x, float* out, int64_t M, int64_t N, int64_t ld, const LaunchCfg& cfg) {
    constexpr int BLOCK = reg_block<TPR>();
    constexpr int ROWS = BLOCK / TPR;
    auto kern = reduce_reg_kernel<T, TPR, VPT, BLOCK, Op>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), BLOCK, 0, (M + ROWS - 1) / ROWS, cfg);
    kern<<<grid, BLOCK, 0, cfg.stream>>>(static_cast<const T*>(x), out, M, int(N), ld);
    return cudaGetLastError();
}

template <typename T, class Op>
cudaError_t launch_reduce_looped(const void* x, float* out, int64_t M, int64_t N, int64_t ld, const LaunchCfg& cfg) {
    auto kern = reduce_looped_kernel<T, kLoopedBlock, kLoopedUnroll, Op>;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), kLoopedBlock, 0, M, cfg);
    kern<<<grid, kLoopedBlock, 0, cfg.stream>>>(static_cast<const T*>(x), out, M, N, ld);
    return cudaGetLastError();
}

#define ROWOPS_RED_TMA_ROW(T, B, F, OP) \
    {launch_reduce_tma<T, B, 1, F, OP>, launch_reduce_tma<T, B, 2, F, OP>, launch_reduce_tma<T, B, 3, F, OP>, \
     launch_reduce_tma<T, B, 4, F, OP>, launch_reduce_tma<T, B, 8, F, OP>}
#define ROWOPS_RED_TMA(T, F, OP) \
    {ROWOPS_RED_TMA_ROW(T, 64, F, OP), ROWOPS_RED_TMA_ROW(T, 128, F, OP), ROWOPS_RED_TMA_ROW(T, 256, F, OP), \
     ROWOPS_RED_TMA_ROW(T, 512, F, OP)}
#define ROWOPS_RED_REG_ROW(T, P, OP) \
    {launch_reduce_reg<T, P, 1, OP>, launch_reduce_reg<T, P, 2, OP>, launch_reduce_reg<T, P, 3, OP>, \
     launch_reduce_reg<T, P, 4, OP>}
#define ROWOPS_RED_REG(T, OP) \
    {ROWOPS_RED_REG_ROW(T, 16, OP), ROWOPS_RED_REG_ROW(T, 32, OP), ROWOPS_RED_REG_ROW(T, 64, OP), \
     ROWOPS_RED_REG_ROW(T, 128, OP), ROWOPS_RED_REG_ROW(T, 256, OP), ROWOPS_RED_REG_ROW(T, 512, OP), \
     ROWOPS_RED_REG_ROW(T, 1024, OP)}

// op: 0 row sum, 1 row max
template <typename T>
TmaReduceLaunch reduce_tma_table(int block_index, int vpt_index, bool full, int op) {
    static const TmaReduceLaunch sum_f[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_RED_TMA(T, true, RowSum);
    static const TmaReduceLaunch sum_g[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_RED_TMA(T, false, RowSum);
    static const TmaReduceLaunch max_f[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_RED_TMA(T, true, RowMax);
    static const TmaReduceLaunch max_g[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_RED_TMA(T, false, RowMax);
    if (block_index < 0 || block_index >= kNumTmaBlocks || vpt_index < 0 || vpt_index >= kNumTmaVpts) return nullptr;
    if (op == 0) return full ? sum_f[block_index][vpt_index] : sum_g[block_index][vpt_index];
    return full ? max_f[block_index][vpt_index] : max_g[block_index][vpt_index];
}

template <typename T>
ReduceLaunch reduce_reg_table(int tpr_index, int vpt, int op) {
    static const ReduceLaunch sum_t[kNumTpr][kMaxVpt] = ROWOPS_RED_REG(T, RowSum);
    static const ReduceLaunch max_t[kNumTpr][kMaxVpt] = ROWOPS_RED_REG(T, RowMax);
    if (tpr_index < 0 || tpr_index >= kNumTpr || vpt < 1 || vpt > kMaxVpt) return nullptr;
    return op == 0 ? sum_t[tpr_index][vpt - 1] : max_t[tpr_index][vpt - 1];
}
#undef ROWOPS_RED_TMA_ROW
#undef ROWOPS_RED_TMA
#undef ROWOPS_RED_REG_ROW
#undef ROWOPS_RED_REG

}  // namespace rowops
