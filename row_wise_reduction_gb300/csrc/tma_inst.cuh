// Launch wrappers and dispatch tables of the TMA-fed row-pipeline kernels for
// one element type. Included once per (operation, dtype) unit.
#pragma once

#include "rowops_launch.h"
#include "tma_row_kernels.cuh"

namespace rowops {

template <typename T>
inline size_t tma_ring_bytes(int64_t N, int nbuf) {
    return kRingHeader + size_t(nbuf) * ring_row_bytes(N, Elem<T>::kBytes);
}

template <typename T, int TPR, int VPT, bool FULL>
cudaError_t launch_softmax_tma(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                               const LaunchCfg& cfg) {
    auto kern = softmax_tma_kernel<T, TPR, VPT, 1, FULL>;
    const size_t smem = tma_ring_bytes<T>(N, nbuf);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg);
    kern<<<grid, TPR, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, int(N), ld, nbuf,
                                          cfg.dev_error, cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

// ROWS row groups per CTA share one staging of w, b; nbuf buffers per group.
template <typename T, int TPR, int VPT, int ROWS, bool FULL>
cudaError_t launch_ln_gelu_tma_rows(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                                    int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg) {
    auto kern = ln_gelu_tma_kernel<T, TPR, VPT, ROWS, FULL>;
    const size_t smem = kRingHeader + size_t(ROWS) * nbuf * ring_row_bytes(N, Elem<T>::kBytes) +
                        tma_affine_bytes<T, TPR, VPT>();
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, (M + ROWS - 1) / ROWS, cfg);
    kern<<<grid, TPR * ROWS, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                                 static_cast<const T*>(w), static_cast<const T*>(b), eps, M, int(N),
                                                 ld, nbuf, cfg.dev_error, cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, bool FULL>
cudaError_t launch_ln_gelu_tma(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                               int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg) {
    return launch_ln_gelu_tma_rows<T, TPR, VPT, 1, FULL>(x, y, w, b, eps, M, N, ld, nbuf, cfg);
}

// tables indexed [block index into kTmaBlocks][vpt index into kTmaVpts]
#define ROWOPS_TMA_ROW(FN, T, B, F) {FN<T, B, 1, F>, FN<T, B, 2, F>, FN<T, B, 3, F>, FN<T, B, 4, F>, FN<T, B, 8, F>}
#define ROWOPS_TMA_TABLE(FN, T, F)                                                                         \
    {ROWOPS_TMA_ROW(FN, T, 64, F), ROWOPS_TMA_ROW(FN, T, 128, F), ROWOPS_TMA_ROW(FN, T, 256, F),           \
     ROWOPS_TMA_ROW(FN, T, 512, F)}

template <typename T>
TmaSoftmaxLaunch softmax_tma_table(int block_index, int vpt_index, bool full) {
    static const TmaSoftmaxLaunch full_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_softmax_tma, T, true);
    static const TmaSoftmaxLaunch part_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_softmax_tma, T, false);
    if (block_index < 0 || block_index >= kNumTmaBlocks || vpt_index < 0 || vpt_index >= kNumTmaVpts) return nullptr;
    return full ? full_t[block_index][vpt_index] : part_t[block_index][vpt_index];
}

template <typename T>
TmaLnGeluLaunch ln_gelu_tma_table(int block_index, int vpt_index, bool full) {
    static const TmaLnGeluLaunch full_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_ln_gelu_tma, T, true);
    static const TmaLnGeluLaunch part_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_ln_gelu_tma, T, false);
    if (block_index < 0 || block_index >= kNumTmaBlocks || vpt_index < 0 || vpt_index >= kNumTmaVpts) return nullptr;
    return full ? full_t[block_index][vpt_index] : part_t[block_index][vpt_index];
}
#undef ROWOPS_TMA_TABLE
#undef ROWOPS_TMA_ROW

// Multi-row LayerNorm+GELU, full rows only: [tpr index into kTmaMultiTpr]
// [vpt index into kTmaMultiVpt][rows index into kTmaMultiRows]; nullptr where
// TPR * ROWS would exceed 1024 threads.
#define ROWOPS_TMA_M3(T, P, V) {launch_ln_gelu_tma_rows<T, P, V, 2, true>, launch_ln_gelu_tma_rows<T, P, V, 4, true>}
template <typename T>
TmaLnGeluLaunch ln_gelu_tma_multi_table(int tpr_index, int vpt_index, int rows_index) {
    static const TmaLnGeluLaunch t[kNumTmaMultiTpr][kNumTmaMultiVpt][kNumTmaMultiRows] = {
        {ROWOPS_TMA_M3(T, 128, 2), ROWOPS_TMA_M3(T, 128, 4), ROWOPS_TMA_M3(T, 128, 8)},
        {ROWOPS_TMA_M3(T, 256, 2), ROWOPS_TMA_M3(T, 256, 4), ROWOPS_TMA_M3(T, 256, 8)},
    };
    if (tpr_index < 0 || tpr_index >= kNumTmaMultiTpr || vpt_index < 0 || vpt_index >= kNumTmaMultiVpt ||
        rows_index < 0 || rows_index >= kNumTmaMultiRows)
        return nullptr;
    return t[tpr_index][vpt_index][rows_index];
}
#undef ROWOPS_TMA_M3

}  // namespace rowops
