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

template <typename T, int TPR, int VPT, bool FULL, bool CAUSAL = false>
cudaError_t launch_softmax_tma_mask(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                                    CausalMask cm, const LaunchCfg& cfg) {
    auto kern = softmax_tma_kernel<T, TPR, VPT, 1, FULL, CAUSAL>;
    const size_t smem = tma_ring_bytes<T>(N, nbuf);
    // softmax bf16 32768 x 4096 on GB300: 89.9 -> 84.6 us with the largest
    // carveout (the row sum's pipeline ran slower with it and keeps the default)
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg, true);
    if (e != cudaSuccess) return e;
    // CTAs per SM, side by side on bf16 32768 x 4096: the causal softmax 68.2 us with 5 (75.0 with
    // 4, 69.8 with 6); the softmax inside the bench step 89.7 us with 4 (91.5 with 3, although 3
    // is faster alone: 88.7 against 92.0; 93.5 alone with the 10 that fit)
    const int grid = cap_ctas(grid_for(reinterpret_cast<const void*>(kern), TPR, smem, M, cfg), CAUSAL ? 5 : 4, cfg);
    kern<<<grid, TPR, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y), M, int(N), ld, nbuf,
                                          cfg.dev_error, cfg.wait_ns, cfg.stall_row, cm);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, bool FULL>
cudaError_t launch_softmax_tma(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                               const LaunchCfg& cfg) {
    return launch_softmax_tma_mask<T, TPR, VPT, FULL, false>(x, y, M, N, ld, nbuf, CausalMask{1, 0}, cfg);
}

// the causal softmax on full rows: row r keeps the columns c <= (r mod period) + offset
template <typename T, int TPR, int VPT, bool FULL>
cudaError_t launch_softmax_tma_causal(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int nbuf,
                                      int64_t period, int64_t offset, const LaunchCfg& cfg) {
    return launch_softmax_tma_mask<T, TPR, VPT, true, true>(x, y, M, N, ld, nbuf, CausalMask{period, offset}, cfg);
}

// ROWS row groups per CTA share one staging of w, b; nbuf buffers per group.
template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool ERF = false>
size_t ln_gelu_tma_smem(int64_t N, int nbuf) {
    return kRingHeader + size_t(ROWS) * nbuf * ln_slot_bytes<T, TPR, VPT, FULL>(N) +
           affine_stage_bytes<T, TPR, VPT, FULL>();
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool ERF = false>
cudaError_t launch_ln_gelu_tma_rows(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                                    int64_t N, int64_t ld, int nbuf, const LaunchCfg& cfg) {
    auto kern = ln_gelu_tma_kernel<T, TPR, VPT, ROWS, FULL, ERF>;
    const size_t smem = ln_gelu_tma_smem<T, TPR, VPT, ROWS, FULL>(N, nbuf);
    cudaError_t e = allow_smem(reinterpret_cast<const void*>(kern), smem, cfg);
    if (e != cudaSuccess) return e;
    int grid = grid_for(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, (M + ROWS - 1) / ROWS, cfg);
    if (ROWS == 1) grid = cap_ctas(grid, 4, cfg);  // one group per CTA: as before the constant barrier id
    if (!FULL) {  // whole phase classes: every class needs a CTA, and they share the grid evenly
        const int period = row_phase_period(ld * int64_t(Elem<T>::kBytes));
        grid = grid >= period ? grid - grid % period : period;
    }
    kern<<<grid, TPR * ROWS, smem, cfg.stream>>>(static_cast<const T*>(x), static_cast<T*>(y),
                                                 static_cast<const T*>(w), static_cast<const T*>(b), eps, M, int(N),
                                                 ld, nbuf, cfg.dev_error, cfg.wait_ns, cfg.stall_row);
    return cudaGetLastError();
}

template <typename T, int TPR, int VPT, int ROWS, bool FULL, bool ERF = false>
int ctas_ln_gelu_tma_rows(int64_t N, int nbuf, const LaunchCfg& cfg) {
    auto kern = ln_gelu_tma_kernel<T, TPR, VPT, ROWS, FULL, ERF>;
    const size_t smem = ln_gelu_tma_smem<T, TPR, VPT, ROWS, FULL>(N, nbuf);
    if (smem + 1024 > size_t(cfg.max_smem_optin)) return 0;  // 1 KB for the static reduction buffers
    if (allow_smem(reinterpret_cast<const void*>(kern), smem, cfg) != cudaSuccess) {
        cudaGetLastError();  // a candidate that does not fit must not fail the launch that follows
        return 0;
    }
    return ctas_per_sm(reinterpret_cast<const void*>(kern), TPR * ROWS, smem, cfg);
}

// tables indexed [block index into kTmaBlocks][vpt index into kTmaVpts]
#define ROWOPS_TMA_ROW(FN, T, B, F) {FN<T, B, 1, F>, FN<T, B, 2, F>, FN<T, B, 3, F>, FN<T, B, 4, F>, FN<T, B, 8, F>}
#define ROWOPS_TMA_TABLE(FN, T, F)                                                                         \
    {ROWOPS_TMA_ROW(FN, T, 64, F), ROWOPS_TMA_ROW(FN, T, 128, F), ROWOPS_TMA_ROW(FN, T, 256, F),           \
     ROWOPS_TMA_ROW(FN, T, 512, F)}

template <typename T>
TmaSoftmaxCausalLaunch softmax_tma_causal_table(int block_index, int vpt_index) {
    static const TmaSoftmaxCausalLaunch t[kNumTmaBlocks][kNumTmaVpts] =
        ROWOPS_TMA_TABLE(launch_softmax_tma_causal, T, true);
    if (block_index < 0 || block_index >= kNumTmaBlocks || vpt_index < 0 || vpt_index >= kNumTmaVpts) return nullptr;
    return t[block_index][vpt_index];
}

template <typename T>
TmaSoftmaxLaunch softmax_tma_table(int block_index, int vpt_index, bool full) {
    static const TmaSoftmaxLaunch full_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_softmax_tma, T, true);
    static const TmaSoftmaxLaunch part_t[kNumTmaBlocks][kNumTmaVpts] = ROWOPS_TMA_TABLE(launch_softmax_tma, T, false);
    if (block_index < 0 || block_index >= kNumTmaBlocks || vpt_index < 0 || vpt_index >= kNumTmaVpts) return nullptr;
    return full ? full_t[block_index][vpt_index] : part_t[block_index][vpt_index];
}

#undef ROWOPS_TMA_TABLE
#undef ROWOPS_TMA_ROW

// LayerNorm+GELU instantiations by (TPR, VPT, ROWS); none where TPR * ROWS
// would exceed 512 threads with ROWS > 1 (at 1024 threads a CTA gets at most 64
// registers per thread and these kernels spill).
template <typename T, int P, int V, int R, bool F, bool ERF>
constexpr TmaLnGeluKernel ln_gelu_entry() {
    // 5 groups of 128 x 8 for the tanh form only: the exact form's longer
    // polynomial spills at 640 threads (bf16 65536 x 8192: 381.6 us with 4
    // groups, 400.2 with 5)
    if constexpr (R == 1 || (P * R <= 512 && R != 5) || (P == 128 && V == 8 && R == 5 && !ERF) ||
                  (P == 128 && V == 4 && R == 5 && !ERF) || (P == 64 && V == 8 && R == 10 && !ERF))
        return TmaLnGeluKernel{launch_ln_gelu_tma_rows<T, P, V, R, F, ERF>, ctas_ln_gelu_tma_rows<T, P, V, R, F, ERF>};
    else
        return TmaLnGeluKernel{nullptr, nullptr};
}
#define ROWOPS_LN1(T, P, F) \
    {ln_gelu_entry<T, P, 1, 1, F, ERF>(), ln_gelu_entry<T, P, 2, 1, F, ERF>(), ln_gelu_entry<T, P, 3, 1, F, ERF>(), \
     ln_gelu_entry<T, P, 4, 1, F, ERF>(), ln_gelu_entry<T, P, 8, 1, F, ERF>()}
#define ROWOPS_LN3(T, P, V, F) \
    {ln_gelu_entry<T, P, V, 2, F, ERF>(), ln_gelu_entry<T, P, V, 4, F, ERF>(), ln_gelu_entry<T, P, V, 5, F, ERF>(), \
     ln_gelu_entry<T, P, V, 8, F, ERF>(), ln_gelu_entry<T, P, V, 10, F, ERF>()}
#define ROWOPS_LN2(T, P, F) {ROWOPS_LN3(T, P, 2, F), ROWOPS_LN3(T, P, 4, F), ROWOPS_LN3(T, P, 8, F)}

template <int N>
int index_of(const int (&a)[N], int v) {
    for (int i = 0; i < N; ++i)
        if (a[i] == v) return i;
    return -1;
}

// ERF: the exact GELU instead of the tanh approximation
template <typename T, bool ERF = false>
TmaLnGeluKernel ln_gelu_tma_lookup(int tpr, int vpt, int rows, bool full) {
    static const TmaLnGeluKernel one_f[kNumTmaBlocks][kNumTmaVpts] = {
        ROWOPS_LN1(T, 64, true), ROWOPS_LN1(T, 128, true), ROWOPS_LN1(T, 256, true), ROWOPS_LN1(T, 512, true)};
    static const TmaLnGeluKernel one_g[kNumTmaBlocks][kNumTmaVpts] = {
        ROWOPS_LN1(T, 64, false), ROWOPS_LN1(T, 128, false), ROWOPS_LN1(T, 256, false), ROWOPS_LN1(T, 512, false)};
    static const TmaLnGeluKernel multi_f[kNumTmaMultiTpr][kNumTmaMultiVpt][kNumTmaMultiRows] = {
        ROWOPS_LN2(T, 64, true), ROWOPS_LN2(T, 128, true), ROWOPS_LN2(T, 256, true)};
    static const TmaLnGeluKernel multi_g[kNumTmaMultiTpr][kNumTmaMultiVpt][kNumTmaMultiRows] = {
        ROWOPS_LN2(T, 64, false), ROWOPS_LN2(T, 128, false), ROWOPS_LN2(T, 256, false)};
    const TmaLnGeluKernel none{nullptr, nullptr};
    if (rows == 1) {
        const int i = index_of(kTmaBlocks, tpr), j = index_of(kTmaVpts, vpt);
        if (i < 0 || j < 0) return none;
        return full ? one_f[i][j] : one_g[i][j];
    }
    const int i = index_of(kTmaMultiTpr, tpr), j = index_of(kTmaMultiVpt, vpt), r = index_of(kTmaMultiRows, rows);
    if (i < 0 || j < 0 || r < 0) return none;
    return full ? multi_f[i][j][r] : multi_g[i][j][r];
}
#undef ROWOPS_LN1
#undef ROWOPS_LN2
#undef ROWOPS_LN3

}  // namespace rowops
